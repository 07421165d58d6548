"""Write tiny_oracle_snapshot.json from the oracle alone (regression guard).

Run from the repository root: python tests/golden/make_oracle_snapshot.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402

TOKENS = [0, 1, 77, 255]


def snapshot():
    w = synth.workload("tiny")
    inp = synth.make_inputs(w, seed=0)
    x = oracle.decode_bf16(synth.bf16_bits(inp["x"]))[TOKENS]
    W = oracle.decode_bf16(synth.bf16_bits(inp["W"]))
    b = oracle.decode_bf16(synth.bf16_bits(inp["b"]))
    pos = inp["pos"].numpy()[TOKENS]
    q, codes, scales = oracle.forward(x, W, w.H, w.Dn, w.Dr, inp["cos"].numpy(),
                                      inp["sin"].numpy(), pos, b, quantize=True)
    return {
        "workload": "tiny", "seed": 0, "tokens": TOKENS,
        "q": [float(v) for v in q.reshape(-1)],
        "codes": [int(v) for v in codes.reshape(-1)],
        "scales": [int(v) for v in scales.reshape(-1)],
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_oracle_snapshot.json"), "w") as f:
        json.dump(snapshot(), f)
    print("wrote tiny_oracle_snapshot.json")
