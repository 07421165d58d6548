#!/usr/bin/env python3
"""Benchmark of the fused MLA query up-projection on GB300.

One step = one training pass of the layer on the long-context DeepSeek-V3
workload: T=16384 tokens (four packed 4096-token sequences, positions
t mod 4096), q_lora_rank K=1536, H=128 heads of Dn=128 + Dr=64 (N=24576),
YaRN cos/sin table (factor 40, original length 4096, beta 32/1, mscale 1)
in fp32, bf16 weights, no bias: the fused forward (GEMM + RoPE + MXFP8
output), then dgrad (inverse RoPE, dx) and wgrad (dW). Work per step =
6 T K N FLOP (2 TKN forward, 4 TKN backward).

    python bench.py --gpus N --steps K --warmup W [--impl reference]

Prints ONE JSON line (rank 0). ``value`` is TFLOP/s of the whole job with
inputs resident in HBM (CUDA events on the launch stream, L2 flushed by a
256 MiB write between steps, outside the events; the step's inputs, 0.9 GB,
are larger than L2 anyway). ``e2e`` is the same metric through the public
API with pinned host buffers: per step the inputs (x, dq) go host->device
and every output (q codes + scales, dx, dW) comes back; uploads and
downloads of neighbouring steps overlap the step's kernels on separate
streams. ``parts`` times each kernel and the other rows of the path (the
T=4096 step, MXFP8 weights, the standalone quantizers, the backward at
T=8192 with bias, the MXFP8 backward, the KV side). ``cpu_baseline`` is the
fp64 oracle on this host's cores over a bounded token sample. Under
torchrun, every rank runs its own replica (the op does not exchange data);
rank 0 prints.

``--impl reference`` times the fp64 CPU oracle on the same workload (a
bounded token sample per step, rank 0 only) and prints its line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused Q-uproj fwd/bwd TFLOP/s and % of GB300 BF16/FP8 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s)


# --------------------------------------------------------------------- utils
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(values, world):
    """Element-wise max over ranks (gloo on CPU; identity for one process)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(step_ms_per_rank_max, flop_per_step, world):
    """Whole-job throughput: all ranks' work over the slowest rank's time."""
    return world * flop_per_step / (step_ms_per_rank_max * 1e-3) / 1e12


class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) while the timed loop runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 20):
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", str(period_ms), "-i", gpu_id]
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""

    def summary(self, busy_from_mhz: float = 0.0):
        rows = []
        for ln in self.out.strip().splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[4:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r[0] > busy_from_mhz] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i in range(4) if r[2][i + 1].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(loaded)}


def gpu_id_for(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v.strip() for v in vis.split(",") if v.strip()]
    if ids and local_rank < len(ids):
        return ids[local_rank]
    return str(local_rank)


def device_info(dev):
    """Name, SM count and L2 size of the GPU the step ran on."""
    import torch
    pr = torch.cuda.get_device_properties(dev)
    out = {"name": pr.name, "sm_count": pr.multi_processor_count,
           "compute_capability": f"{pr.major}.{pr.minor}"}
    l2 = getattr(pr, "L2_cache_size", None)
    if l2:
        out["l2_mb"] = round(l2 / 2 ** 20, 1)
    return out


def source_hash(name):
    """Hash of one kernel source's code (csrc/<name>): comments and blank
    space removed, so an edit to a comment does not invalidate the DRAM
    counters captured for it."""
    import re
    with open(os.path.join(ROOT, "up_proj_gemm_gb300", "csrc", name)) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)   # block comments
    src = re.sub(r"//[^\n]*", " ", src)                  # line comments
    return hashlib.sha256(" ".join(src.split()).encode()).hexdigest()[:16]


# the sources each captured call's kernels are built from
TRAFFIC_SOURCES = {"fwd": ("fwd.cu", "ptx.cuh", "mx.cuh"), "dgrad": ("bwd.cu", "ptx.cuh", "mx.cuh"),
                   "wgrad": ("bwd.cu", "ptx.cuh", "mx.cuh")}


def kernel_hashes(call):
    return {n: source_hash(n) for n in TRAFFIC_SOURCES[call]}


def traffic_for(key: str):
    """DRAM bytes per launch of a call from the committed ncu summary, if it
    was taken on the kernel sources as they are now (same hashes); else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d["entries"][key]
        if e["sources"] != kernel_hashes(e["call"]):
            return None
        return e["bytes"]
    except Exception:
        return None


# ----------------------------------------------------------------- workload
# The largest single-GPU configuration: T = 4 x 4096 tokens, YaRN table,
# positions t mod 4096, bf16 weights, no bias, MXFP8 q; forward + backward.
HEADLINE = "dsv3_long_yarn"


def shapes(name=HEADLINE):
    import synth
    return synth.workload(name)


def make_device_inputs(w, dev, seed=0):
    """Seeded synthetic inputs drawn on the device (same distributions as the
    CPU generators the parity tests use): x ~ N(0,1) (with the workload's
    outliers), W ~ N(0,0.02), b ~ N(0,1) when the workload has a bias,
    dq ~ N(0,0.01), all rounded to bf16; the workload's cos/sin table
    (standard or YaRN) and positions."""
    import torch
    import synth
    g = torch.Generator(device=dev)
    g.manual_seed(seed)

    def nrm(shape, std):
        return (torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std).to(torch.bfloat16)

    x = nrm((w.T, w.K), w.x_std)
    if w.outlier_frac > 0:
        pick = torch.rand((w.T, w.K), generator=g, device=dev) < w.outlier_frac
        x = torch.where(pick, (x.float() * w.outlier_mult).to(torch.bfloat16), x)
    cos, sin = synth.make_tables(w)
    return {
        "x": x, "W": nrm((w.N, w.K), w.w_std), "b": nrm((w.N,), w.b_std) if w.bias else None,
        "dq": nrm((w.T, w.H, w.D), w.dq_std), "cos": cos.to(dev), "sin": sin.to(dev),
        "pos": synth.positions(w.T, w.seq_len).to(dev),
    }


def make_step(w, inp, status, dev):
    """The training step's three calls on preallocated outputs: the forward
    (MXFP8 q), dgrad (dx; it stores the rotated rope channels in ``rope``)
    and wgrad (dW, and db when the workload has a bias) reading them. Returns
    (calls dict, outputs dict, kernels launched per step)."""
    import torch
    import up_proj_gemm_gb300 as mlaq
    nb = (w.D + 31) // 32
    o = {"q": torch.empty((w.T, w.H, w.D), dtype=torch.uint8, device=dev),
         "qs": torch.empty((w.T, w.H, nb), dtype=torch.uint8, device=dev),
         "dx": torch.empty((w.T, w.K), dtype=torch.bfloat16, device=dev),
         "dW": torch.empty((w.N, w.K), dtype=torch.bfloat16, device=dev),
         "db": torch.empty((w.N,), dtype=torch.bfloat16, device=dev) if w.bias else None,
         # rotated rope channels, written by dgrad and read by wgrad (T*H*Dr bf16)
         "rope": torch.empty((w.T, w.H, w.Dr), dtype=torch.bfloat16, device=dev)}
    cs_rows, cs_width = inp["cos"].shape
    need = mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, cs_rows, cs_width, 1)
    ws = torch.empty((need,), dtype=torch.uint8, device=dev) if need else None
    # the rotary table is a model constant: packed once into the layout the
    # forward reads fastest (a copy; the forward's bytes are the same)
    packed = mlaq.rope_table_pack(inp["cos"], inp["sin"], w.Dr)

    def k_fwd():
        mlaq.fwd(inp["x"], inp["W"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, bias=inp["b"],
                 pos=inp["pos"], out_mode="mxfp8", q_out=o["q"], q_scales=o["qs"], status=status,
                 rope_packed=packed)

    def k_fwd_plain():  # the same forward reading the plain cos/sin tables
        mlaq.fwd(inp["x"], inp["W"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, bias=inp["b"],
                 pos=inp["pos"], out_mode="mxfp8", q_out=o["q"], q_scales=o["qs"], status=status)

    def k_dgrad():
        mlaq.bwd_dgrad(inp["dq"], inp["W"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, pos=inp["pos"],
                       dx=o["dx"], status=status, workspace=ws, dq_pre_rope=o["rope"])

    def k_wgrad():
        mlaq.bwd_wgrad(inp["dq"], inp["x"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, pos=inp["pos"],
                       dW=o["dW"], db=o["db"], status=status, dq_pre_rope=o["rope"])

    def k_wgrad_self():  # a delayed wgrad without dgrad's buffer: rotates dq itself
        mlaq.bwd_wgrad(inp["dq"], inp["x"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, pos=inp["pos"],
                       dW=o["dW"], db=o["db"], status=status)

    # our kernels per step: forward; dgrad = the rope pass + the stream-K GEMM
    # on its pre-rotated path (Dr = 64, Dn % 64 == 0, K % 64 == 0 with the
    # workspace it asks for), else the fused GEMM (+ the partial-sum
    # reduction when its channel reduction is split); wgrad
    pre = w.Dr == 64 and w.Dn % 64 == 0 and w.K % 64 == 0
    kernels = 1 + (2 if pre else 1 + (1 if need > 0 else 0)) + 1
    calls = {"fwd": k_fwd, "fwd_plain": k_fwd_plain, "dgrad": k_dgrad, "wgrad": k_wgrad,
             "wgrad_self": k_wgrad_self}
    return calls, o, kernels


# the other rows' timing: warm-up calls, then timed calls (mean of CUDA events)
PART_WARMUP = 10
PART_ITERS = 50


def time_loop(fn, iters, flush, stream, warmup=3):
    """Mean ms per call: CUDA events on `stream` around each call, the L2
    flush between calls outside the events."""
    import torch
    for _ in range(warmup):
        fn()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(iters)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(iters)]
    torch.cuda.synchronize()
    for i in range(iters):
        flush()
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))


def time_step(calls, steps, flush, stream):
    """Per-call CUDA events over `steps` steps of fwd -> dgrad -> wgrad, the L2
    flush between steps outside the events. Returns (mean ms of each call,
    sorted step times in ms)."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        calls["fwd"]()
        ev[i][1].record(stream)
        calls["dgrad"]()
        ev[i][2].record(stream)
        calls["wgrad"]()
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    per = [[e[j].elapsed_time(e[j + 1]) for e in ev] for j in range(3)]
    return [statistics.mean(p) for p in per], sorted(e[0].elapsed_time(e[3]) for e in ev)


def workload_config(w, world):
    table = ("YaRN (factor 40, original 4096, beta_fast 32, beta_slow 1, mscale 1), fp32"
             if w.table == "yarn" else f"standard base {w.rope_base:g}, fp32")
    return {"workload": f"{w.name}: T={w.T} fwd(bf16 W{', +bias' if w.bias else ''}, RoPE, MXFP8 q) + "
                        f"dgrad + wgrad{' + db' if w.bias else ''}",
            "T": w.T, "K": w.K, "H": w.H, "Dn": w.Dn, "Dr": w.Dr, "N": w.N,
            "pos": f"t mod {w.seq_len}" if w.seq_len else "t", "bias": w.bias,
            "rope_handoff": "dgrad stores the rotated rope channels [T, H, Dr] bf16; wgrad reads them",
            "rope_table": table + "; packed once (mla_rope_table_pack) outside the timed steps",
            "l2": "flushed (256 MiB write) between steps, outside the timed events; step inputs > L2",
            "parallelism": f"replicas x{world} (no data exchange)"}


# -------------------------------------------------------------- our arm
def tensor_peak_for(pk, timed_s, clocks):
    """The bf16 tensor peak a timed region is measured against, and whether
    it is the sustained one: a region of half a second or more, or one whose
    clock samples show the power cap, ran at the cap (the sustained figure);
    a shorter one at full clocks takes the burst figure."""
    capped = "sw_power_cap" in (clocks or {}).get("reasons", [])
    sustained = capped or timed_s >= 0.5
    return (pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]), sustained


def run_ours(args):
    import torch
    import up_proj_gemm_gb300 as mlaq

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    mlaq.lib()  # fails loudly without the CUDA library
    stream = torch.cuda.current_stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.fill_(1)

    if args.only:
        return run_only(args, flush, stream, status, dev)

    w = shapes()
    inp = make_device_inputs(w, dev, seed=rank)
    calls, _, kernels_per_step = make_step(w, inp, status, dev)
    for _ in range(args.warmup):
        flush()
        for k in ("fwd", "dgrad", "wgrad"):
            calls[k]()
    torch.cuda.synchronize()
    mlaq.check_status(status, "warm-up")

    K = args.steps
    with ClockSampler(gpu_id_for(local)) as clk:
        barrier(world)
        torch.cuda.synchronize()
        mean_k, step_times = time_step(calls, K, flush, stream)
        barrier(world)
    mlaq.check_status(status, "timed steps")
    step_ms = statistics.mean(step_times)
    step_ms_max = reduce_max([step_ms], world)[0]

    def pct(q):  # nearest-rank percentile of this rank's step times
        return step_times[min(len(step_times) - 1, max(0, int(round(q * (len(step_times) - 1)))))]
    flop_step = w.fwd_flop() + w.bwd_flop()
    value = aggregate(step_ms_max, flop_step, world)
    clocks = clk.summary(busy_from_mhz=500.0)

    pk, pk_src = peaks()
    names = ["fwd_bf16w_mxfp8out", "dgrad", "wgrad"]
    flops = [w.fwd_flop(), w.bwd_flop() / 2, w.bwd_flop() / 2]
    dom = max(range(3), key=lambda j: mean_k[j])
    # The denominator follows how the kernels ran: a timed region of half a
    # second or more, or one during which the power cap lowered the clocks,
    # is a long loop at the cap (the measured sustained figure); a short one
    # runs at full clocks (the burst figure).
    timed_s = K * step_ms / 1e3
    capped = "sw_power_cap" in clocks.get("reasons", [])
    peak, sustained = tensor_peak_for(pk, timed_s, clocks)
    achieved = flops[dom] / (mean_k[dom] * 1e-3) / 1e12
    labels = {"dgrad": "dgrad (rope pass + stream-K GEMM, one call)"}
    why = (f"the timed region is {K} steps of ~{step_ms:.2f} ms = {timed_s:.2f} s"
           + (", sw_power_cap seen" if capped else ""))
    roofline = {"bound": "tensor", "kernel": labels.get(names[dom], names[dom]), "achieved": round(achieved, 1),
                "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "traffic": traffic_for(f"{('fwd', 'dgrad', 'wgrad')[dom]}_T{w.T}"),
                "peak_source": (f"{pk_src} bf16_tflops_sustained (cuBLAS bf16 at the power cap; {why})" if sustained
                                else f"{pk_src} bf16_tflops (cuBLAS bf16 burst; {why}, full clocks)"),
                "frac_of_burst": round(achieved / pk["bf16_tflops"], 4),
                "algorithmic_flop_per_launch": flops[dom]}

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(step_ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded device-side draws, DeepSeek-V3 shapes; no datasets or weights)",
        "config": workload_config(w, world),
        "roofline": roofline,
        "gpu_launches": kernels_per_step * K,
        "clocks": clocks,
        "ms_per_step_p10_p50_p90": [round(pct(0.1), 4), round(pct(0.5), 4), round(pct(0.9), 4)],
        "device": device_info(dev),
        "kernels_ms": {n: round(m, 4) for n, m in zip(names, mean_k)},
        "kernels_tflops": {n: round(f / (m * 1e-3) / 1e12, 1) for n, f, m in zip(names, flops, mean_k)},
        "kernels_frac_bf16_burst": {n: round(f / (m * 1e-3) / 1e12 / pk["bf16_tflops"], 4)
                                    for n, f, m in zip(names, flops, mean_k)},
        "kernels_frac_of_peak": {n: round(f / (m * 1e-3) / 1e12 / peak, 4) for n, f, m in zip(names, flops, mean_k)},
        "step_frac_of_peak": round(value / world / peak, 4),
    }

    # ---------------------------------------------------------------- e2e
    e2e_steps = max(3, min(args.e2e_steps, K))
    out["e2e"] = run_e2e(w, inp, status, flop_step, world, e2e_steps, args.warmup, dev)
    del inp, calls
    torch.cuda.empty_cache()

    if rank == 0 and not args.no_parts:
        out["parts"] = run_parts(dev, stream, flush, pk, pk_src)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_e2e(w, inp, status, flop_step, world, steps, warmup, dev):
    """The step end to end through the public API with pinned host buffers:
    every step uploads its inputs (x, dq) and downloads every output (q
    codes + scales, dx, dW, and db when the workload has a bias). Two device
    buffer sets and three streams (upload, compute, download) let step i+1's
    upload and step i-1's download run while step i's kernels do, as a
    training loop fed from host memory would; each step still moves all of
    its own bytes. Timed with CUDA events from the first upload to the last
    download, divided by the steps."""
    import torch
    import up_proj_gemm_gb300 as mlaq
    hx = inp["x"].cpu().pin_memory()
    hdq = inp["dq"].cpu().pin_memory()
    nb = (w.D + 31) // 32
    hq = torch.empty((w.T, w.H, w.D), dtype=torch.uint8).pin_memory()
    hs = torch.empty((w.T, w.H, nb), dtype=torch.uint8).pin_memory()
    hdx = torch.empty((w.T, w.K), dtype=torch.bfloat16).pin_memory()
    hdW = torch.empty((w.N, w.K), dtype=torch.bfloat16).pin_memory()
    hdb = torch.empty((w.N,), dtype=torch.bfloat16).pin_memory() if w.bias else None
    sets = []
    for _ in range(2):
        sets.append({
            "x": torch.empty_like(inp["x"]), "dq": torch.empty_like(inp["dq"]),
            "q": torch.empty((w.T, w.H, w.D), dtype=torch.uint8, device=dev),
            "qs": torch.empty((w.T, w.H, nb), dtype=torch.uint8, device=dev),
            "dx": torch.empty((w.T, w.K), dtype=torch.bfloat16, device=dev),
            "dW": torch.empty((w.N, w.K), dtype=torch.bfloat16, device=dev),
            "db": torch.empty((w.N,), dtype=torch.bfloat16, device=dev) if w.bias else None,
            "rope": torch.empty((w.T, w.H, w.Dr), dtype=torch.bfloat16, device=dev),
        })
    need = mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, inp["cos"].shape[0], inp["cos"].shape[1], 1)
    ws = torch.empty((need,), dtype=torch.uint8, device=dev) if need else None
    packed = mlaq.rope_table_pack(inp["cos"], inp["sin"], w.Dr)  # a model constant, packed once
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)
    in_done, cmp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def step(i):
        j = i % 2
        b = sets[j]
        with torch.cuda.stream(s_in):
            s_in.wait_event(cmp_done[j])  # step i-2's kernels are done with set j's inputs
            b["x"].copy_(hx, non_blocking=True)
            b["dq"].copy_(hdq, non_blocking=True)
            in_done[j].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(in_done[j])
            s_cmp.wait_event(out_done[j])  # step i-2's outputs in set j have been read back
            mlaq.fwd(b["x"], inp["W"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, bias=inp["b"], pos=inp["pos"],
                     out_mode="mxfp8", q_out=b["q"], q_scales=b["qs"], status=status, rope_packed=packed)
            mlaq.bwd_dgrad(b["dq"], inp["W"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, pos=inp["pos"],
                           dx=b["dx"], status=status, workspace=ws, dq_pre_rope=b["rope"])
            mlaq.bwd_wgrad(b["dq"], b["x"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, pos=inp["pos"],
                           dW=b["dW"], db=b["db"], status=status, dq_pre_rope=b["rope"])
            cmp_done[j].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(cmp_done[j])
            hq.copy_(b["q"], non_blocking=True)
            hs.copy_(b["qs"], non_blocking=True)
            hdx.copy_(b["dx"], non_blocking=True)
            hdW.copy_(b["dW"], non_blocking=True)
            if hdb is not None:
                hdb.copy_(b["db"], non_blocking=True)
            out_done[j].record(s_out)

    for i in range(max(3, warmup)):
        step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(steps):
        step(i)
    t1.record(s_out)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    ms = reduce_max([ms], world)[0]
    mlaq.check_status(status, "e2e steps")
    h2d = hx.numel() * 2 + hdq.numel() * 2
    d2h = hq.numel() + hs.numel() + hdx.numel() * 2 + hdW.numel() * 2 + (hdb.numel() * 2 if hdb is not None else 0)
    return {"value": round(aggregate(ms, flop_step, world), 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "h2d_plus_d2h_GBps": round((h2d + d2h) / (ms * 1e-3) / 1e9, 1),
            "pipeline": "2 buffer sets; upload, compute and download on separate streams"}


def run_only(args, flush, stream, status, dev):
    """One kernel alone, K timed calls (for profiling: a short, fixed launch
    sequence), on ``--workload`` (default: the step's workload; the MXFP8
    weight forward defaults to its own T=4096 workload). Prints a JSON line
    with its mean time."""
    import torch
    import synth
    import up_proj_gemm_gb300 as mlaq
    name = args.workload or ("dsv3_fwd_mxfp8w" if args.only == "fwd_mxfp8w" else HEADLINE)
    w = shapes(name)
    inp = make_device_inputs(w, dev, seed=0)
    kernels, _, _ = make_step(w, inp, status, dev)
    kernels["dgrad"]()  # fills the rope buffer wgrad reads
    if args.only in kernels:
        fn = kernels[args.only]
        flop = w.fwd_flop() if args.only in ("fwd", "fwd_plain") else w.bwd_flop() / 2
    elif args.only == "fwd_mxfp8w":
        xq, xs = mlaq.mxfp8_quantize_rows(inp["x"])
        Wq, Ws = mlaq.mxfp8_quantize_rows(inp["W"])
        qc = torch.empty((w.T, w.H, w.D), dtype=torch.uint8, device=dev)
        qs = torch.empty((w.T, w.H, (w.D + 31) // 32), dtype=torch.uint8, device=dev)

        # operands quantized outside the timing, scales written in the GEMM's tiled order
        G = mlaq.w_scale_group(w.T, w.K, w.H, w.Dn, w.Dr, inp["cos"].shape[0], inp["cos"].shape[1])
        _, xst = mlaq.mxfp8_quantize_rows(inp["x"], group=128)
        _, Wst = mlaq.mxfp8_quantize_rows(inp["W"], group=G)

        packed = mlaq.rope_table_pack(inp["cos"], inp["sin"], w.Dr)

        def fn():
            mlaq.fwd(xq, Wq, inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, pos=inp["pos"], weight_mode="mxfp8_tiled",
                     out_mode="mxfp8", x_scales=xst, w_scales=Wst, q_out=qc, q_scales=qs, status=status,
                     rope_packed=packed)
        flop = w.fwd_flop()
    elif args.only == "bwd_mxfp8":
        dx = torch.empty((w.T, w.K), dtype=torch.bfloat16, device=dev)
        dW = torch.empty((w.N, w.K), dtype=torch.bfloat16, device=dev)
        db = torch.empty((w.N,), dtype=torch.bfloat16, device=dev)
        ws = torch.empty((mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, inp["cos"].shape[0],
                                              inp["cos"].shape[1], 3),), dtype=torch.uint8, device=dev)

        def fn():
            mlaq.bwd_mxfp8(inp["dq"], inp["W"], inp["x"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr,
                           pos=inp["pos"], dx=dx, dW=dW, db=db, status=status, workspace=ws)
        flop = w.bwd_flop()
    elif args.only == "quant_cols":
        a = torch.randn((w.T, w.N), device=dev).to(torch.bfloat16)
        codes = torch.empty((w.N, w.T), dtype=torch.uint8, device=dev)
        sc = torch.empty((w.N, (w.T + 31) // 32), dtype=torch.uint8, device=dev)

        def fn():
            mlaq.mxfp8_quantize_cols(a, codes, sc)
        flop = 0
    elif args.only == "quant":
        a = torch.randn((w.T, w.N), device=dev).to(torch.bfloat16)
        codes = torch.empty((w.T, w.N), dtype=torch.uint8, device=dev)
        sc = torch.empty((w.T, (w.N + 31) // 32), dtype=torch.uint8, device=dev)

        def fn():
            mlaq.mxfp8_quantize_rows(a, codes, sc)
        flop = 0
    elif args.only == "kv":
        # the KV side at the DeepSeek-V3 shape: kv_lora_rank 512, H 128, 128 + 128 + 64
        T, K, H, Dn, Dv, Dr = w.T, 512, w.H, 128, 128, 64
        g = torch.Generator(device=dev)
        g.manual_seed(5)
        c_kv = torch.randn((T, K), generator=g, device=dev).to(torch.bfloat16)
        Wkv = (torch.randn((H * (Dn + Dv), K), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        k_pe = torch.randn((T, Dr), generator=g, device=dev).to(torch.bfloat16)
        kcos, ksin = [t.to(dev) for t in synth.rope_table_standard(T, Dr)]
        o_key = torch.empty((T, H, Dn + Dr), dtype=torch.bfloat16, device=dev)
        o_value = torch.empty((T, H, Dv), dtype=torch.bfloat16, device=dev)

        def fn():
            mlaq.kv_fwd(c_kv, Wkv, k_pe, kcos, ksin, H, Dn, Dv, Dr, o_key=o_key, o_value=o_value, status=status)
        flop = 2 * T * K * H * (Dn + Dv)
    else:
        raise SystemExit(f"unknown --only {args.only}")
    ms = time_loop(fn, args.steps, flush, stream, warmup=args.warmup)
    mlaq.check_status(status, args.only)
    print(json.dumps({"only": args.only, "workload": name, "T": w.T, "ms": round(ms, 4), "steps": args.steps,
                      "warmup": args.warmup,
                      "TFLOP/s": round(flop / (ms * 1e-3) / 1e12, 1) if flop else None}), flush=True)


def run_parts(dev, stream, flush, pk, pk_src):
    """The other rows of the path, each timed on its own (CUDA events, L2
    flushed between calls): the standalone quantizers, the MXFP8-weight
    forward, the forward alone, the backward at T=8192 (bf16 and MXFP8), the
    KV side and the training step at T=4096."""
    import torch
    import synth
    import up_proj_gemm_gb300 as mlaq
    parts = {}
    bf16_peak = pk["bf16_tflops"]  # kernels timed alone: burst figure
    fp8_peak = bf16_peak * FP8_OVER_BF16
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    # standalone quantizer, [4096, 24576] bf16 and [24576, 1536] bf16 (W)
    for R, C in ((4096, 24576), (24576, 1536), (16384, 24576)):
        a = torch.randn((R, C), device=dev, dtype=torch.float32).to(torch.bfloat16)
        codes = torch.empty((R, C), dtype=torch.uint8, device=dev)
        sc = torch.empty((R, (C + 31) // 32), dtype=torch.uint8, device=dev)
        ms = time_loop(lambda: mlaq.mxfp8_quantize_rows(a, codes, sc), PART_ITERS, flush, stream, warmup=PART_WARMUP)
        byts = R * C * 2 + R * C + R * ((C + 31) // 32)
        gbs = byts / (ms * 1e-3) / 1e9
        parts[f"quantize_rows_bf16_{R}x{C}"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                                "frac_hbm": round(gbs / pk["hbm_gbs"], 4),
                                                "algorithmic_bytes": byts}
        del a, codes, sc

    # columnwise copy (the transpose helper): dq [4096, 24576] and x [4096, 1536] reduced over tokens
    for R, C in ((4096, 24576), (4096, 1536)):
        a = torch.randn((R, C), device=dev, dtype=torch.float32).to(torch.bfloat16)
        codes = torch.empty((C, R), dtype=torch.uint8, device=dev)
        sc = torch.empty((C, (R + 31) // 32), dtype=torch.uint8, device=dev)
        ms = time_loop(lambda: mlaq.mxfp8_quantize_cols(a, codes, sc), PART_ITERS, flush, stream, warmup=PART_WARMUP)
        byts = R * C * 2 + R * C + C * ((R + 31) // 32)
        gbs = byts / (ms * 1e-3) / 1e9
        parts[f"quantize_cols_bf16_{R}x{C}"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                                "frac_hbm": round(gbs / pk["hbm_gbs"], 4),
                                                "algorithmic_bytes": byts}
        del a, codes, sc

    # forward with MXFP8 weights (x with 1% x50 outliers), MXFP8 out
    w = synth.workload("dsv3_fwd_mxfp8w")
    inp = make_device_inputs(w, dev, seed=11)
    xq, xs = mlaq.mxfp8_quantize_rows(inp["x"])
    Wq, Ws = mlaq.mxfp8_quantize_rows(inp["W"])
    qc = torch.empty((w.T, w.H, w.D), dtype=torch.uint8, device=dev)
    qs = torch.empty((w.T, w.H, (w.D + 31) // 32), dtype=torch.uint8, device=dev)
    ms_g = time_loop(lambda: mlaq.fwd(xq, Wq, inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, pos=inp["pos"],
                                      weight_mode="mxfp8", out_mode="mxfp8", x_scales=xs, w_scales=Ws,
                                      q_out=qc, q_scales=qs, status=st), PART_ITERS, flush, stream, warmup=PART_WARMUP)
    # the same operands with the quantizer writing the scales in the GEMM's tiled order
    G = mlaq.w_scale_group(w.T, w.K, w.H, w.Dn, w.Dr, inp["cos"].shape[0], inp["cos"].shape[1])
    _, xst = mlaq.mxfp8_quantize_rows(inp["x"], group=128)
    _, Wst = mlaq.mxfp8_quantize_rows(inp["W"], group=G)
    packed = mlaq.rope_table_pack(inp["cos"], inp["sin"], w.Dr)  # a model constant, packed once
    ms_t = time_loop(lambda: mlaq.fwd(xq, Wq, inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, pos=inp["pos"],
                                      weight_mode="mxfp8_tiled", out_mode="mxfp8", x_scales=xst, w_scales=Wst,
                                      q_out=qc, q_scales=qs, status=st), PART_ITERS, flush, stream,
                     warmup=PART_WARMUP)
    ms = time_loop(lambda: mlaq.fwd(xq, Wq, inp["cos"], inp["sin"], w.H, w.Dn, w.Dr, pos=inp["pos"],
                                    weight_mode="mxfp8_tiled", out_mode="mxfp8", x_scales=xst, w_scales=Wst,
                                    q_out=qc, q_scales=qs, status=st, rope_packed=packed), PART_ITERS, flush,
                   stream, warmup=PART_WARMUP)
    tf = w.fwd_flop() / (ms * 1e-3) / 1e12
    parts["fwd_mxfp8w_mxfp8out_T4096"] = {"ms": round(ms, 4), "TFLOP/s": round(tf, 1),
                                          "frac_fp8_peak": round(tf / fp8_peak, 4),
                                          "peak": f"{pk_src} bf16 burst x{FP8_OVER_BF16:g} (nominal fp8/bf16)",
                                          "scales": "in the GEMM's tiled order (mxfp8_quantize_rows_tiled)",
                                          "rope_table": "packed (mla_rope_table_pack)",
                                          "ms_plain_table": round(ms_t, 4),
                                          "ms_row_major_scales_plain_table": round(ms_g, 4)}
    ms_p = time_loop(lambda: mlaq.fwd(inp["x"], inp["W"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr,
                                      pos=inp["pos"], out_mode="mxfp8", q_out=qc, q_scales=qs, status=st),
                     PART_ITERS, flush, stream, warmup=PART_WARMUP)
    ms = time_loop(lambda: mlaq.fwd(inp["x"], inp["W"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr,
                                    pos=inp["pos"], out_mode="mxfp8", q_out=qc, q_scales=qs, status=st,
                                    rope_packed=packed), PART_ITERS, flush, stream, warmup=PART_WARMUP)
    tf = w.fwd_flop() / (ms * 1e-3) / 1e12
    parts["fwd_bf16w_mxfp8out_T4096_alone"] = {"ms": round(ms, 4), "TFLOP/s": round(tf, 1),
                                               "frac_bf16_peak": round(tf / bf16_peak, 4),
                                               "rope_table": "packed", "ms_plain_table": round(ms_p, 4)}
    # the same forward writing its scales per head in the block-scaled GEMM's tiled order
    qsw = torch.empty((w.H, int(mlaq.lib().mxfp8_swizzled_scale_bytes(w.T, (w.D + 31) // 32))),
                      dtype=torch.uint8, device=dev)
    ms = time_loop(lambda: mlaq.fwd(inp["x"], inp["W"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr,
                                    pos=inp["pos"], out_mode="mxfp8_bhsd_swizzled", q_out=qc, q_scales=qsw,
                                    status=st), PART_ITERS, flush, stream, warmup=PART_WARMUP)
    tf = w.fwd_flop() / (ms * 1e-3) / 1e12
    parts["fwd_bf16w_mxfp8out_swizzled_scales_T4096"] = {"ms": round(ms, 4), "TFLOP/s": round(tf, 1),
                                                         "frac_bf16_peak": round(tf / bf16_peak, 4)}
    del inp, xq, xs, Wq, Ws, qc, qs, qsw, Wst, xst, packed

    # backward at T = 2 x 4096, bias on
    w = synth.workload("dsv3_bwd")
    inp = make_device_inputs(w, dev, seed=12)
    dx = torch.empty((w.T, w.K), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((w.N, w.K), dtype=torch.bfloat16, device=dev)
    db = torch.empty((w.N,), dtype=torch.bfloat16, device=dev)
    rope = torch.empty((w.T, w.H, w.Dr), dtype=torch.bfloat16, device=dev)
    ms_d = time_loop(lambda: mlaq.bwd_dgrad(inp["dq"], inp["W"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr,
                                            pos=inp["pos"], dx=dx, status=st, dq_pre_rope=rope),
                     PART_ITERS, flush, stream, warmup=PART_WARMUP)
    ms_w = time_loop(lambda: mlaq.bwd_wgrad(inp["dq"], inp["x"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr,
                                            pos=inp["pos"], dW=dW, db=db, status=st, dq_pre_rope=rope),
                     PART_ITERS, flush, stream, warmup=PART_WARMUP)
    ms_ws = time_loop(lambda: mlaq.bwd_wgrad(inp["dq"], inp["x"], inp["cos"], inp["sin"], w.H, w.Dn, w.Dr,
                                             pos=inp["pos"], dW=dW, db=db, status=st), PART_ITERS, flush, stream, warmup=PART_WARMUP)
    half = w.bwd_flop() / 2
    parts["bwd_T8192"] = {"dgrad_ms": round(ms_d, 4), "wgrad_db_ms": round(ms_w, 4),
                          "wgrad_db_self_rotating_ms": round(ms_ws, 4),
                          "TFLOP/s": round(w.bwd_flop() / ((ms_d + ms_w) * 1e-3) / 1e12, 1),
                          "dgrad_TFLOP/s": round(half / (ms_d * 1e-3) / 1e12, 1),
                          "wgrad_TFLOP/s": round(half / (ms_w * 1e-3) / 1e12, 1),
                          "frac_bf16_peak": round(w.bwd_flop() / ((ms_d + ms_w) * 1e-3) / 1e12 / bf16_peak, 4)}
    # the same backward with MXFP8 GEMMs: rotate + both quantized copies of dq_pre, the
    # columnwise copies of W and x, the two block-scaled GEMMs and db, in one call
    ws = torch.empty((mlaq.workspace_size(w.T, w.K, w.H, w.Dn, w.Dr, inp["cos"].shape[0],
                                          inp["cos"].shape[1], 3),), dtype=torch.uint8, device=dev)
    ms_mx = time_loop(lambda: mlaq.bwd_mxfp8(inp["dq"], inp["W"], inp["x"], inp["cos"], inp["sin"], w.H, w.Dn,
                                             w.Dr, pos=inp["pos"], dx=dx, dW=dW, db=db, status=st,
                                             workspace=ws), PART_ITERS, flush, stream, warmup=PART_WARMUP)
    tf = w.bwd_flop() / (ms_mx * 1e-3) / 1e12
    parts["bwd_mxfp8_T8192"] = {"ms": round(ms_mx, 4), "TFLOP/s": round(tf, 1),
                                "frac_fp8_peak": round(tf / fp8_peak, 4),
                                "speedup_vs_bf16_bwd": round((ms_d + ms_w) / ms_mx, 3),
                                "note": "whole call: quantization passes included"}
    del inp, dx, dW, db, rope, ws

    # KV side: c_kv [4096, 512] x W_UKV [128 x (128 + 128), 512]^T, shared k_pe rotated into every key
    T, K, H, Dn, Dv, Dr = 4096, 512, 128, 128, 128, 64
    g = torch.Generator(device=dev)
    g.manual_seed(14)
    c_kv = torch.randn((T, K), generator=g, device=dev).to(torch.bfloat16)
    W = (torch.randn((H * (Dn + Dv), K), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    k_pe = torch.randn((T, Dr), generator=g, device=dev).to(torch.bfloat16)
    cos, sin = [t.to(dev) for t in synth.rope_table_standard(T, Dr)]
    o_key = torch.empty((T, H, Dn + Dr), dtype=torch.bfloat16, device=dev)
    o_value = torch.empty((T, H, Dv), dtype=torch.bfloat16, device=dev)
    ms = time_loop(lambda: mlaq.kv_fwd(c_kv, W, k_pe, cos, sin, H, Dn, Dv, Dr, o_key=o_key, o_value=o_value,
                                       status=st), PART_ITERS, flush, stream, warmup=PART_WARMUP)
    flop = 2 * T * K * H * (Dn + Dv)
    byts = (T * K + H * (Dn + Dv) * K + T * Dr + T * H * (Dn + Dr) + T * H * Dv) * 2
    parts["kv_uproj_rope_T4096"] = {"ms": round(ms, 4), "TFLOP/s": round(flop / (ms * 1e-3) / 1e12, 1),
                                    "GB/s": round(byts / (ms * 1e-3) / 1e9, 1),
                                    "frac_hbm": round(byts / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                                    "algorithmic_bytes": byts, "algorithmic_flop": flop}
    del c_kv, W, k_pe, o_key, o_value

    # the training step at T = 4096 (the forward configuration's batch, bias on), each call timed
    w = synth.workload("dsv3_fwd_bf16w", bias=True, passes=("fwd", "bwd"))
    inp = make_device_inputs(w, dev, seed=13)
    calls, _, _ = make_step(w, inp, st, dev)
    for _ in range(PART_WARMUP):
        flush()
        for k in ("fwd", "dgrad", "wgrad"):
            calls[k]()
    mean_k, step_times = time_step(calls, PART_ITERS, flush, stream)
    ms = statistics.mean(step_times)
    flops = [w.fwd_flop(), w.bwd_flop() / 2, w.bwd_flop() / 2]
    tf = (w.fwd_flop() + w.bwd_flop()) / (ms * 1e-3) / 1e12
    parts["train_step_T4096"] = {
        "ms": round(ms, 4), "TFLOP/s": round(tf, 1), "frac_bf16_peak": round(tf / bf16_peak, 4),
        "kernels_ms": {n: round(m, 4) for n, m in zip(("fwd", "dgrad", "wgrad_db"), mean_k)},
        "kernels_frac_bf16_peak": {n: round(f / (m * 1e-3) / 1e12 / bf16_peak, 4)
                                   for n, f, m in zip(("fwd", "dgrad", "wgrad_db"), flops, mean_k)},
        "workload": "T=4096, pos = t, standard table, bias on: fwd (MXFP8 q) + dgrad + wgrad + db"}
    del inp, calls
    torch.cuda.synchronize()
    mlaq.check_status(st, "parts")
    parts["peak_note"] = f"{pk_src} peaks; kernels timed alone use the burst bf16 figure"
    return parts


# -------------------------------------------------- CPU oracle (baseline)
def oracle_step_sample(w, tokens, inputs):
    """The oracle on a token sample of the step: forward (linear, bias, RoPE,
    MXFP8), RoPE backward, dgrad, and the sample's share of wgrad and bgrad.
    Returns seconds; the work is 6 * tokens * K * N FLOP."""
    import numpy as np
    import oracle
    x, W, b, dq, cos, sin, pos = inputs
    t0 = time.perf_counter()
    oracle.forward(x[:tokens], W, w.H, w.Dn, w.Dr, cos, sin, pos[:tokens], b, quantize=True)
    oracle.backward(dq[:tokens], x[:tokens], W, w.H, w.Dn, w.Dr, cos, sin, pos[:tokens])
    return time.perf_counter() - t0


def oracle_inputs(w, tokens):
    import numpy as np
    import oracle
    import synth
    sub = synth.workload(w.name, T=tokens, bias=w.bias, seq_len=w.seq_len)
    inp = synth.make_inputs(sub, seed=0)
    cos, sin = synth.make_tables(w)
    f = lambda t: oracle.decode_bf16(synth.bf16_bits(t))
    return (f(inp["x"]), f(inp["W"]), f(inp["b"]) if inp["b"] is not None else None, f(inp["dq"]),
            cos.numpy(), sin.numpy(), synth.positions(tokens, w.seq_len).numpy())


def cpu_baseline(w, budget_s=15.0):
    import oracle
    probe = 8
    t = oracle_step_sample(w, probe, oracle_inputs(w, probe))
    tokens = int(max(probe, min(w.T, probe * budget_s / max(t, 1e-6))))
    if tokens > probe:
        t = oracle_step_sample(w, tokens, oracle_inputs(w, tokens))
        # a small probe under-uses the cores, so the first sample can land well
        # under the budget: rescale once from that sample
        if t < 0.5 * budget_s and tokens < w.T:
            tokens = int(min(w.T, tokens * budget_s / max(t, 1e-6)))
            t = oracle_step_sample(w, tokens, oracle_inputs(w, tokens))
    flop = 6.0 * tokens * w.K * w.N
    return {"value": round(flop / t / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(t, 3),
            "sample": f"{tokens} of {w.T} tokens of the step (fwd + MXFP8, RoPE bwd, dgrad, the sample's "
                      f"wgrad{'/bgrad' if w.bias else ''} share), fp64, OpenMP over rows"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = shapes()
    inputs = oracle_inputs(w, 64)
    per_step_budget = max(0.05, args.ref_budget / max(1, args.steps + args.warmup))
    t = oracle_step_sample(w, 1, inputs)
    tokens = int(max(1, min(64, per_step_budget / max(t, 1e-6))))
    for _ in range(args.warmup):
        oracle_step_sample(w, tokens, inputs)
    times = [oracle_step_sample(w, tokens, inputs) for _ in range(args.steps)]
    ms = statistics.mean(times) * 1e3
    value = 6.0 * tokens * w.K * w.N / (ms * 1e-3) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": dict(workload_config(w, world), tokens_per_step=tokens,
                                            sample="a token sample of the step per step (fp64 CPU oracle)"),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": f"{tokens} of {w.T} tokens per step"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--only", choices=("fwd", "fwd_plain", "dgrad", "wgrad", "wgrad_self", "fwd_mxfp8w", "quant",
                                      "quant_cols",
                                          "bwd_mxfp8", "kv"),
                    help="time one kernel alone (profiling)")
    ap.add_argument("--workload", choices=("tiny", "dsv3_fwd_bf16w", "dsv3_fwd_mxfp8w", "dsv3_bwd", HEADLINE),
                    help="workload of --only (default: the step's)")
    ap.add_argument("--no-parts", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--ref-budget", type=float, default=120.0, help="seconds for --impl reference")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
