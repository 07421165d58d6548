"""bench.py's multi-process plumbing on CPU: two gloo ranks, max-over-ranks
timing and whole-job aggregation (the op itself runs as independent replicas,
one per GPU, with no data exchange)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo")
    w, r, l = bench.dist_env()
    bench.barrier(w)
    step_ms = [2.0, 3.0][rank]
    m = bench.reduce_max([step_ms, 10.0 * rank], w)
    q.put((r, w, m, bench.aggregate(m[0], 1e12, w)))
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, m, agg in res:
        assert w == 2 and m == [3.0, 10.0]
        # 2 ranks x 1 TFLOP each over the slowest rank's 3 ms
        assert agg == pytest.approx(2 * 1e12 / 3e-3 / 1e12)


def test_single_process_helpers():
    assert bench.reduce_max([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.aggregate(1.0, 1e12, 1) == pytest.approx(1000.0)


def test_tensor_peak_follows_how_the_step_ran():
    """Short region at full clocks: burst; long region or power cap: sustained."""
    pk = {"bf16_tflops": 1910.7, "bf16_tflops_sustained": 1710.9}
    full = {"reasons": []}
    capped = {"reasons": ["sw_power_cap"]}
    assert bench.tensor_peak_for(pk, 0.05, full) == (1910.7, False)
    assert bench.tensor_peak_for(pk, 0.05, capped) == (1710.9, True)
    assert bench.tensor_peak_for(pk, 1.2, full) == (1710.9, True)
    assert bench.tensor_peak_for(pk, 0.499, None) == (1910.7, False)
