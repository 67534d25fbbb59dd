"""The N > 1 path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Each rank runs its own replica of the workload (weak scaling, no collective on
the data path); the only cross-rank steps are the barrier around the timed
region and the max / sum reductions of the timings and byte counts.  Rank 0
alone runs the oracle reference arm.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "QMM_BENCH_BACKEND": "gloo"})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup()
    res = {"world": w, "rank": r, "local": local}
    bench.barrier(w)
    res["max"] = bench.max_over_ranks(w, 1.5 + r)
    res["sum"] = bench.sum_over_ranks(w, 10.0 * (r + 1))

    class Args:
        steps, warmup = 3, 3

    if r != 0:
        # only rank 0 runs the reference arm; the others return at once
        res["reference_returned"] = bench.run_reference(Args, w, r) is None
    bench.barrier(w)
    dist.destroy_process_group()
    out.put(res)


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = [out.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort(key=lambda d: d["rank"])
    assert [d["rank"] for d in results] == [0, 1]
    for d in results:
        assert d["world"] == 2 and d["local"] == d["rank"]
        assert d["max"] == pytest.approx(2.5)      # max over ranks of 1.5 + rank
        assert d["sum"] == pytest.approx(30.0)     # 10 + 20
    assert results[1]["reference_returned"]
