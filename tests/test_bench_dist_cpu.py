"""Host-side multi-rank logic of bench.py on CPU (gloo, world size 2): each
rank runs an independent replica, the timing is reduced by max over ranks,
only rank 0 prints, and the reference arm runs on rank 0 alone."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_env()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    worst = bench.max_over_ranks(1.5 + r, w, torch.device("cpu"))
    # replicas draw different inputs (seed offset by rank), same shapes
    wl = bench.wl.CONFIGS["tiny"]
    topk = bench.wl.make_inputs(bench.dataclass_replace_seed(wl, wl.seed + r), with_partial=False).topk_idx
    q.put((r, w, worst, topk.shape, int(topk.sum())))
    torch.distributed.destroy_process_group()


def test_two_rank_replicas_max_over_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 and r[2] == pytest.approx(2.5) for r in res)
    assert res[0][3] == res[1][3] and res[0][4] != res[1][4]


def _reference_rank1(port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    import contextlib
    import io
    import sys
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup = 1, 3
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(A(), 2, 1)
    q.put(buf.getvalue())


def test_reference_arm_runs_on_rank0_only():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_reference_rank1, args=(_free_port(), q))
    p.start()
    p.join(timeout=120)
    assert p.exitcode == 0
    assert q.get(timeout=10) == ""


@pytest.mark.parametrize("E,R,k", [(2048, 256, 8), (256, 8, 8), (256, 64, 8), (16, 4, 2), (256, 256, 8), (64, 8, 6)])
def test_bench_expected_distinct_ranks_is_the_closed_form(E, R, k):
    # the figure bench.py prints beside each layout's realised mean is the pages' closed form
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from oracle.expected_topk import get_expected_topk
    assert bench.expected_distinct_ranks(E, R, k) == pytest.approx(get_expected_topk(E, R, k), rel=1e-12, abs=1e-12)
