"""The path as a pipeline: several steps captured in one CUDA graph (and the
same launches issued eagerly on a side stream), every kernel launched with
programmatic dependent launch. Each kernel reads what the one before it wrote
(the combine reads the dispatch's receive rows: identity experts), and the
second step's layout and dispatch overwrite buffers the first step's combine
reads, so a kernel that touched memory before its predecessor finished would
change a result. Every step is checked bit for bit against the oracle's chain
of layout, dispatch and combine."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_moe_get_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    from combine_moe_get_gb300 import binding
    return binding


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def routings(T, k, E, seeds):
    out = []
    for s in seeds:
        g = torch.Generator().manual_seed(s)
        out.append(wl.mask_random_lanes(g, wl.make_topk_uniform(g, T, E, k), 0.2))
    return out


def expected_chain(x, topk, E, R, cap, fp8):
    lay = oracle.layout(topk.numpy(), E, R)
    N = lay["num_recv"]
    d = oracle.dispatch(bits16(x), topk.numpy(), None, E, R, lay["token_dst_row"], cap, fp8=fp8)
    if fp8:
        ref, flags = oracle.combine_fp8(d["recv_x"][:N], d["recv_x_scales"][:N], lay["token_dst_row"])
    else:
        ref, flags = oracle.combine(d["recv_x"][:N], lay["token_dst_row"])
    assert flags == 0
    return ref


class Pipeline:
    """Buffers shared by every step: the layout, its workspace and the receive
    rows; each step has its own routing, input and output."""

    def __init__(self, moe, T, H, k, E, R, fp8, steps, seed):
        self.moe, self.E, self.R, self.fp8 = moe, E, R, fp8
        self.cap = wl.recv_capacity(T, k, R)
        g = torch.Generator().manual_seed(seed)
        self.xs = [wl.make_x(g, T, H) for _ in range(steps)]
        self.topks = routings(T, k, E, [seed + 11 * i for i in range(steps)])
        self.xd = [x.to(DEV) for x in self.xs]
        self.td = [t.to(DEV) for t in self.topks]
        self.outs = [torch.empty(T, H, dtype=torch.bfloat16, device=DEV) for _ in range(steps)]
        self.status = moe.new_status(DEV)
        self.ws = torch.empty(moe.moe_get_layout_workspace_size(T, E, R), dtype=torch.uint8, device=DEV)
        self.lay = moe.moe_get_layout(self.td[0], E, R, workspace=self.ws, status=self.status)
        self.d = moe.moe_dispatch(self.xd[0], self.td[0], None, E, R, self.lay.token_dst_row, self.cap,
                                  quantize_fp8=fp8, status=self.status)

    def step(self, i, fused=False):
        moe, E, R = self.moe, self.E, self.R
        if fused:
            moe.moe_layout_dispatch(self.xd[i], self.td[i], None, E, R, self.cap, quantize_fp8=self.fp8,
                                    x_scales=self.d.x_scales, layout=self.lay, workspace=self.ws, out=self.d,
                                    status=self.status)
        else:
            moe.moe_get_layout(self.td[i], E, R, out=self.lay, workspace=self.ws, status=self.status)
            moe.moe_dispatch(self.xd[i], self.td[i], None, E, R, self.lay.token_dst_row, self.cap, out=self.d,
                             quantize_fp8=self.fp8, status=self.status)
        if self.fp8:
            moe.moe_combine_fp8(self.d.recv_x, self.d.recv_x_scales, self.lay.token_dst_row, out=self.outs[i],
                                status=self.status)
        else:
            moe.moe_combine(self.d.recv_x, self.lay.token_dst_row, out=self.outs[i], status=self.status)

    def check(self):
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0
        for i, (x, topk) in enumerate(zip(self.xs, self.topks)):
            ref = expected_chain(x, topk, self.E, self.R, self.cap, self.fp8)
            np.testing.assert_array_equal(bits16(self.outs[i]), ref, err_msg=f"step {i}")
        for o in self.outs:
            o.fill_(0)


SHAPES = [
    (1000, 1024, 8, 64, 8),     # several layout tiles (cooperative layout launch)
    (96, 7168, 8, 256, 8),      # one layout tile (an ordinary launch, overlapped like the rest)
]


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("T,H,k,E,R", SHAPES)
def test_steps_in_one_graph(moe, T, H, k, E, R, fp8):
    p = Pipeline(moe, T, H, k, E, R, fp8, 3, T + H)
    for i in range(3):       # outside the graph first: warm-up, no attribute set during capture
        p.step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(3):
            p.step(i)
    for _ in range(2):
        g.replay()
        p.check()


@pytest.mark.parametrize("T,H,k,E,R", SHAPES)
def test_steps_eager_on_side_stream(moe, T, H, k, E, R):
    p = Pipeline(moe, T, H, k, E, R, False, 3, 7 * T)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            for i in range(3):
                p.step(i)
    torch.cuda.current_stream().wait_stream(s)
    p.check()


@pytest.mark.parametrize("T,fp8", [(128, False), (2000, False), (2000, True)])
def test_layout_dispatch_steps_in_one_graph(moe, T, fp8):
    # moe_layout_dispatch: one fused launch (T <= 1024), or the layout and then a dispatch
    # that loads input rows before its dependency wait and balances its tail through a
    # counter in the layout workspace
    p = Pipeline(moe, T, 7168, 8, 256, 8, fp8, 3, 5 + T)
    for i in range(3):
        p.step(i, fused=True)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(3):
            p.step(i, fused=True)
    for _ in range(2):
        g.replay()
        p.check()
