"""The benchmark's timed calls, at the benchmark's sizes, against the oracle.

bench.py times one step as moe_layout_dispatch (the layout, then a dispatch
that loads input rows before the layout has finished and balances its tail
through the layout workspace; one fused launch at decode size) followed by
moe_combine_ex with a balance counter, captured once in a CUDA graph and
replayed. This file runs those same calls through bench.py's own Step object
on the DeepSeek-V3 shape (4096 tokens over 8 ranks, cluster layout), the
skewed shape (8192 tokens over 64 ranks with Zipf expert popularity, direct
layout) and the decode shape (128 tokens over 256 ranks): eagerly twice in a
row, then as graph replays, and then every variant bench.py times alone.
Each result is compared with the CPU oracle: layout, indices, metadata and
rows bit for bit; combine outputs within the stated bf16 gate (1e-2 relative,
1e-3 absolute) and bit for bit (same fp32 additions in the same order)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bench
import oracle
from combine_moe_get_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

LAYOUT_KEYS = ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "rank_prefix",
               "expert_prefix", "token_dst_row")


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32_bits(t) -> np.ndarray:
    a = t.detach().cpu().numpy() if isinstance(t, torch.Tensor) else t
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


class Case:
    """A workload, bench.py's Step over it on cuda:0, and the oracle's chain
    (layout, bf16 dispatch, combine) over the same seeded inputs."""

    def __init__(self, name):
        from combine_moe_get_gb300 import binding as moe
        self.moe = moe
        self.w = w = wl.CONFIGS[name]
        self.inp = inp = wl.make_inputs(w)
        self.st = bench.Step(moe, w, inp, torch.device("cuda", 0))
        self.topk = inp.topk_idx.numpy()
        self.xb = bits16(inp.x)
        self.wts = inp.topk_weights.numpy()
        self.pb = bits16(inp.partial)
        self.lay = oracle.layout(self.topk, w.num_experts, w.num_ranks)
        assert self.lay["flags"] == 0
        self.N = self.lay["num_recv"]
        self.disp = oracle.dispatch(self.xb, self.topk, self.wts, w.num_experts, w.num_ranks,
                                    self.lay["token_dst_row"], self.st.cap)
        assert self.disp["flags"] == 0
        self.out, flags = oracle.combine(self.pb, self.lay["token_dst_row"])
        assert flags == 0
        self._fp8 = None

    def fp8(self):
        if self._fp8 is None:
            w = self.w
            self._fp8 = oracle.dispatch(self.xb, self.topk, self.wts, w.num_experts, w.num_ranks,
                                        self.lay["token_dst_row"], self.st.cap, fp8=True)
            assert self._fp8["flags"] == 0
        return self._fp8

    def poison(self):
        st = self.st
        for t in (st.lay.token_dst_row, st.lay.is_token_in_rank, st.lay.num_tokens_per_rank,
                  st.lay.num_tokens_per_expert, st.lay.rank_prefix, st.lay.expert_prefix):
            t.fill_(0x55)
        st.disp.recv_x.view(torch.int16).fill_(0x7FBF)
        st.disp.recv_src_idx.fill_(-7)
        st.disp.recv_topk_idx.fill_(-7)
        st.disp.recv_topk_weights.fill_(-7.0)
        st.disp8.recv_x.fill_(0xEE)
        st.disp8.recv_x_scales.fill_(-1.0)
        st.disp8.x_scales.fill_(-1.0)
        st.out.view(torch.int16).fill_(0x7FBF)

    def check_layout(self):
        for key in LAYOUT_KEYS:
            np.testing.assert_array_equal(getattr(self.st.lay, key).cpu().numpy(), self.lay[key], err_msg=key)

    def check_meta(self, ref):
        n, d = self.N, self.st.disp
        np.testing.assert_array_equal(d.recv_src_idx[:n].cpu().numpy(), ref["recv_src_idx"][:n])
        np.testing.assert_array_equal(d.recv_topk_idx[:n].cpu().numpy(), ref["recv_topk_idx"][:n])
        np.testing.assert_array_equal(f32_bits(d.recv_topk_weights[:n]), f32_bits(ref["recv_topk_weights"][:n]))
        assert np.all(d.recv_src_idx[n:].cpu().numpy() == -7), "a row beyond N was written"

    def check_dispatch_bf16(self):
        n = self.N
        got = bits16(self.st.disp.recv_x)
        np.testing.assert_array_equal(got[:n], self.disp["recv_x"][:n])
        assert np.all(got[n:] == 0x7FBF), "a row beyond N was written"
        self.check_meta(self.disp)

    def check_combine(self, ref):
        got = bits16(self.st.out)
        g32 = (got.astype(np.uint32) << 16).view(np.float32)
        r32 = (ref.astype(np.uint32) << 16).view(np.float32)
        np.testing.assert_allclose(g32, r32, rtol=1e-2, atol=1e-3)
        np.testing.assert_array_equal(got, ref)

    def check_step(self):
        torch.cuda.synchronize()
        self.moe.check_status(self.st.status, "step")
        assert self.st.bal.tolist() == [0, 0], "combine balance counter not left zero"
        self.check_layout()
        self.check_dispatch_bf16()
        self.check_combine(self.out)


@pytest.fixture(scope="module", params=["dsv3", "skewed", "decode"])
def case(request):
    c = Case(request.param)
    yield c
    del c.st
    torch.cuda.empty_cache()


def test_timed_step_eager_twice(case):
    for _ in range(2):
        case.poison()
        case.st.layout_dispatch()
        case.st.combine()
        case.check_step()


def test_timed_step_graph_replays(case):
    st = case.st
    st.layout_dispatch()      # every call once outside the capture, as bench.py does
    st.combine()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.layout_dispatch()
        st.combine()
    for _ in range(3):
        case.poison()
        g.replay()
        case.check_step()


def test_timed_separate_calls(case):
    # the per-kernel breakdown: moe_get_layout, moe_dispatch_ex (balanced), moe_combine_ex (balanced)
    case.poison()
    case.st.layout()
    case.st.dispatch()
    case.st.combine()
    case.check_step()
    assert case.st.bal_d.tolist() == [0, 0], "dispatch balance counter not left zero"


def test_timed_variants_fp8_dispatch_and_fp8_combine(case):
    st, ref = case.st, case.fp8()
    case.poison()
    st.layout()
    st.dispatch(fp8=True)
    torch.cuda.synchronize()
    case.moe.check_status(st.status, "fp8 dispatch")
    n = case.N
    np.testing.assert_array_equal(st.disp8.recv_x[:n].cpu().numpy(), ref["recv_x"][:n])
    assert np.all(st.disp8.recv_x[n:].cpu().numpy() == 0xEE)
    np.testing.assert_array_equal(f32_bits(st.disp8.recv_x_scales[:n]), f32_bits(ref["recv_x_scales"][:n]))
    np.testing.assert_array_equal(f32_bits(st.disp8.x_scales), f32_bits(ref["x_scales"]))
    case.check_meta(ref)
    st.combine_fp8()          # E4M3 partial rows: the FP8 dispatch's own rows and scales
    torch.cuda.synchronize()
    case.moe.check_status(st.status, "fp8 combine")
    assert st.bal.tolist() == [0, 0], "combine balance counter not left zero"
    assert st.bal_d.tolist() == [0, 0], "dispatch balance counter not left zero"
    out, flags = oracle.combine_fp8(ref["recv_x"][:n], ref["recv_x_scales"][:n], case.lay["token_dst_row"])
    assert flags == 0
    case.check_combine(out)


def test_timed_variants_fp8_input_dispatch(case):
    st, w = case.st, case.w
    case.poison()
    st.layout()
    st.dispatch_fp8_input()
    torch.cuda.synchronize()
    case.moe.check_status(st.status, "fp8 pass-through dispatch")
    codes = (case.inp.x.view(torch.int16) & 0xFF).to(torch.uint8).numpy()   # bench.py's E4M3 input rows
    scales = np.ones((w.num_tokens, w.hidden // 128), np.float32)
    ref = oracle.dispatch_fp8_input(codes, scales, case.topk, case.wts, w.num_experts, w.num_ranks,
                                    case.lay["token_dst_row"], st.cap)
    assert ref["flags"] == 0
    n = case.N
    np.testing.assert_array_equal(st.disp8.recv_x[:n].cpu().numpy(), ref["recv_x"][:n])
    np.testing.assert_array_equal(f32_bits(st.disp8.recv_x_scales[:n]), f32_bits(ref["recv_x_scales"][:n]))
    case.check_meta(ref)


def test_timed_variants_weighted_and_unbalanced_combine(case):
    st = case.st
    case.poison()
    st.layout()
    st.dispatch()
    st.combine_weighted()
    torch.cuda.synchronize()
    case.moe.check_status(st.status, "weighted combine")
    row_w = torch.rand(st.cap, generator=torch.Generator().manual_seed(case.w.seed + 2)).numpy()
    np.testing.assert_array_equal(f32_bits(st.row_w), f32_bits(row_w))     # bench.py's seeded row weights
    out, cw, flags = oracle.combine_weighted(case.pb, case.lay["token_dst_row"], row_w,
                                             case.disp["recv_topk_weights"])
    assert flags == 0
    case.check_combine(out)
    np.testing.assert_array_equal(f32_bits(st.cw), f32_bits(cw))
    assert st.bal.tolist() == [0, 0]
    st.out.view(torch.int16).fill_(0x7FBF)
    st.combine_unbalanced()
    torch.cuda.synchronize()
    case.moe.check_status(st.status, "static combine")
    case.check_combine(case.out)


def test_pipelined_steps(case):
    # bench.py's back-to-back measurement: three buffer sets cycled in one graph with no flush in
    # between; it raises unless every set reproduces its first output bit for bit, and the timed
    # set's output is the oracle's
    if case.w.name != "dsv3":
        pytest.skip("the benchmark runs the pipelined steps at the DeepSeek-V3 shape")
    case.poison()
    res = bench.measure_pipelined(case.moe, case.st, case.w, torch.device("cuda", 0), 0, rounds=2, reps=2)
    assert res["steps_per_graph"] == 6 and res["ms_per_step_mean"] > 0
    case.check_step()
