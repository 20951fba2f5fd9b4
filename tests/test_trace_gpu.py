"""The tracing build (libmoe_get_trace.so, compiled with MOE_PROFILE).

Every warp of every launch leaves exactly one timer record (one per CTA index
and warp index, the same warp count in every CTA, all warps of a CTA on one
SM, start <= end); the cluster layout, dispatch and combine kernels add one
record per phase per CTA, contiguous and inside the lifetime of the CTA's
warp 0; a dependent launch never starts before the launch it follows;
records past the buffer are counted, not written; stopping stops them; and
tracing changes no result: the outputs are the oracle's.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_moe_get_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
LAYOUT_IDS = {1, 2, 3, 12}          # tiles, direct, cluster, rows after tiles
SCAN_IDS = {4, 5, 6}                # count, scan, rows (the scan mode)
EXPAND_IDS = {7, 8}
DISPATCH_IDS = {9, 10}
COMBINE_IDS = {11}


@pytest.fixture(scope="module")
def moe():
    from combine_moe_get_gb300 import binding, build
    tl = binding.load_library(build.build_trace())
    with binding.using(tl):
        yield binding
        binding.trace_enable(None, None)


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Trace:
    """Records of the launches made inside the block."""

    def __init__(self, moe, capacity=1 << 20, what=None):
        self.moe = moe
        self.what = moe.TRACE_WARPS | moe.TRACE_PHASES if what is None else what
        self.buf = torch.zeros(capacity * moe.TRACE_RECORD.itemsize, dtype=torch.uint8, device=DEV)
        self.count = torch.zeros(1, dtype=torch.int32, device=DEV)

    def __enter__(self):
        self.moe.trace_enable(self.buf, self.count, self.what)
        return self

    def __exit__(self, *exc):
        self.moe.trace_enable(None, None)
        torch.cuda.synchronize()

    def records(self) -> np.ndarray:
        return self.moe.trace_read(self.buf, self.count)


def check_launch(r: np.ndarray) -> tuple[int, int]:
    """One launch's records: every (CTA, warp) once, the same warps in every CTA,
    one SM per CTA. Returns (CTAs, warps per CTA)."""
    assert len(r) > 0
    assert np.all(r["start_ns"] > 0) and np.all(r["start_ns"] <= r["end_ns"])
    assert int(r["end_ns"].max() - r["start_ns"].min()) < 1_000_000_000
    ctas = int(r["cta"].max()) + 1
    warps = int(r["warp"].max()) + 1
    assert len(r) == ctas * warps
    key = r["cta"].astype(np.int64) * warps + r["warp"]
    assert np.array_equal(np.sort(key), np.arange(ctas * warps))
    for c in np.unique(r["cta"])[:64]:
        assert len(np.unique(r["sm"][r["cta"] == c])) == 1
    return ctas, warps


def by_kernel(r: np.ndarray) -> dict:
    """Per kernel id, its per-warp records (phase records left out)."""
    r = r[r["warp"] < 0x10000]
    return {int(k): r[r["kernel"] == k] for k in np.unique(r["kernel"])}


def check_phases(moe, rec: np.ndarray, kernel: int, ctas: int):
    """The kernel's phase records: every phase of every CTA once, each CTA's
    phases contiguous, on the SM of its warps and inside its warp 0's life."""
    warps, phases = moe.trace_split(rec[rec["kernel"] == kernel])
    n = len(moe.TRACE_PHASE_NAMES[kernel])
    assert len(phases) == ctas * n
    for c in range(ctas):
        p = phases[phases["cta"] == c]
        p = p[np.argsort(p["warp"])]
        assert p["warp"].tolist() == [moe.TRACE_PHASE + i for i in range(1, n + 1)]
        assert np.all(p["start_ns"] <= p["end_ns"])
        assert np.array_equal(p["start_ns"][1:], p["end_ns"][:-1])
        w0 = warps[(warps["cta"] == c) & (warps["warp"] == 0)]
        assert len(w0) == 1
        assert w0["start_ns"][0] <= p["start_ns"][0] and p["end_ns"][-1] <= w0["end_ns"][0]
        assert np.all(p["sm"] == w0["sm"][0])
    return phases


def test_trace_dsv3_step(moe):
    # layout -> dispatch -> combine at the DeepSeek-V3 shape, one trace per call and one over all three
    w = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(w)
    E, R = w.num_experts, w.num_ranks
    T, k = inp.topk_idx.shape
    cap = wl.recv_capacity(T, k, R)
    topk, x, pd = inp.topk_idx.to(DEV), inp.x.to(DEV), inp.partial.to(DEV)
    status = moe.new_status(DEV)
    ids = {}
    for name, expect in (("layout", LAYOUT_IDS), ("dispatch", DISPATCH_IDS), ("combine", COMBINE_IDS)):
        with Trace(moe) as tr:
            if name == "layout":
                lay = moe.moe_get_layout(topk, E, R, status=status)
            elif name == "dispatch":
                out = moe.moe_dispatch(x, topk, inp.topk_weights.to(DEV), E, R, lay.token_dst_row, cap,
                                       status=status)
            else:
                comb = moe.moe_combine(pd, lay.token_dst_row, status=status)
        rec = tr.records()
        assert int(tr.count.item()) == len(rec)
        kinds = by_kernel(rec)
        assert set(kinds) <= expect and kinds, (name, set(kinds))
        for kid, r in kinds.items():
            ctas, _ = check_launch(r)
            if kid in moe.TRACE_PHASE_NAMES:
                check_phases(moe, rec, kid, ctas)
            else:
                assert not np.any((rec["kernel"] == kid) & (rec["warp"] >= moe.TRACE_PHASE))
        ids[name] = set(kinds)
    assert int(status.item()) == 0

    ref_lay = oracle.layout(inp.topk_idx.numpy(), E, R)
    np.testing.assert_array_equal(lay.token_dst_row.cpu().numpy(), ref_lay["token_dst_row"])
    N = ref_lay["num_recv"]
    ref = oracle.dispatch(bits16(inp.x), inp.topk_idx.numpy(), inp.topk_weights.numpy(), E, R,
                          ref_lay["token_dst_row"], N)
    np.testing.assert_array_equal(bits16(out.recv_x[:N]), ref["recv_x"])
    np.testing.assert_array_equal(out.recv_src_idx[:N].cpu().numpy(), ref["recv_src_idx"])
    ref_c, flags = oracle.combine(bits16(inp.partial), ref_lay["token_dst_row"])
    assert flags == 0
    np.testing.assert_array_equal(bits16(comb), ref_c)

    # the three calls back to back: each launch starts no earlier than the one before it started
    with Trace(moe) as tr:
        lay2 = moe.moe_get_layout(topk, E, R, status=status)
        moe.moe_dispatch(x, topk, inp.topk_weights.to(DEV), E, R, lay2.token_dst_row, cap, status=status)
        moe.moe_combine(pd, lay2.token_dst_row, status=status)
    kinds = by_kernel(tr.records())
    first = {kk: int(r["start_ns"].min()) for kk, r in kinds.items()}
    lay_id, = ids["layout"] - {12} or ids["layout"]
    dis_id, = ids["dispatch"]
    assert first[lay_id] <= first[dis_id] <= first[11]
    if 12 in kinds:
        assert first[lay_id] <= first[12] <= first[dis_id]


@pytest.mark.parametrize("name", ["dsv3_fp8", "decode"])
def test_trace_quantising_dispatch(moe, name):
    w = wl.CONFIGS[name]
    inp = wl.make_inputs(w, with_partial=False)
    E, R = w.num_experts, w.num_ranks
    T, k = inp.topk_idx.shape
    topk = inp.topk_idx.to(DEV)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk, E, R, status=status)
    with Trace(moe) as tr:
        out = moe.moe_dispatch(inp.x.to(DEV), topk, None, E, R, lay.token_dst_row, wl.recv_capacity(T, k, R),
                               quantize_fp8=True, status=status)
    rec = tr.records()
    kinds = by_kernel(rec)
    assert set(kinds) <= DISPATCH_IDS and kinds
    for kid, r in kinds.items():
        ctas, _ = check_launch(r)
        check_phases(moe, rec, kid, ctas)
    assert int(status.item()) == 0
    ref_lay = oracle.layout(inp.topk_idx.numpy(), E, R)
    N = ref_lay["num_recv"]
    ref = oracle.dispatch(bits16(inp.x), inp.topk_idx.numpy(), None, E, R, ref_lay["token_dst_row"], N, fp8=True)
    np.testing.assert_array_equal(out.recv_x[:N].cpu().numpy(), ref["recv_x"])
    np.testing.assert_array_equal(out.recv_x_scales[:N].cpu().numpy().view(np.uint32),
                                  ref["recv_x_scales"].view(np.uint32))


@pytest.mark.parametrize("layout_mode,expect", [(0, SCAN_IDS), (2, {1, 12})])
def test_trace_large_layout(moe, layout_mode, expect):
    # 2^20 tokens, 2048 experts: the scan mode's three launches, or the lookback tiles and their rows
    w = wl.CONFIGS["layout_2048_1m"]
    topk_cpu = wl.make_inputs(w, with_partial=False).topk_idx
    E, R = w.num_experts, w.num_ranks
    status = moe.new_status(DEV)
    with Trace(moe) as tr:
        lay = moe.moe_get_layout(topk_cpu.to(DEV), E, R, status=status, layout_mode=layout_mode)
    kinds = by_kernel(tr.records())
    assert set(kinds) == expect
    shapes = {kk: check_launch(r) for kk, r in kinds.items()}
    if layout_mode == 0:
        assert shapes[5][0] == R          # one CTA per rank scans that rank's column
        assert shapes[4][0] > 152         # more tiles than fit on the GPU at once
    assert int(status.item()) == 0
    ref = oracle.layout(topk_cpu.numpy(), E, R)
    np.testing.assert_array_equal(lay.token_dst_row.cpu().numpy(), ref["token_dst_row"])
    np.testing.assert_array_equal(lay.num_tokens_per_expert.cpu().numpy(), ref["num_tokens_per_expert"])


def test_trace_expand_layout(moe):
    w = wl.CONFIGS["dsv3"]
    topk_cpu = wl.make_inputs(w, with_partial=False).topk_idx
    E, R = w.num_experts, w.num_ranks
    topk = topk_cpu.to(DEV)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk, E, R, status=status)
    with Trace(moe) as tr:
        rows = moe.moe_get_expand_layout(topk, lay.expert_prefix, E, status=status)
    kinds = by_kernel(tr.records())
    assert set(kinds) <= EXPAND_IDS and len(kinds) == 1
    check_launch(next(iter(kinds.values())))
    assert int(status.item()) == 0
    np.testing.assert_array_equal(rows.cpu().numpy(), oracle.expand_layout(topk_cpu.numpy(), E)["token_expert_row"])


def test_trace_overflow_and_stop(moe):
    # a buffer of 4 records: the rest are counted, not written; after stopping, nothing is counted
    w = wl.CONFIGS["tiny"]
    inp = wl.make_inputs(w)
    E, R = w.num_experts, w.num_ranks
    topk = inp.topk_idx.to(DEV)
    size = moe.TRACE_RECORD.itemsize
    buf = torch.full((64 * size,), 0xAB, dtype=torch.uint8, device=DEV)
    count = torch.zeros(1, dtype=torch.int32, device=DEV)
    status = moe.new_status(DEV)
    moe.trace_enable(buf[: 4 * size], count)
    lay = moe.moe_get_layout(topk, E, R, status=status)
    out = moe.moe_combine(inp.partial.to(DEV), lay.token_dst_row, status=status)
    moe.trace_enable(None, None)
    torch.cuda.synchronize()
    n = int(count.item())
    assert n > 4
    assert np.all(buf[4 * size:].cpu().numpy() == 0xAB)
    rec = moe.trace_read(buf[: 4 * size], count)
    assert len(rec) == 4 and set(np.unique(rec["kernel"]).tolist()) <= LAYOUT_IDS | COMBINE_IDS | {9}
    moe.moe_combine(inp.partial.to(DEV), lay.token_dst_row, out=out, status=status)
    torch.cuda.synchronize()
    assert int(count.item()) == n
    assert int(status.item()) == 0
    ref_c, _ = oracle.combine(bits16(inp.partial), oracle.layout(inp.topk_idx.numpy(), E, R)["token_dst_row"])
    np.testing.assert_array_equal(bits16(out), ref_c)


def test_trace_warps_or_phases_alone(moe):
    # what = warps only: no phase record; phases only: exactly the phase records, nothing else
    w = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(w)
    E, R = w.num_experts, w.num_ranks
    T, k = inp.topk_idx.shape
    topk, x, pd = inp.topk_idx.to(DEV), inp.x.to(DEV), inp.partial.to(DEV)
    status = moe.new_status(DEV)

    def step():
        lay = moe.moe_get_layout(topk, E, R, status=status)
        out = moe.moe_dispatch(x, topk, None, E, R, lay.token_dst_row, wl.recv_capacity(T, k, R), status=status)
        comb = moe.moe_combine(pd, lay.token_dst_row, status=status)
        return lay, out, comb

    step()
    torch.cuda.synchronize()
    with Trace(moe, what=moe.TRACE_WARPS) as tr:
        step()
    full = tr.records()
    warps, phases = moe.trace_split(full)
    assert len(phases) == 0 and len(warps) == len(full) > 0
    shapes = {kid: check_launch(r) for kid, r in by_kernel(full).items()}
    with Trace(moe, what=moe.TRACE_PHASES) as tr:
        lay, out, comb = step()
    rec = tr.records()
    warps, phases = moe.trace_split(rec)
    assert len(warps) == 0
    expect = sum(ctas * len(moe.TRACE_PHASE_NAMES[kid]) for kid, (ctas, _) in shapes.items()
                 if kid in moe.TRACE_PHASE_NAMES)
    assert len(phases) == int(tr.count.item()) == expect
    for kid in set(np.unique(phases["kernel"]).tolist()):
        ph = phases[phases["kernel"] == kid]
        n = len(moe.TRACE_PHASE_NAMES[kid])
        for c in np.unique(ph["cta"]):
            p = ph[ph["cta"] == c]
            p = p[np.argsort(p["warp"])]
            assert p["warp"].tolist() == [moe.TRACE_PHASE + i for i in range(1, n + 1)]
            assert np.array_equal(p["start_ns"][1:], p["end_ns"][:-1]) and np.all(p["start_ns"] <= p["end_ns"])
    assert int(status.item()) == 0
    ref_lay = oracle.layout(inp.topk_idx.numpy(), E, R)
    ref_c, _ = oracle.combine(bits16(inp.partial), ref_lay["token_dst_row"])
    np.testing.assert_array_equal(bits16(comb), ref_c)

