"""Parity of expand mode (one receive row per valid top-k entry, grouped by
expert) through the C ABI with the CPU oracle.

Bit-exact for the expand rows, the receive rows (bf16 bits, E4M3 codes, fp32
scales) and the metadata; combine within 1e-2 relative / 1e-3 absolute and,
since both sides add the same fp32 values in the same (ascending-row) order
and round once, bit-exact as well. Ragged token counts across the 256-token
tiles, the largest expert count, duplicates, masked and invalid entries, an
empty batch, workspace reuse and the bounded-wait failure path.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_moe_get_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
POISON_BF16 = 0x7FBF


@pytest.fixture(scope="module")
def moe():
    from combine_moe_get_gb300 import binding
    return binding


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def gpu_expand(moe, topk_cpu, E, R, **kw):
    """Layout, then the expand rows; returns (layout, token_expert_row on device, status)."""
    topk = topk_cpu.to(DEV)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk, E, R, status=status)
    rows = torch.full(tuple(topk.shape), -77, dtype=torch.int32, device=DEV)
    moe.moe_get_expand_layout(topk, lay.expert_prefix, E, out=rows, status=status, **kw)
    torch.cuda.synchronize()
    return lay, rows, int(status.item())


def check_expand_layout(moe, topk, E, R, layout_mode=0):
    _, rows, st = gpu_expand(moe, topk, E, R, layout_mode=layout_mode)
    ref = oracle.expand_layout(topk.numpy(), E)
    assert st == (moe.MOE_ERR_BAD_TOPK if ref["flags"] & oracle.ORACLE_BAD_TOPK else 0)
    np.testing.assert_array_equal(rows.cpu().numpy(), ref["token_expert_row"])


# ------------------------------------------------------------------ expand layout

@pytest.mark.parametrize("layout_mode", [0, 1])   # 1: never the cluster mode
@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed", "decode", "layout_2048", "layout_2048_1m"])
def test_expand_layout_parity_configs(moe, name, layout_mode):
    w = wl.CONFIGS[name]
    check_expand_layout(moe, wl.make_inputs(w, with_partial=False).topk_idx, w.num_experts, w.num_ranks, layout_mode)


EXPAND_SHAPES = [  # (T, k, E, R)
    (1, 2, 16, 4), (255, 8, 256, 8), (256, 8, 256, 64), (257, 8, 256, 256), (511, 6, 48, 3), (513, 1, 8, 1),
    (4097, 8, 256, 8), (300, 32, 64, 8), (200, 32, 8192, 1024), (1030, 3, 7, 7), (2500, 5, 20, 5),
    (4096, 8, 256, 8), (4096, 32, 1024, 8), (3999, 1, 1024, 1024),
]


@pytest.mark.parametrize("layout_mode", [0, 1])   # 1: never the cluster mode
@pytest.mark.parametrize("T,k,E,R", EXPAND_SHAPES)
@pytest.mark.parametrize("mask", [0.0, 0.3])
def test_expand_layout_parity_shapes(moe, T, k, E, R, mask, layout_mode):
    g = torch.Generator().manual_seed(T * 17 + k * 5 + E)
    topk = wl.make_topk_uniform(g, T, E, k)
    if mask:
        topk = wl.mask_random_lanes(g, topk, mask)
    check_expand_layout(moe, topk, E, R, layout_mode)


def test_expand_layout_duplicates_all_masked_and_bad_entries(moe):
    g = torch.Generator().manual_seed(21)
    T, k, E, R = 900, 8, 64, 8
    topk = torch.randint(0, E, (T, k), generator=g)          # duplicates inside rows
    topk[::5] = -1                                            # all-masked tokens
    topk[11, 3] = E + 2                                       # invalid entries
    topk[600, 7] = -3
    topk[300:340] = 5                                         # one expert named k times by 40 tokens
    check_expand_layout(moe, topk, E, R)


def test_expand_layout_empty(moe):
    topk = torch.zeros(0, 8, dtype=torch.int64, device=DEV)
    prefix = torch.zeros(257, dtype=torch.int32, device=DEV)
    status = moe.new_status(DEV)
    rows = moe.moe_get_expand_layout(topk, prefix, 256, status=status)
    torch.cuda.synchronize()
    assert rows.shape == (0, 8) and int(status.item()) == 0


def test_expand_layout_deterministic_and_reuses_workspace(moe):
    w = wl.CONFIGS["skewed"]
    topk = wl.make_inputs(w, with_partial=False).topk_idx.to(DEV)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk, w.num_experts, w.num_ranks, status=status)
    ws = torch.empty(moe.moe_get_expand_layout_workspace_size(w.num_tokens, w.num_experts), dtype=torch.uint8,
                     device=DEV)
    outs = []
    for _ in range(3):
        ws.fill_(0xAB)    # the call must clear its own workspace
        outs.append(moe.moe_get_expand_layout(topk, lay.expert_prefix, w.num_experts, workspace=ws,
                                              status=status).cpu())
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_expand_layout_bounded_wait_reports_timeout(moe):
    # one tile never publishes its scan status: the tiles after it give up after the
    # bounded wait and report MOE_ERR_TIMEOUT; the context stays usable afterwards
    T, k, E, R = 2048, 8, 256, 8
    topk = wl.make_topk_uniform(torch.Generator().manual_seed(2), T, E, k)
    _, _, st = gpu_expand(moe, topk, E, R, wait_timeout_ns=20_000_000, test_unpublished_tile=3)
    assert st == moe.MOE_ERR_TIMEOUT
    check_expand_layout(moe, topk, E, R)


# ------------------------------------------------------------------ expand dispatch

MODES = ("bf16", "quantize_fp8", "fp8")


def run_expand_dispatch(moe, x, topk, w, E, R, mode, scales=None, balance=None):
    T, H = x.shape
    k = topk.shape[1]
    lay, rows, st = gpu_expand(moe, topk, E, R)
    assert st == 0
    cap = T * k + 8
    fp8_out = mode != "bf16"
    out = moe.Dispatched(
        recv_x=(torch.full((cap, H), 0xEE, dtype=torch.uint8, device=DEV) if fp8_out else
                torch.full((cap, H), POISON_BF16, dtype=torch.int16, device=DEV).view(torch.bfloat16)),
        recv_x_scales=torch.full((cap, H // 128), -1.0, device=DEV) if fp8_out else None,
        recv_topk_idx=torch.full((cap, k), -7, dtype=torch.int64, device=DEV),
        recv_topk_weights=torch.full((cap, k), -7.0, device=DEV),
        recv_src_idx=torch.full((cap,), -7, dtype=torch.int32, device=DEV),
        x_scales=(torch.full((T, H // 128), -1.0, device=DEV) if mode == "quantize_fp8" else
                  (scales.to(DEV) if mode == "fp8" else None)))
    status = moe.new_status(DEV)
    moe.moe_dispatch(x.to(DEV), topk.to(DEV), None if w is None else w.to(DEV), E, R, rows, cap,
                     quantize_fp8=mode == "quantize_fp8", x_scales=out.x_scales, expand=True, out=out,
                     balance=balance, status=status)
    torch.cuda.synchronize()
    return lay, rows, out, int(status.item())


def check_expand_dispatch(moe, topk, E, R, H, mode, seed, weights=True, balance=None):
    T, k = topk.shape
    g = torch.Generator().manual_seed(seed)
    w = wl.make_weights(g, T, k) if weights else None
    if mode == "fp8":
        rng = np.random.default_rng(seed)
        x_np = rng.integers(0, 256, (T, H), dtype=np.uint8)
        scales = torch.from_numpy(rng.standard_normal((T, H // 128)).astype(np.float32))
        x = torch.from_numpy(x_np)
        x_ref = x_np
    else:
        scales = None
        x = wl.make_x(g, T, H)
        x_ref = bits16(x)
    _, rows, out, st = run_expand_dispatch(moe, x, topk, w, E, R, mode, scales, balance)
    assert st == 0
    if balance is not None:
        assert balance.tolist() == [0, 0]
    ex = oracle.expand_layout(topk.numpy(), E)
    N = ex["num_recv"]
    ref = oracle.dispatch_expand(MODES.index(mode), x_ref, topk.numpy(), None if w is None else w.numpy(), E, R,
                                 ex["token_expert_row"], N, x_scales=None if scales is None else scales.numpy())
    assert ref["flags"] == 0
    if mode == "bf16":
        np.testing.assert_array_equal(bits16(out.recv_x[:N]), ref["recv_x"])
        assert np.all(bits16(out.recv_x[N:]) == POISON_BF16)
    else:
        np.testing.assert_array_equal(out.recv_x[:N].cpu().numpy(), ref["recv_x"])
        np.testing.assert_array_equal(out.recv_x_scales[:N].cpu().numpy().view(np.uint32),
                                      ref["recv_x_scales"].view(np.uint32))
        assert np.all(out.recv_x[N:].cpu().numpy() == 0xEE)
        if mode == "quantize_fp8":
            np.testing.assert_array_equal(out.x_scales.cpu().numpy().view(np.uint32),
                                          ref["x_scales"].view(np.uint32))
    np.testing.assert_array_equal(out.recv_src_idx[:N].cpu().numpy(), ref["recv_src_idx"])
    np.testing.assert_array_equal(out.recv_topk_idx[:N].cpu().numpy(), ref["recv_topk_idx"])
    np.testing.assert_array_equal(out.recv_topk_weights[:N].cpu().numpy().view(np.uint32),
                                  ref["recv_topk_weights"].view(np.uint32))
    assert np.all(out.recv_src_idx[N:].cpu().numpy() == -7)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed", "decode"])
def test_expand_dispatch_parity_configs(moe, name, mode):
    w = wl.CONFIGS[name]
    topk = wl.make_inputs(w, with_partial=False).topk_idx
    check_expand_dispatch(moe, topk, w.num_experts, w.num_ranks, w.hidden, mode, 31)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("T,H,k,E,R", [(1, 128, 2, 16, 4), (257, 384, 8, 256, 256), (300, 4096, 32, 64, 8),
                                       (513, 7040, 5, 20, 5), (77, 16384, 6, 48, 3)])
def test_expand_dispatch_parity_shapes(moe, T, H, k, E, R, mode):
    g = torch.Generator().manual_seed(T + 3 * H + k)
    topk = wl.mask_random_lanes(g, wl.make_topk_uniform(g, T, E, k), 0.2)
    check_expand_dispatch(moe, topk, E, R, H, mode, T + H, weights=(T % 2 == 1))


@pytest.mark.parametrize("mode", ["bf16", "fp8"])
def test_expand_dispatch_balanced_parity(moe, mode):
    # with a balance counter (a pool of units): the same bytes, and the counter left zero
    w = wl.CONFIGS["dsv3"]
    topk = wl.make_inputs(w, with_partial=False).topk_idx
    bal = moe.new_balance_counter(DEV)
    for seed in (41, 42):
        check_expand_dispatch(moe, topk, w.num_experts, w.num_ranks, w.hidden, mode, seed, balance=bal)


def test_expand_dispatch_duplicate_experts(moe):
    # a token naming one expert twice is copied to two rows, each with its own entry
    g = torch.Generator().manual_seed(4)
    topk = torch.randint(0, 32, (400, 8), generator=g)
    topk[::9] = -1
    check_expand_dispatch(moe, topk, 32, 4, 1024, "bf16", 4)
    check_expand_dispatch(moe, topk, 32, 4, 1024, "quantize_fp8", 5)


# ------------------------------------------------------------------ expand combine

def _check_close_and_exact(got_bits, ref_bits):
    g32 = (got_bits.astype(np.uint32) << 16).view(np.float32)
    r32 = (ref_bits.astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_allclose(g32, r32, rtol=1e-2, atol=1e-3)
    np.testing.assert_array_equal(got_bits, ref_bits)


@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed", "decode"])
def test_expand_combine_parity_configs(moe, name):
    w = wl.CONFIGS[name]
    inp = wl.make_inputs(w, with_partial=False)
    g = torch.Generator().manual_seed(9)
    topk = wl.mask_random_lanes(g, inp.topk_idx, 0.1)
    T, k = topk.shape
    _, rows, st = gpu_expand(moe, topk, w.num_experts, w.num_ranks)
    assert st == 0
    partial = wl.make_partial(g, T * k, w.hidden)
    status = moe.new_status(DEV)
    out = moe.moe_combine(partial.to(DEV), rows, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ex = oracle.expand_layout(topk.numpy(), w.num_experts)
    ref, flags = oracle.combine(bits16(partial), ex["token_expert_row"])
    assert flags == 0
    _check_close_and_exact(bits16(out), ref)


@pytest.mark.parametrize("name", ["dsv3", "skewed"])
def test_expand_weighted_combine_parity(moe, name):
    # dispatch in expand mode, weight each expert row by its entry's weight, reduce the
    # received weights: the combined weights are the routing weights of the valid entries
    w = wl.CONFIGS[name]
    inp = wl.make_inputs(w, with_partial=False, num_tokens=1536)
    g = torch.Generator().manual_seed(13)
    topk = wl.mask_random_lanes(g, inp.topk_idx, 0.15)
    T, k = topk.shape
    _, rows, out_d, st = run_expand_dispatch(moe, inp.x, topk, inp.topk_weights, w.num_experts, w.num_ranks, "bf16")
    assert st == 0
    N = int((topk >= 0).sum())
    partial = wl.make_partial(g, out_d.recv_x.shape[0], w.hidden).to(DEV)
    row_w = out_d.recv_topk_weights.clone()
    row_w[N:] = 0.0
    row_w = row_w.sum(dim=1).contiguous()
    rtw = out_d.recv_topk_weights.clone()
    rtw[N:] = 0.0
    status = moe.new_status(DEV)
    out, cw = moe.moe_combine_ex(partial, rows, row_weights=row_w, recv_topk_weights=rtw.contiguous(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ex = oracle.expand_layout(topk.numpy(), w.num_experts)
    ref_out, ref_cw, flags = oracle.combine_weighted(bits16(partial), ex["token_expert_row"], row_w.cpu().numpy(),
                                                     rtw.cpu().numpy())
    assert flags == 0
    _check_close_and_exact(bits16(out), ref_out)
    np.testing.assert_array_equal(cw.cpu().numpy().view(np.uint32), ref_cw.view(np.uint32))
    expect = np.where(topk.numpy() >= 0, inp.topk_weights.numpy(), 0.0).astype(np.float32)
    np.testing.assert_array_equal(cw.cpu().numpy(), expect)


def test_expand_identity_experts_return_count_times_x(moe):
    # partial = recv_x on the expand rows: every valid entry sends x_t back once, so the
    # combine returns bf16(n_t * x_t); with k = 4 entries all valid the sum is exact
    w = wl.CONFIGS["dsv3"]
    T, k = 3000, 4
    topk = wl.make_topk_uniform(torch.Generator().manual_seed(6), T, w.num_experts, k)
    x = wl.make_x(torch.Generator().manual_seed(7), T, w.hidden)
    _, rows, out_d, st = run_expand_dispatch(moe, x, topk, None, w.num_experts, w.num_ranks, "bf16")
    assert st == 0
    status = moe.new_status(DEV)
    y = moe.moe_combine(out_d.recv_x[: T * k].contiguous(), rows, status=status).cpu()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(y.view(torch.int16), (x.float() * 4).to(torch.bfloat16).view(torch.int16))
