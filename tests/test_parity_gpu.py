"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact for layout outputs, receive rows (bf16 bits, E4M3 codes, fp32
scales) and metadata; combine within 1e-2 relative / 1e-3 absolute, and
additionally bit-exact, since both sides add the same fp32 values in the same
(ascending-rank) order and round once. Full configuration sizes, ragged token
counts across tile and chunk boundaries, masked / invalid routing, capacity
overflow, maximum sizes, determinism and the bounded-wait failure path.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_moe_get_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
POISON_BF16 = 0x7FBF          # a NaN pattern no kernel writes on purpose
LAYOUT_KEYS = ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "rank_prefix",
               "expert_prefix", "token_dst_row")


@pytest.fixture(scope="module")
def moe():
    from combine_moe_get_gb300 import binding
    return binding


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def gpu_layout(moe, topk_cpu, E, R, **kw):
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk_cpu.to(DEV), E, R, status=status, **kw)
    torch.cuda.synchronize()
    out = {k: getattr(lay, k).cpu().numpy() for k in LAYOUT_KEYS}
    return lay, out, int(status.item())


def assert_layout_equal(got, ref):
    for key in LAYOUT_KEYS:
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)


def topk_for(w: wl.Workload, T=None):
    return wl.make_inputs(w, with_partial=False, num_tokens=T).topk_idx


# ------------------------------------------------------------------ layout

@pytest.mark.parametrize("layout_mode", [0, 1, 2])   # 1: never the cluster mode; 2: only the lookback modes
@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed", "decode", "layout_2048", "layout_2048_1m"])
def test_layout_parity_configs(moe, name, layout_mode):
    w = wl.CONFIGS[name]
    topk = topk_for(w)
    _, got, st = gpu_layout(moe, topk, w.num_experts, w.num_ranks, layout_mode=layout_mode)
    ref = oracle.layout(topk.numpy(), w.num_experts, w.num_ranks)
    assert st == 0 and ref["flags"] == 0
    assert_layout_equal(got, ref)


SHAPES = [  # (T, k, E, R)
    (1, 2, 16, 4), (31, 2, 16, 4), (32, 8, 256, 8), (33, 8, 256, 8), (127, 8, 256, 256), (128, 8, 256, 64),
    (129, 8, 256, 8), (1000, 6, 48, 3), (257, 1, 8, 1), (300, 32, 64, 8), (513, 5, 20, 5), (4097, 8, 256, 8),
    (200, 32, 8192, 1024), (130, 3, 7, 7), (4096, 8, 256, 8), (4095, 4, 16, 4), (3000, 8, 1024, 1024),
]


@pytest.mark.parametrize("layout_mode", [0, 1])   # 1: never the cluster mode
@pytest.mark.parametrize("T,k,E,R", SHAPES)
@pytest.mark.parametrize("mask", [0.0, 0.3])
def test_layout_parity_shapes(moe, T, k, E, R, mask, layout_mode):
    g = torch.Generator().manual_seed(T * 131 + k * 7 + R)
    topk = wl.make_topk_uniform(g, T, E, min(k, E)) if k <= E else None
    if mask:
        topk = wl.mask_random_lanes(g, topk, mask)
    _, got, st = gpu_layout(moe, topk, E, R, layout_mode=layout_mode)
    ref = oracle.layout(topk.numpy(), E, R)
    assert st == 0
    assert_layout_equal(got, ref)


def test_layout_many_distinct_shapes_in_one_process(moe):
    # more distinct (experts, ranks, top-k) shapes than the library's per-shape launch caches hold (16):
    # each shape's shared memory differs, the caches wrap, and every layout is still the oracle's
    T = 16384        # 128 tiles of 128 tokens: the cooperative lookback, whose co-residency is cached per shape
    shapes = [(E, R, k) for (E, R) in ((64, 8), (128, 16), (256, 8), (256, 32), (512, 64)) for k in (2, 4, 6, 8)]
    assert len(set(shapes)) > 16
    for i, (E, R, k) in enumerate(shapes + shapes[:3]):     # and back to the first shapes after the wrap
        g = torch.Generator().manual_seed(1000 + i)
        topk = wl.make_topk_uniform(g, T, E, k)
        _, got, st = gpu_layout(moe, topk, E, R)
        assert st == 0, (E, R, k)
        assert_layout_equal(got, oracle.layout(topk.numpy(), E, R))


@pytest.mark.parametrize("T,k,E,R,mask", [
    (1 << 20, 8, 256, 8, 0.0),          # 8192 tiles of 128 tokens: more than fit on the GPU at once
    (1 << 20, 8, 2048, 256, 0.1),
    (400_000, 6, 48, 3, 0.3),            # a ragged last tile, ranks not a power of two
    (300_001, 2, 16, 4, 0.0),
    (250_000, 32, 8192, 1024, 0.2),      # the largest rank and expert counts
])
def test_layout_scan_mode_parity(moe, T, k, E, R, mask):
    # the scan mode (per-tile counts, a scan per rank, then the rows; no waits) against the oracle, and
    # against the lookback modes (layout_mode 2) on the same inputs; twice, reusing the workspace
    g = torch.Generator().manual_seed(T % 1009 + R)
    topk = wl.mask_random_lanes(g, wl.make_topk_uniform(g, T, E, k), mask) if mask else wl.make_topk_uniform(g, T, E, k)
    ref = oracle.layout(topk.numpy(), E, R)
    assert ref["flags"] == 0
    for _ in range(2):
        _, got, st = gpu_layout(moe, topk, E, R)
        assert st == 0
        assert_layout_equal(got, ref)
    _, got2, st2 = gpu_layout(moe, topk, E, R, layout_mode=2)
    assert st2 == 0
    assert_layout_equal(got2, ref)


def test_layout_scan_mode_bad_entries_and_duplicates(moe):
    g = torch.Generator().manual_seed(71)
    T, k, E, R = 300_000, 8, 64, 8
    topk = torch.randint(0, E, (T, k), generator=g)          # duplicates inside rows
    topk[::13] = -1
    topk[12345, 3] = E + 1
    topk[299_999, 0] = -5
    _, got, st = gpu_layout(moe, topk, E, R)
    ref = oracle.layout(topk.numpy(), E, R)
    assert ref["flags"] & oracle.ORACLE_BAD_TOPK and st == moe.MOE_ERR_BAD_TOPK
    assert_layout_equal(got, ref)


def test_layout_duplicates_all_masked_and_bad_entries(moe):
    g = torch.Generator().manual_seed(5)
    T, k, E, R = 700, 8, 64, 8
    topk = torch.randint(0, E, (T, k), generator=g)          # with duplicates inside rows
    topk[::7] = -1                                            # all-masked tokens
    topk[3, 2] = E + 5                                        # invalid entries
    topk[400, 0] = -9
    _, got, st = gpu_layout(moe, topk, E, R)
    ref = oracle.layout(topk.numpy(), E, R)
    assert ref["flags"] & oracle.ORACLE_BAD_TOPK
    assert st == moe.MOE_ERR_BAD_TOPK
    assert_layout_equal(got, ref)


def test_layout_empty(moe):
    topk = torch.zeros(0, 8, dtype=torch.int64)
    lay, got, st = gpu_layout(moe, topk, 256, 8)
    assert st == 0
    for key in ("num_tokens_per_rank", "num_tokens_per_expert", "rank_prefix", "expert_prefix"):
        assert np.all(got[key] == 0), key


def test_layout_deterministic_and_reuses_workspace(moe):
    w = wl.CONFIGS["skewed"]
    topk = topk_for(w).to(DEV)
    ws = torch.empty(moe.moe_get_layout_workspace_size(w.num_tokens, w.num_experts, w.num_ranks),
                     dtype=torch.uint8, device=DEV)
    outs = []
    for _ in range(3):
        ws.fill_(0xAB)   # the call must clear its own workspace
        status = moe.new_status(DEV)
        lay = moe.moe_get_layout(topk, w.num_experts, w.num_ranks, workspace=ws, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append({k: getattr(lay, k).cpu().numpy() for k in LAYOUT_KEYS})
    for o in outs[1:]:
        assert_layout_equal(o, outs[0])


@pytest.mark.parametrize("T", [65536, 1 << 20])
def test_layout_lookback_modes_report_timeout(moe, T):
    # 512 tiles (too many for the direct sweep: cooperative lookback) and 8192 tiles (more than fit on the GPU:
    # ticket lookback); one tile never publishes, the bounded waits expire, the context stays usable
    k, E, R = 8, 256, 8
    topk = wl.make_topk_uniform(torch.Generator().manual_seed(T % 997), T, E, k)
    _, _, st = gpu_layout(moe, topk, E, R, wait_timeout_ns=20_000_000, test_unpublished_tile=3)
    assert st == moe.MOE_ERR_TIMEOUT
    _, got, st = gpu_layout(moe, topk, E, R)
    assert st == 0
    assert_layout_equal(got, oracle.layout(topk.numpy(), E, R))


def test_layout_bounded_wait_reports_timeout(moe):
    # one tile never publishes its scan status: the tiles after it give up after
    # the bounded wait and report MOE_ERR_TIMEOUT; the context stays usable
    T, k, E, R = 1024, 8, 256, 8
    topk = wl.make_topk_uniform(torch.Generator().manual_seed(1), T, E, k)
    _, _, st = gpu_layout(moe, topk, E, R, wait_timeout_ns=20_000_000, test_unpublished_tile=2)
    assert st == moe.MOE_ERR_TIMEOUT
    # last tile unpublished: nobody waits on it, the count step must still notice
    _, _, st = gpu_layout(moe, topk, E, R, wait_timeout_ns=20_000_000, test_unpublished_tile=7)
    assert st == moe.MOE_ERR_TIMEOUT
    _, got, st = gpu_layout(moe, topk, E, R)
    assert st == 0
    assert_layout_equal(got, oracle.layout(topk.numpy(), E, R))


# ------------------------------------------------------------------ dispatch

def run_dispatch(moe, inp, E, R, fp8, cap=None, guard=0, weights=True):
    T, H = inp.x.shape
    k = inp.topk_idx.shape[1]
    cap = wl.recv_capacity(T, k, R) if cap is None else cap
    topk = inp.topk_idx.to(DEV)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk, E, R, status=status)
    rows = cap + guard
    out = moe.Dispatched(
        recv_x=(torch.full((rows, H), 0xEE, dtype=torch.uint8, device=DEV) if fp8 else
                torch.full((rows, H), POISON_BF16, dtype=torch.int16, device=DEV).view(torch.bfloat16)),
        recv_x_scales=torch.full((rows, H // 128), -1.0, device=DEV) if fp8 else None,
        recv_topk_idx=torch.full((rows, k), -7, dtype=torch.int64, device=DEV),
        recv_topk_weights=torch.full((rows, k), -7.0, device=DEV),
        recv_src_idx=torch.full((rows,), -7, dtype=torch.int32, device=DEV),
        x_scales=torch.full((T, H // 128), -1.0, device=DEV) if fp8 else None)
    w = inp.topk_weights.to(DEV) if weights else None
    moe.moe_dispatch(inp.x.to(DEV), topk, w, E, R, lay.token_dst_row, cap, quantize_fp8=fp8, out=out, status=status)
    torch.cuda.synchronize()
    return lay, out, int(status.item())


def check_dispatch(moe, inp, E, R, fp8, weights=True):
    lay, out, st = run_dispatch(moe, inp, E, R, fp8, weights=weights)
    assert st == 0
    topk = inp.topk_idx.numpy()
    ref_lay = oracle.layout(topk, E, R)
    N = ref_lay["num_recv"]
    cap = out.recv_x.shape[0]
    ref = oracle.dispatch(bits16(inp.x), topk, inp.topk_weights.numpy() if weights else None, E, R,
                          ref_lay["token_dst_row"], N, fp8=fp8)
    assert int(lay.rank_prefix[-1].item()) == N
    if fp8:
        np.testing.assert_array_equal(out.recv_x[:N].cpu().numpy(), ref["recv_x"])
        np.testing.assert_array_equal(out.recv_x_scales[:N].cpu().numpy().view(np.uint32),
                                      ref["recv_x_scales"].view(np.uint32))
        np.testing.assert_array_equal(out.x_scales.cpu().numpy().view(np.uint32), ref["x_scales"].view(np.uint32))
        assert np.all(out.recv_x[N:].cpu().numpy() == 0xEE)
    else:
        np.testing.assert_array_equal(bits16(out.recv_x[:N]), ref["recv_x"])
        assert np.all(bits16(out.recv_x[N:]) == POISON_BF16)
    np.testing.assert_array_equal(out.recv_src_idx[:N].cpu().numpy(), ref["recv_src_idx"])
    np.testing.assert_array_equal(out.recv_topk_idx[:N].cpu().numpy(), ref["recv_topk_idx"])
    np.testing.assert_array_equal(out.recv_topk_weights[:N].cpu().numpy().view(np.uint32),
                                  ref["recv_topk_weights"].view(np.uint32))
    assert np.all(out.recv_src_idx[N:cap].cpu().numpy() == -7)


@pytest.mark.parametrize("name,fp8", [("tiny", False), ("tiny", True), ("dsv3", False), ("dsv3_fp8", True),
                                      ("skewed", False), ("skewed", True), ("decode", False), ("decode", True)])
def test_dispatch_parity_configs(moe, name, fp8):
    w = wl.CONFIGS[name]
    inp = wl.make_inputs(w, with_partial=False)
    check_dispatch(moe, inp, w.num_experts, w.num_ranks, fp8)


DISPATCH_SHAPES = [  # (T, H, k, E, R)
    (1, 128, 2, 16, 4), (33, 7168, 8, 256, 8), (129, 384, 8, 256, 256), (1000, 1024, 6, 48, 3),
    (77, 8, 2, 16, 4), (300, 4096, 32, 64, 8), (513, 7040, 5, 20, 5), (64, 16384, 8, 256, 8),
    (250, 7160, 8, 256, 64),
]


@pytest.mark.parametrize("T,H,k,E,R", DISPATCH_SHAPES)
@pytest.mark.parametrize("fp8", [False, True])
def test_dispatch_parity_shapes(moe, T, H, k, E, R, fp8):
    if fp8 and H % 128:
        pytest.skip("FP8 needs H % 128 == 0")
    g = torch.Generator().manual_seed(T + H + k)
    x = wl.make_x(g, T, H)
    topk = wl.mask_random_lanes(g, wl.make_topk_uniform(g, T, E, k), 0.2)
    inp = wl.Inputs(None, x, topk, wl.make_weights(g, T, k), None)
    check_dispatch(moe, inp, E, R, fp8, weights=(T % 2 == 0))


def test_dispatch_fp8_special_blocks(moe):
    # zero blocks (scale 0, codes 0), tiny values (E4M3 subnormals), exact ties, large magnitudes
    T, H, E, R, k = 8, 1024, 16, 4, 2
    x = torch.zeros(T, H)
    x[1] = torch.linspace(-3e-3, 3e-3, H)
    x[2, :128] = 1.0
    x[2, 128:256] = torch.tensor([448.0 * (i + 1) / 128 for i in range(128)])
    x[3] = torch.randn(H, generator=torch.Generator().manual_seed(0)) * 1e4
    x[4, ::2] = -2.0 ** -20
    x[5] = torch.arange(H) % 17 - 8.0
    inp = wl.Inputs(None, x.to(torch.bfloat16), torch.tensor([[0, 5], [1, 2], [3, 15], [8, 9], [0, 12],
                                                                [4, 7], [-1, -1], [11, 10]]),
                    torch.full((T, k), 0.5), None)
    check_dispatch(moe, inp, E, R, True)


def _e4m3_midpoints():
    vals = []
    for code in range(1, 126):
        e, m = code >> 3, code & 7
        lo = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        c2 = code + 1
        e2, m2 = c2 >> 3, c2 & 7
        hi = (m2 / 8.0) * 2.0 ** -6 if e2 == 0 else (1 + m2 / 8.0) * 2.0 ** (e2 - 7)
        vals.append((lo + hi) / 2)
    return torch.tensor(vals, dtype=torch.float64)


def test_dispatch_fp8_rounding_boundaries(moe):
    # blocks whose quotients x / scale land on or next to E4M3 rounding midpoints, for
    # scales that are powers of two (exact ties) and scales that are not
    g = torch.Generator().manual_seed(11)
    mids = _e4m3_midpoints()
    amaxes = [1.75, 3.5, 2.625, 0.4375, 5.25, 1.3125, 2.0 ** -3 * 1.75, 448.0, 7.0, 0.21875, 3.0, 1.0]
    T, H = 96, 1024
    x = torch.zeros(T, H, dtype=torch.float64)
    for t in range(T):
        for b in range(H // 128):
            amax = amaxes[(t * 8 + b) % len(amaxes)]
            s = amax / 448.0
            pick = mids[torch.randint(0, len(mids), (127,), generator=g)]
            sign = torch.where(torch.rand(127, generator=g) < 0.5, -1.0, 1.0)
            blk = (pick * s * sign).to(torch.bfloat16).to(torch.float64)
            # nudge some entries one bf16 step either way
            nud = torch.randint(-1, 2, (127,), generator=g)
            bits = blk.to(torch.bfloat16).view(torch.int16).to(torch.int32) + nud * (blk != 0).to(torch.int32)
            blk = bits.to(torch.int16).view(torch.bfloat16).to(torch.float64).clamp(-amax, amax)
            x[t, b * 128:(b + 1) * 128 - 1] = blk
            x[t, (b + 1) * 128 - 1] = amax
    E, R, k = 64, 8, 4
    topk = wl.make_topk_uniform(g, T, E, k)
    inp = wl.Inputs(None, x.to(torch.bfloat16), topk, wl.make_weights(g, T, k), None)
    check_dispatch(moe, inp, E, R, True)


def check_dispatch_fp8_input(moe, topk, E, R, H, seed, weights=True):
    g = np.random.default_rng(seed)
    T, k = topk.shape
    codes = g.integers(0, 256, (T, H), dtype=np.uint8)          # any byte pattern: this is a copy
    scales = g.standard_normal((T, H // 128)).astype(np.float32)
    w = wl.make_weights(torch.Generator().manual_seed(seed), T, k)
    topk_d = topk.to(DEV)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk_d, E, R, status=status)
    cap = wl.recv_capacity(T, k, R)
    d = moe.moe_dispatch(torch.from_numpy(codes).to(DEV), topk_d, w.to(DEV) if weights else None, E, R,
                         lay.token_dst_row, cap, x_scales=torch.from_numpy(scales).to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_lay = oracle.layout(topk.numpy(), E, R)
    N = ref_lay["num_recv"]
    ref = oracle.dispatch_fp8_input(codes, scales, topk.numpy(), w.numpy() if weights else None, E, R,
                                    ref_lay["token_dst_row"], N)
    np.testing.assert_array_equal(d.recv_x[:N].cpu().numpy(), ref["recv_x"])
    np.testing.assert_array_equal(d.recv_x_scales[:N].cpu().numpy().view(np.uint32),
                                  ref["recv_x_scales"].view(np.uint32))
    np.testing.assert_array_equal(d.recv_src_idx[:N].cpu().numpy(), ref["recv_src_idx"])
    np.testing.assert_array_equal(d.recv_topk_idx[:N].cpu().numpy(), ref["recv_topk_idx"])
    np.testing.assert_array_equal(d.recv_topk_weights[:N].cpu().numpy().view(np.uint32),
                                  ref["recv_topk_weights"].view(np.uint32))


@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed", "decode"])
def test_dispatch_fp8_input_parity_configs(moe, name):
    w = wl.CONFIGS[name]
    check_dispatch_fp8_input(moe, topk_for(w), w.num_experts, w.num_ranks, w.hidden, 17)


@pytest.mark.parametrize("T,H,k,E,R", [(1, 128, 2, 16, 4), (129, 384, 8, 256, 256), (300, 16384, 6, 48, 3),
                                       (77, 7040, 5, 20, 5)])
def test_dispatch_fp8_input_parity_shapes(moe, T, H, k, E, R):
    g = torch.Generator().manual_seed(T + H)
    topk = wl.mask_random_lanes(g, wl.make_topk_uniform(g, T, E, k), 0.2)
    check_dispatch_fp8_input(moe, topk, E, R, H, T, weights=(T % 2 == 1))


@pytest.mark.parametrize("T,H", [(4096, 1024), (8192, 512), (3000, 384)])
def test_dispatch_fp8_many_rows_per_cta_small_rows(moe, T, H):
    # one slice per row and tens of rows per CTA: workers claim items several input-ring slots ahead
    # of the producer, so every wait must first see the row's load armed
    g = torch.Generator().manual_seed(T + H)
    E, R, k = 64, 8, 8
    topk = wl.make_topk_uniform(g, T, E, k)
    inp = wl.Inputs(None, wl.make_x(g, T, H), topk, wl.make_weights(g, T, k), None)
    check_dispatch(moe, inp, E, R, True)


@pytest.mark.parametrize("T,H,k,E,R,mode", [(4096, 7168, 8, 256, 8, "bf16"), (2000, 1024, 8, 256, 8, "fp8in"),
                                            (3000, 512, 6, 48, 3, "bf16"), (100, 256, 8, 64, 8, "bf16")])
def test_dispatch_balanced_parity(moe, T, H, k, E, R, mode):
    # a balance counter changes which CTA copies which unit, never a byte; each call leaves it zero
    g = torch.Generator().manual_seed(T + H + k)
    topk = wl.mask_random_lanes(g, wl.make_topk_uniform(g, T, E, k), 0.15)
    w = wl.make_weights(g, T, k)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk.to(DEV), E, R, status=status)
    cap = wl.recv_capacity(T, k, R)
    ref_lay = oracle.layout(topk.numpy(), E, R)
    if mode == "fp8in":
        rng = np.random.default_rng(T)
        x = torch.from_numpy(rng.integers(0, 256, (T, H), dtype=np.uint8))
        sc = torch.from_numpy(rng.standard_normal((T, H // 128)).astype(np.float32))
        ref = oracle.dispatch_fp8_input(x.numpy(), sc.numpy(), topk.numpy(), w.numpy(), E, R, ref_lay["token_dst_row"], cap)
    else:
        x, sc = wl.make_x(g, T, H), None
        ref = oracle.dispatch(bits16(x), topk.numpy(), w.numpy(), E, R, ref_lay["token_dst_row"], cap)
    bal = moe.new_balance_counter(DEV)
    N = ref_lay["num_recv"]
    for _ in range(2):
        out = moe.moe_dispatch(x.to(DEV), topk.to(DEV), w.to(DEV), E, R, lay.token_dst_row, cap,
                               x_scales=None if sc is None else sc.to(DEV), balance=bal, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0 and bal.tolist() == [0, 0]
        if mode == "fp8in":
            np.testing.assert_array_equal(out.recv_x[:N].cpu().numpy(), ref["recv_x"][:N])
            np.testing.assert_array_equal(out.recv_x_scales[:N].cpu().numpy().view(np.uint32),
                                          ref["recv_x_scales"][:N].view(np.uint32))
        else:
            np.testing.assert_array_equal(bits16(out.recv_x[:N]), ref["recv_x"][:N])
        np.testing.assert_array_equal(out.recv_src_idx[:N].cpu().numpy(), ref["recv_src_idx"][:N])
        np.testing.assert_array_equal(out.recv_topk_idx[:N].cpu().numpy(), ref["recv_topk_idx"][:N])


@pytest.mark.parametrize("T,H,k,E,R,balanced", [
    (1000, 7168, 8, 256, 8, True),      # pool on, first stage loads spill into the pool: dealt units prefetched only
    (3000, 7168, 8, 256, 8, True),      # pool on, pool units prefetched too
    (3000, 7168, 8, 256, 8, False),     # every unit dealt
    (16384, 7168, 8, 256, 8, True),     # more input than the prefetch budget: part of each CTA's units prefetched
    (700, 4104, 6, 48, 3, True),        # rows not a multiple of the chunk alignment, ranks not a power of two
])
def test_dispatch_l2_prefetch_regimes(moe, T, H, k, E, R, balanced):
    # the dispatch prefetches its input rows into L2 in every regime of the prefetch rule (with or
    # without a pool, within or beyond the L2 budget); results are the oracle's, call after call
    g = torch.Generator().manual_seed(7 * T + H + k)
    topk = wl.mask_random_lanes(g, wl.make_topk_uniform(g, T, E, k), 0.1)
    w = wl.make_weights(g, T, k)
    x = wl.make_x(g, T, H)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk.to(DEV), E, R, status=status)
    cap = wl.recv_capacity(T, k, R)
    ref_lay = oracle.layout(topk.numpy(), E, R)
    ref = oracle.dispatch(bits16(x), topk.numpy(), w.numpy(), E, R, ref_lay["token_dst_row"], cap)
    N = ref_lay["num_recv"]
    bal = moe.new_balance_counter(DEV) if balanced else None
    xd, td, wd = x.to(DEV), topk.to(DEV), w.to(DEV)
    for _ in range(2):
        out = moe.moe_dispatch(xd, td, wd, E, R, lay.token_dst_row, cap, balance=bal, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        if bal is not None:
            assert bal.tolist() == [0, 0]
        np.testing.assert_array_equal(bits16(out.recv_x[:N]), ref["recv_x"][:N])
        np.testing.assert_array_equal(out.recv_src_idx[:N].cpu().numpy(), ref["recv_src_idx"][:N])
        np.testing.assert_array_equal(out.recv_topk_idx[:N].cpu().numpy(), ref["recv_topk_idx"][:N])
        np.testing.assert_array_equal(out.recv_topk_weights[:N].cpu().numpy().view(np.uint32),
                                      ref["recv_topk_weights"][:N].view(np.uint32))


def test_dispatch_capacity_overflow_writes_nothing_beyond(moe):
    w = wl.CONFIGS["tiny"]
    inp = wl.make_inputs(w, with_partial=False)
    ref = oracle.layout(inp.topk_idx.numpy(), w.num_experts, w.num_ranks)
    N = ref["num_recv"]
    cap, guard = N - 9, 16
    lay, out, st = run_dispatch(moe, inp, w.num_experts, w.num_ranks, False, cap=cap, guard=guard)
    assert st == moe.MOE_ERR_CAPACITY
    assert np.all(bits16(out.recv_x[cap:]) == POISON_BF16)
    assert np.all(out.recv_src_idx[cap:].cpu().numpy() == -7)
    d = oracle.dispatch(bits16(inp.x), inp.topk_idx.numpy(), inp.topk_weights.numpy(), w.num_experts, w.num_ranks,
                        ref["token_dst_row"], cap)
    np.testing.assert_array_equal(bits16(out.recv_x[:cap]), d["recv_x"])


def test_dispatch_deterministic(moe):
    w = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(w, with_partial=False, num_tokens=1024)
    a = run_dispatch(moe, inp, w.num_experts, w.num_ranks, True)[1]
    b = run_dispatch(moe, inp, w.num_experts, w.num_ranks, True)[1]
    assert torch.equal(a.recv_x, b.recv_x) and torch.equal(a.recv_x_scales, b.recv_x_scales)


# ------------------------------------------------------------------ combine

def check_combine(moe, topk, partial, E, R):
    topk_d = topk.to(DEV)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk_d, E, R, status=status)
    out = moe.moe_combine(partial.to(DEV), lay.token_dst_row, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_lay = oracle.layout(topk.numpy(), E, R)
    ref, flags = oracle.combine(bits16(partial), ref_lay["token_dst_row"])
    assert flags == 0
    got = bits16(out)
    # the stated gate: 1e-2 relative / 1e-3 absolute in bf16
    g32 = (got.astype(np.uint32) << 16).view(np.float32)
    r32 = (ref.astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_allclose(g32, r32, rtol=1e-2, atol=1e-3)
    # and the stronger one: same fp32 additions in the same order, one rounding
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed", "decode"])
def test_combine_parity_configs(moe, name):
    w = wl.CONFIGS[name]
    inp = wl.make_inputs(w)
    check_combine(moe, inp.topk_idx, inp.partial, w.num_experts, w.num_ranks)


@pytest.mark.parametrize("T,H,k,E,R", DISPATCH_SHAPES)
def test_combine_parity_shapes(moe, T, H, k, E, R):
    g = torch.Generator().manual_seed(7 * T + H)
    topk = wl.mask_random_lanes(g, wl.make_topk_uniform(g, T, E, k), 0.2)
    partial = wl.make_partial(g, wl.recv_capacity(T, k, R), H)
    check_combine(moe, topk, partial, E, R)


@pytest.mark.parametrize("T,H,k,E,R", [(0, 256, 8, 64, 8), (1, 512, 2, 16, 4), (5, 1024, 8, 256, 8),
                                       (300, 7168, 8, 256, 8), (4096, 7168, 8, 256, 8), (2000, 1536, 6, 48, 3)])
def test_combine_balanced_parity(moe, T, H, k, E, R):
    # a balance counter changes which CTA reduces which token, never a result; each call leaves it zero
    g = torch.Generator().manual_seed(11 * T + H)
    topk = wl.mask_random_lanes(g, wl.make_topk_uniform(g, T, E, k), 0.2)
    partial = wl.make_partial(g, max(wl.recv_capacity(T, k, R), 1), H)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk.to(DEV), E, R, status=status)
    bal = moe.new_balance_counter(DEV)
    ref, flags = oracle.combine(bits16(partial), oracle.layout(topk.numpy(), E, R)["token_dst_row"])
    assert flags == 0
    pd = partial.to(DEV)
    for _ in range(3):
        out, _ = moe.moe_combine_ex(pd, lay.token_dst_row, balance=bal, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert bal.tolist() == [0, 0]
        np.testing.assert_array_equal(bits16(out), ref)


@pytest.mark.parametrize("name", ["dsv3", "skewed"])
def test_combine_right_behind_a_new_layout(moe, name):
    # The combine prefetches its first rows into L2 before its dependency wait, from row lists the
    # previous grid may still be writing. Here that grid is a layout of a different routing writing
    # the same buffers in place (launched back to back, each allowed to overlap the one before):
    # every result must still be the oracle's for the routing of the moment.
    w = wl.CONFIGS[name]
    E, R, H = w.num_experts, w.num_ranks, w.hidden
    T, k = w.num_tokens, w.num_topk
    g = torch.Generator().manual_seed(99)
    routings = [wl.make_inputs(w, with_partial=False).topk_idx, wl.make_topk_uniform(g, T, E, k),
                wl.mask_random_lanes(g, wl.make_topk_uniform(g, T, E, k), 0.3)]
    partial = wl.make_partial(g, wl.recv_capacity(T, k, R), H)
    pd = partial.to(DEV)
    lay = moe.Layout.empty(T, k, E, R, DEV)
    ws = torch.empty(max(16, moe.moe_get_layout_workspace_size(T, E, R)), dtype=torch.uint8, device=DEV)
    status = moe.new_status(DEV)
    bal = moe.new_balance_counter(DEV)
    seq = routings + routings[::-1]
    topk_d = [t.to(DEV) for t in seq]
    outs = [torch.empty(T, H, dtype=torch.bfloat16, device=DEV) for _ in seq]
    torch.cuda.synchronize()
    for topk, out in zip(topk_d, outs):     # nothing but these kernels on the stream
        moe.moe_get_layout(topk, E, R, out=lay, workspace=ws, status=status)
        moe.moe_combine_ex(pd, lay.token_dst_row, out=out, balance=bal, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert bal.tolist() == [0, 0]
    pbits = bits16(partial)
    for topk, out in zip(seq, outs):
        ref, flags = oracle.combine(pbits, oracle.layout(topk.numpy(), E, R)["token_dst_row"])
        assert flags == 0
        np.testing.assert_array_equal(bits16(out), ref)


def test_combine_weighted_balanced_parity(moe):
    # weighted rows and combined top-k weights with a balance counter: the oracle's results, counter left zero
    w = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(w)
    E, R = w.num_experts, w.num_ranks
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(inp.topk_idx.to(DEV), E, R, status=status)
    N = int(lay.rank_prefix[-1].item())
    g = torch.Generator().manual_seed(17)
    row_w = torch.rand(inp.partial.shape[0], generator=g)
    rtw = torch.rand(inp.partial.shape[0], w.num_topk, generator=g)
    ref_lay = oracle.layout(inp.topk_idx.numpy(), E, R)
    ref, cref, flags = oracle.combine_weighted(bits16(inp.partial), ref_lay["token_dst_row"], row_w.numpy(),
                                               rtw.numpy())
    assert flags == 0
    bal = moe.new_balance_counter(DEV)
    for _ in range(2):
        out, cw = moe.moe_combine_ex(inp.partial.to(DEV), lay.token_dst_row, row_weights=row_w.to(DEV),
                                     recv_topk_weights=rtw.to(DEV), balance=bal, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0 and bal.tolist() == [0, 0] and N > 0
        np.testing.assert_array_equal(bits16(out), ref)
        np.testing.assert_array_equal(cw.cpu().numpy().view(np.uint32), cref.view(np.uint32))


@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed", "decode"])
def test_combine_ex_parity_configs(moe, name):
    w = wl.CONFIGS[name]
    inp = wl.make_inputs(w)
    g = torch.Generator().manual_seed(5)
    topk = wl.mask_random_lanes(g, inp.topk_idx, 0.1)
    topk_d = topk.to(DEV)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk_d, w.num_experts, w.num_ranks, status=status)
    cap = inp.partial.shape[0]
    d = moe.moe_dispatch(inp.x.to(DEV), topk_d, inp.topk_weights.to(DEV), w.num_experts, w.num_ranks,
                         lay.token_dst_row, cap, status=status)
    row_w = (torch.rand(cap, generator=g) * 2 - 0.5).to(DEV)
    out, cw = moe.moe_combine_ex(inp.partial.to(DEV), lay.token_dst_row, row_weights=row_w,
                                 recv_topk_weights=d.recv_topk_weights, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_lay = oracle.layout(topk.numpy(), w.num_experts, w.num_ranks)
    N = ref_lay["num_recv"]
    rtw = d.recv_topk_weights.cpu().numpy()
    rtw[N:] = 0.0
    ref_out, ref_cw, flags = oracle.combine_weighted(bits16(inp.partial), ref_lay["token_dst_row"],
                                                     row_w.cpu().numpy(), rtw)
    assert flags == 0
    got = bits16(out)
    g32 = (got.astype(np.uint32) << 16).view(np.float32)
    r32 = (ref_out.astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_allclose(g32, r32, rtol=1e-2, atol=1e-3)
    np.testing.assert_array_equal(got, ref_out)
    np.testing.assert_array_equal(cw.cpu().numpy().view(np.uint32), ref_cw.view(np.uint32))
    # the combined weights are the routing weights of the valid entries
    expect = np.where(topk.numpy() >= 0, inp.topk_weights.numpy(), 0.0).astype(np.float32)
    np.testing.assert_array_equal(cw.cpu().numpy(), expect)


def test_combine_ex_without_options_is_combine(moe):
    w = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(w, num_tokens=1000)
    topk_d = inp.topk_idx.to(DEV)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk_d, w.num_experts, w.num_ranks, status=status)
    part = inp.partial.to(DEV)
    a, cw = moe.moe_combine_ex(part, lay.token_dst_row, status=status)
    b = moe.moe_combine(part, lay.token_dst_row, status=status)
    torch.cuda.synchronize()
    assert cw is None and torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_combine_partial_rows_short_reports_capacity(moe):
    w = wl.CONFIGS["tiny"]
    inp = wl.make_inputs(w)
    topk = inp.topk_idx.to(DEV)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk, w.num_experts, w.num_ranks, status=status)
    N = int(lay.rank_prefix[-1].item())
    moe.moe_combine(inp.partial[: N - 3].to(DEV), lay.token_dst_row, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == moe.MOE_ERR_CAPACITY


# ------------------------------------------------------------------ composite

def test_dispatch_then_combine_identity_expert(moe):
    # expert = identity times the row's local weights; weights sum to 1, so combine
    # gives x back within two bf16 roundings; and with partial = recv_x, D_t * x_t exactly
    w = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(w, with_partial=False, num_tokens=2048)
    lay, out, st = run_dispatch(moe, inp, w.num_experts, w.num_ranks, False)
    assert st == 0
    N = int(lay.rank_prefix[-1].item())
    rx = out.recv_x[:N]
    partial = (rx.float() * out.recv_topk_weights[:N].sum(dim=1, keepdim=True)).to(torch.bfloat16)
    status = moe.new_status(DEV)
    y = moe.moe_combine(partial, lay.token_dst_row, status=status).float().cpu()
    x = inp.x.float()
    assert torch.all((y - x).abs() <= 2.0 ** -7 * x.abs() * 1.01)
    y2 = moe.moe_combine(rx, lay.token_dst_row, status=status).cpu()
    D = lay.is_token_in_rank.sum(dim=1).float().cpu()
    assert torch.equal(y2.view(torch.int16), (x * D[:, None]).to(torch.bfloat16).view(torch.int16))
    torch.cuda.synchronize()
    assert int(status.item()) == 0


# ------------------------------------------------------------------ combine of E4M3 partial rows

def _fp8_rows(seed, rows, H):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, (rows, H), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38          # no NaN codes
    scales = (rng.standard_normal((rows, H // 128)) * 2.0 ** rng.integers(-6, 6, (rows, H // 128))).astype(np.float32)
    return codes, scales


def check_combine_fp8(moe, topk, E, R, H, seed):
    topk_d = topk.to(DEV)
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk_d, E, R, status=status)
    rows = wl.recv_capacity(topk.shape[0], topk.shape[1], R)
    codes, scales = _fp8_rows(seed, max(rows, 1), H)
    out = moe.moe_combine_fp8(torch.from_numpy(codes).to(DEV), torch.from_numpy(scales).to(DEV), lay.token_dst_row,
                              status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_lay = oracle.layout(topk.numpy(), E, R)
    ref, flags = oracle.combine_fp8(codes, scales, ref_lay["token_dst_row"])
    assert flags == 0
    got = bits16(out)
    g32 = (got.astype(np.uint32) << 16).view(np.float32)
    r32 = (ref.astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_allclose(g32, r32, rtol=1e-2, atol=1e-3)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("name", ["dsv3", "skewed", "decode"])
def test_combine_fp8_parity_configs(moe, name):
    w = wl.CONFIGS[name]
    check_combine_fp8(moe, topk_for(w), w.num_experts, w.num_ranks, w.hidden, 23)


@pytest.mark.parametrize("T,H,k,E,R", [(1, 512, 2, 16, 4), (33, 7168, 8, 256, 8), (129, 1024, 8, 256, 256),
                                       (1000, 1536, 6, 48, 3), (300, 4096, 32, 64, 8), (64, 16384, 8, 256, 8)])
def test_combine_fp8_parity_shapes(moe, T, H, k, E, R):
    g = torch.Generator().manual_seed(3 * T + H)
    topk = wl.mask_random_lanes(g, wl.make_topk_uniform(g, T, E, k), 0.2)
    check_combine_fp8(moe, topk, E, R, H, T + k)


@pytest.mark.parametrize("name", ["skewed", "dsv3", "decode"])
def test_combine_fp8_balanced_parity(moe, name):
    # moe_combine_fp8_ex with a balance counter (a pool on the long skewed batch, none on the shorter ones):
    # the oracle's result bit for bit, the counter left zero, call after call
    w = wl.CONFIGS[name]
    topk = topk_for(w)
    E, R, H = w.num_experts, w.num_ranks, w.hidden
    lay_ref = oracle.layout(topk.numpy(), E, R)
    rows = wl.recv_capacity(w.num_tokens, w.num_topk, R)
    rng = np.random.default_rng(23)
    codes = rng.integers(0, 256, (rows, H), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x01          # no NaN codes
    scales = rng.uniform(0.001, 2.0, (rows, H // 128)).astype(np.float32)
    ref, flags = oracle.combine_fp8(codes, scales, lay_ref["token_dst_row"])
    assert flags == 0
    status = moe.new_status(DEV)
    lay = moe.moe_get_layout(topk.to(DEV), E, R, status=status)
    bal = moe.new_balance_counter(DEV)
    cd, sd = torch.from_numpy(codes).to(DEV), torch.from_numpy(scales).to(DEV)
    for _ in range(2):
        out = moe.moe_combine_fp8(cd, sd, lay.token_dst_row, balance=bal, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0 and bal.tolist() == [0, 0]
        np.testing.assert_array_equal(bits16(out), ref)


def test_fp8_dispatch_then_fp8_combine(moe):
    # identity experts on FP8 rows: the GPU result equals the oracle's combine of the oracle's dispatch
    w = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(w, with_partial=False, num_tokens=1024)
    lay, out, st = run_dispatch(moe, inp, w.num_experts, w.num_ranks, True)
    assert st == 0
    N = int(lay.rank_prefix[-1].item())
    status = moe.new_status(DEV)
    y = moe.moe_combine_fp8(out.recv_x[:N].contiguous(), out.recv_x_scales[:N].contiguous(), lay.token_dst_row,
                            status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    topk = inp.topk_idx.numpy()
    ref_lay = oracle.layout(topk, w.num_experts, w.num_ranks)
    d = oracle.dispatch(bits16(inp.x), topk, None, w.num_experts, w.num_ranks, ref_lay["token_dst_row"], N, fp8=True)
    ref, _ = oracle.combine_fp8(d["recv_x"], d["recv_x_scales"], ref_lay["token_dst_row"])
    np.testing.assert_array_equal(bits16(y), ref)
