"""Pins for the CPU oracle: each test checks it against something other than
itself -- the page's printed figures, closed forms, invariants, an
independent brute force, exhaustive enumeration, or a library routine.

All CPU; no GPU needed.
"""
from __future__ import annotations

import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import bruteforce as bf
from oracle.expected_topk import expected_topk_exact, get_expected_topk, variance_topk_exact
from combine_moe_get_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _random_small_case(seed: int):
    g = torch.Generator().manual_seed(seed)
    R = [1, 2, 3, 4, 8][seed % 5]
    m = [1, 2, 4][(seed // 5) % 3]
    E = R * m
    k = int(torch.randint(1, min(E, 8) + 1, (1,), generator=g))
    T = int(torch.randint(0, 65, (1,), generator=g))
    topk = wl.make_topk_uniform(g, T, E, k)
    if seed % 2:
        topk = wl.mask_random_lanes(g, topk, 0.25)
    w = wl.make_weights(g, T, k)
    H = 128 * int(torch.randint(1, 3, (1,), generator=g))
    x = wl.make_x(g, T, H)
    return topk, w, x, E, R


# ---------------------------------------------------------------- page figures / closed form

def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "expected_topk_pages.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                G, E, k, val, factor, note = line.split()
                rows.append((int(G), int(E), int(k), float(val), factor, note))
    return rows


def test_expected_topk_pages_worked_figures():
    rows = _golden_rows()
    assert len(rows) == 2
    for G, E, k, printed, factor, note in rows:
        exact = expected_topk_exact(E, G, k)
        if note == "approx":
            # one expert per rank: k distinct experts always land on k distinct ranks
            assert exact == k
            assert abs(float(exact) - printed) < 0.5
        else:
            # reproduce the page's own arithmetic (multiplier `factor`), and show the
            # formula gives a different value
            miss = Fraction(math.comb(E - E // G, k), math.comb(E, k))
            assert abs(int(factor) * float(1 - miss) - printed) < 0.01
            assert abs(float(exact) - 7.904810) < 1e-6


def _enumerate_distinct(E, G, k):
    m = E // G
    ds = [len({e // m for e in s}) for s in itertools.combinations(range(E), k)]
    n = len(ds)
    mean = Fraction(sum(ds), n)
    var = Fraction(sum(d * d for d in ds), n) - mean * mean
    return mean, var


@pytest.mark.parametrize("E,G,k", [(8, 4, 3), (12, 3, 4), (10, 5, 2), (16, 8, 5), (9, 9, 3), (6, 1, 2)])
def test_expected_topk_closed_form_vs_enumeration(E, G, k):
    mean, var = _enumerate_distinct(E, G, k)
    assert expected_topk_exact(E, G, k) == mean
    assert variance_topk_exact(E, G, k) == var


@pytest.mark.parametrize("name,T", [("tiny", None), ("dsv3", None), ("decode", None),
                                    ("layout_2048", None), ("layout_2048", 1 << 16)])
def test_oracle_mean_distinct_ranks_vs_closed_form(name, T):
    w = wl.CONFIGS[name]
    inp = wl.make_inputs(w, with_partial=False, num_tokens=T)
    if not w.layout_only:
        inp.x = None
    lay = oracle.layout(inp.topk_idx.numpy(), w.num_experts, w.num_ranks)
    D = lay["is_token_in_rank"].sum(axis=1).astype(np.float64)
    mu = float(expected_topk_exact(w.num_experts, w.num_ranks, w.num_topk))
    var = float(variance_topk_exact(w.num_experts, w.num_ranks, w.num_topk))
    n = D.size
    if var == 0.0:
        assert np.all(D == mu)
    else:
        se = math.sqrt(var / n)
        assert abs(D.mean() - mu) < 5 * se, (D.mean(), mu, se)
        # sample variance within a loose band of the exact variance
        assert 0.5 * var < D.var() < 1.5 * var


# ---------------------------------------------------------------- layout

def _check_layout_invariants(lay, topk, E, R):
    topk = np.asarray(topk)
    T, k = topk.shape
    m = E // R
    valid = (topk >= 0) & (topk < E)
    N = int(lay["is_token_in_rank"].sum())
    assert lay["num_recv"] == N
    assert lay["num_tokens_per_rank"].sum() == N
    assert lay["num_tokens_per_expert"].sum() == valid.sum()
    assert lay["rank_prefix"][-1] == N and lay["rank_prefix"][0] == 0
    assert np.all(np.diff(lay["rank_prefix"]) == lay["num_tokens_per_rank"])
    assert np.all(np.diff(lay["expert_prefix"]) == lay["num_tokens_per_expert"])
    np.testing.assert_array_equal(lay["num_tokens_per_rank"], lay["is_token_in_rank"].sum(axis=0))
    np.testing.assert_array_equal(lay["num_tokens_per_expert"],
                                  np.bincount(topk[valid], minlength=E))
    dst = lay["token_dst_row"]
    rows = dst[dst >= 0]
    assert rows.size == N
    np.testing.assert_array_equal(np.sort(rows), np.arange(N))
    # each (token, rank) pair has exactly one row, held by its lowest choice index
    for t in range(T):
        seen = {}
        for j in range(k):
            if valid[t, j]:
                r = int(topk[t, j]) // m
                if r not in seen:
                    seen[r] = j
                    row = int(dst[t, j])
                    assert lay["rank_prefix"][r] <= row < lay["rank_prefix"][r + 1]
                    continue
            assert dst[t, j] == -1
        assert set(seen) == set(np.nonzero(lay["is_token_in_rank"][t])[0].tolist())
    # rows of one rank are ordered by source token
    src = np.full(N, -1)
    for t in range(T):
        for j in range(k):
            if dst[t, j] >= 0:
                src[dst[t, j]] = t
    for r in range(R):
        seg = src[lay["rank_prefix"][r]:lay["rank_prefix"][r + 1]]
        assert np.all(np.diff(seg) > 0)


def _cmp_layout(a, b):
    for key in ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank",
                "rank_prefix", "expert_prefix", "token_dst_row"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


@pytest.mark.parametrize("seed", range(30))
def test_oracle_layout_vs_bruteforce_random_small(seed):
    topk, _, _, E, R = _random_small_case(seed)
    a = oracle.layout(topk.numpy(), E, R)
    b = bf.layout(topk.numpy(), E, R)
    _cmp_layout(a, b)
    assert a["flags"] == 0 and not b["bad_topk"]
    if topk.shape[0]:
        _check_layout_invariants(a, topk.numpy(), E, R)


def test_oracle_layout_tiny_vs_bruteforce_and_invariants():
    w = wl.CONFIGS["tiny"]
    inp = wl.make_inputs(w)
    a = oracle.layout(inp.topk_idx.numpy(), w.num_experts, w.num_ranks)
    _cmp_layout(a, bf.layout(inp.topk_idx.numpy(), w.num_experts, w.num_ranks))
    _check_layout_invariants(a, inp.topk_idx.numpy(), w.num_experts, w.num_ranks)


def test_oracle_layout_duplicates_and_bad_entries():
    # duplicate experts in a row count once per choice for experts, once per rank for ranks;
    # entries outside [-1, E) are flagged and treated as masked
    topk = np.array([[3, 3, 2, -1], [7, 0, 17, -5], [-1, -1, -1, -1], [4, 5, 6, 7]], np.int64)
    E, R = 8, 2
    a = oracle.layout(topk, E, R)
    b = bf.layout(topk, E, R)
    _cmp_layout(a, b)
    assert a["flags"] & oracle.ORACLE_BAD_TOPK and b["bad_topk"]
    assert a["num_tokens_per_expert"][3] == 2
    np.testing.assert_array_equal(a["token_dst_row"][2], [-1, -1, -1, -1])
    # token 3 goes to rank 1 only, via its first choice
    assert a["token_dst_row"][3, 0] >= 0 and np.all(a["token_dst_row"][3, 1:] == -1)


def test_oracle_layout_empty():
    topk = np.zeros((0, 4), np.int64)
    a = oracle.layout(topk, 16, 4)
    assert a["num_recv"] == 0 and a["flags"] == 0
    assert np.all(a["rank_prefix"] == 0) and np.all(a["expert_prefix"] == 0)


@pytest.mark.parametrize("name", ["dsv3", "skewed", "decode"])
def test_oracle_layout_invariants_full_configs(name):
    w = wl.CONFIGS[name]
    g = torch.Generator().manual_seed(w.seed)
    if w.routing == "zipf":
        topk = wl.make_topk_zipf(g, w.num_tokens, w.num_experts, w.num_topk, w.zipf_s)
    else:
        topk = wl.make_topk_uniform(g, w.num_tokens, w.num_experts, w.num_topk)
    a = oracle.layout(topk.numpy(), w.num_experts, w.num_ranks)
    assert a["flags"] == 0
    # whole-config invariants (vectorised)
    N = a["num_recv"]
    assert a["num_tokens_per_expert"].sum() == w.num_tokens * w.num_topk
    dst = a["token_dst_row"]
    np.testing.assert_array_equal(np.sort(dst[dst >= 0]), np.arange(N))
    assert N == a["is_token_in_rank"].sum()


# ---------------------------------------------------------------- number formats

def _all_finite_bf16_as_f32():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = bf.bf16_bits_to_f32(bits)
    return f[np.isfinite(f)]


def _e4m3_midpoints():
    vals = bf._E4M3
    mids = (vals[:-1] + vals[1:]) / 2
    out = []
    for mval in mids:
        m32 = np.float32(mval)
        assert float(m32) == mval          # midpoints are exact in fp32
        out += [m32, np.nextafter(m32, np.float32(np.inf)), np.nextafter(m32, np.float32(0))]
    out += [np.float32(448), np.float32(464), np.float32(480), np.float32(1e30), np.float32(2.0 ** -10),
            np.float32(2.0 ** -10 * 3), np.float32(0.0)]
    a = np.array(out, np.float32)
    return np.concatenate([a, -a])


def test_e4m3_encoder_vs_table_search():
    g = np.random.default_rng(0)
    xs = np.concatenate([
        _all_finite_bf16_as_f32(),
        _e4m3_midpoints(),
        g.uniform(-480, 480, 1_000_000).astype(np.float32),
        g.uniform(-0.05, 0.05, 200_000).astype(np.float32),
        (g.standard_normal(200_000) * 2.0 ** -8).astype(np.float32),
    ])
    np.testing.assert_array_equal(oracle.e4m3_from_float_array(xs), bf.e4m3_encode(xs))


def test_e4m3_encoder_vs_torch_cast_in_range():
    # torch's float8_e4m3fn cast rounds to nearest even; it does not saturate, so
    # compare only within the finite range
    g = np.random.default_rng(1)
    xs = np.concatenate([g.uniform(-448, 448, 1_000_000).astype(np.float32), _e4m3_midpoints()])
    xs = xs[np.abs(xs) <= 448]
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_from_float_array(xs), ref)


def test_e4m3_decode_roundtrip_all_codes():
    for c in range(256):
        if c & 0x7F == 0x7F:
            assert math.isnan(oracle.e4m3_to_float(c))
            continue
        v = oracle.e4m3_to_float(c)
        assert oracle.e4m3_from_float(v) == (c if v != 0 or c & 0x80 == 0 else c)
        assert v == bf.e4m3_decode(np.array([c], np.uint8))[0]
    assert oracle.e4m3_to_float(0x7E) == 448.0 and oracle.e4m3_to_float(0x01) == 2.0 ** -9


def test_bf16_rounding_vs_torch_cast():
    g = np.random.default_rng(2)
    bits = g.integers(0, 1 << 32, 2_000_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    # exact ties: low half 0x8000 with odd and even kept halves
    ties = ((g.integers(0, 1 << 16, 4096, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    xs = np.concatenate([f, ties, np.array([3.3895314e38, -3.3895314e38, 0.0, -0.0], np.float32)])
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_from_float_array(xs), ref)


# ---------------------------------------------------------------- dispatch

def _dispatch_both(topk, w, x, E, R, fp8):
    lay = oracle.layout(topk.numpy(), E, R)
    N = lay["num_recv"]
    a = oracle.dispatch(_bits(x), topk.numpy(), w.numpy(), E, R, lay["token_dst_row"], N, fp8=fp8)
    b = bf.dispatch(_bits(x), topk.numpy(), w.numpy(), E, R, fp8=fp8)
    return lay, a, b


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("seed", range(12))
def test_oracle_dispatch_vs_bruteforce_random_small(seed, fp8):
    topk, w, x, E, R = _random_small_case(seed)
    lay, a, b = _dispatch_both(topk, w, x, E, R, fp8)
    assert a["flags"] == 0
    for key in ("recv_x", "recv_src_idx", "recv_topk_idx"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    np.testing.assert_array_equal(a["recv_topk_weights"].view(np.uint32), b["recv_topk_weights"].view(np.uint32))
    if fp8:
        np.testing.assert_array_equal(a["recv_x_scales"].view(np.uint32), b["recv_x_scales"].view(np.uint32))
        np.testing.assert_array_equal(a["x_scales"].view(np.uint32), b["x_scales"].view(np.uint32))


@pytest.mark.parametrize("fp8", [False, True])
def test_oracle_dispatch_tiny_vs_bruteforce(fp8):
    wk = wl.CONFIGS["tiny"]
    inp = wl.make_inputs(wk)
    lay, a, b = _dispatch_both(inp.topk_idx, inp.topk_weights, inp.x, wk.num_experts, wk.num_ranks, fp8)
    np.testing.assert_array_equal(a["recv_x"], b["recv_x"])
    np.testing.assert_array_equal(a["recv_topk_idx"], b["recv_topk_idx"])
    np.testing.assert_array_equal(a["recv_topk_weights"], b["recv_topk_weights"])


def _dispatch_invariants(inp, E, R, fp8):
    topk = inp.topk_idx.numpy()
    T, k = topk.shape
    m = E // R
    lay = oracle.layout(topk, E, R)
    N = lay["num_recv"]
    xb = _bits(inp.x)
    d = oracle.dispatch(xb, topk, inp.topk_weights.numpy(), E, R, lay["token_dst_row"], N, fp8=fp8)
    src = d["recv_src_idx"]
    ridx = d["recv_topk_idx"]
    rank_of_row = np.searchsorted(lay["rank_prefix"], np.arange(N), side="right") - 1
    # localised indices map back to the source choices
    glob = np.where(ridx >= 0, ridx + (rank_of_row * m)[:, None], -1)
    src_topk = topk[src]
    np.testing.assert_array_equal(glob[ridx >= 0], src_topk[ridx >= 0])
    assert np.all((src_topk[ridx < 0] // m != rank_of_row[np.nonzero(ridx < 0)[0]]) | (src_topk[ridx < 0] < 0))
    assert (ridx >= 0).sum() == (topk >= 0).sum()
    # weights: the local weights of a token's rows add up to all its weights
    wsum = np.zeros(T, np.float64)
    np.add.at(wsum, src, d["recv_topk_weights"].astype(np.float64).sum(axis=1))
    np.testing.assert_allclose(wsum, inp.topk_weights.numpy().astype(np.float64).sum(axis=1), rtol=1e-6)
    if not fp8:
        np.testing.assert_array_equal(d["recv_x"], xb[src])
        return
    # FP8: codes and scales are those of the source row, written once per (token, rank)
    q = d["recv_x"]
    s = d["recv_x_scales"]
    np.testing.assert_array_equal(s, d["x_scales"][src])
    xf = bf.bf16_bits_to_f32(xb[src]).reshape(N, -1, 128)
    amax = np.abs(xf).max(axis=2)
    # the block's largest magnitude encodes to +-448
    arg = np.abs(xf).argmax(axis=2)
    qb = q.reshape(N, -1, 128)
    top = np.take_along_axis(qb, arg[..., None], axis=2)[..., 0]
    assert np.all((top & 0x7F) == 0x7E)
    # reconstruction error within half an E4M3 step (relative 2^-4 in the normal range)
    dec = bf.e4m3_decode(qb.reshape(-1)).reshape(qb.shape) * s[..., None].astype(np.float64)
    err = np.abs(dec - xf)
    bound = np.maximum(np.abs(xf) * 2.0 ** -4, 2.0 ** -10 * s[..., None]) * 1.0001
    assert np.all(err <= bound)
    np.testing.assert_array_equal(s, (amax / np.float32(448)).astype(np.float32))


@pytest.mark.parametrize("fp8", [False, True])
def test_oracle_dispatch_invariants_dsv3_slice(fp8):
    wk = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(wk, with_partial=False, num_tokens=512)
    _dispatch_invariants(inp, wk.num_experts, wk.num_ranks, fp8)


def test_oracle_fp8_zero_block_and_capacity():
    x = torch.zeros(2, 256, dtype=torch.bfloat16)
    x[1, 128:] = torch.linspace(-3, 3, 128).to(torch.bfloat16)
    topk = np.array([[0, 5], [1, 6]], np.int64)
    lay = oracle.layout(topk, 8, 2)
    d = oracle.dispatch(_bits(x), topk, None, 8, 2, lay["token_dst_row"], lay["num_recv"], fp8=True)
    assert d["flags"] == 0
    assert np.all(d["x_scales"][0] == 0) and d["x_scales"][1, 0] == 0
    assert d["x_scales"][1, 1] == np.float32(3.0) / np.float32(448.0)
    rows0 = lay["token_dst_row"][0][lay["token_dst_row"][0] >= 0]
    assert np.all(d["recv_x"][rows0] == 0)
    # capacity one short of N: the last row is flagged and not written
    d2 = oracle.dispatch(_bits(x), topk, None, 8, 2, lay["token_dst_row"], lay["num_recv"] - 1,
                         fp8=False, fill_x=0xFFFF)
    assert d2["flags"] & oracle.ORACLE_CAPACITY


# ---------------------------------------------------------------- combine

@pytest.mark.parametrize("seed", range(20))
def test_oracle_combine_vs_bruteforce_random_small(seed):
    topk, _, _, E, R = _random_small_case(seed)
    g = torch.Generator().manual_seed(1000 + seed)
    lay = oracle.layout(topk.numpy(), E, R)
    H = 64
    partial = _bits(wl.make_partial(g, max(lay["num_recv"], 1), H))
    a, flags = oracle.combine(partial, lay["token_dst_row"])
    assert flags == 0
    np.testing.assert_array_equal(a, bf.combine(partial, lay["token_dst_row"]))


def test_oracle_combine_sums_in_ascending_rank_order():
    # one token on all four ranks (rows 0..3 = ranks 0..3) whose choices list the ranks
    # as 2, 3, 1, 0. Row values 1, 2^-8, 2^-24, 2^-24: in ascending row order both 2^-24
    # terms are absorbed (fp32 ties to even) and 1 + 2^-8 is a bf16 tie that rounds to 1;
    # in choice order they add up to 2^-23 first and the result rounds up to 1 + 2^-7.
    topk = np.array([[2, 3, 1, 0]], np.int64)
    lay = oracle.layout(topk, 4, 4)
    np.testing.assert_array_equal(lay["token_dst_row"], [[2, 3, 1, 0]])
    vals = np.array([[1.0], [2.0 ** -8], [2.0 ** -24], [2.0 ** -24]], np.float32)
    partial = bf.f32_to_bf16_bits(vals)
    out, _ = oracle.combine(partial, lay["token_dst_row"])
    assert bf.bf16_bits_to_f32(out)[0, 0] == np.float32(1.0)
    # the other order really does differ (so the check above can see a wrong order)
    acc = np.float32(0)
    for row in (2, 3, 1, 0):
        acc = np.float32(acc + vals[row, 0])
    assert bf.bf16_bits_to_f32(bf.f32_to_bf16_bits(np.array([acc])))[0] == np.float32(1.0 + 2.0 ** -7)


def test_oracle_dispatch_then_combine_is_d_times_x():
    # partial = recv_x: each token comes back as bf16(D_t * x_t); sums of <= 8 copies of a
    # bf16 value are exact in fp32, so only the final rounding remains (torch's cast)
    wk = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(wk, with_partial=False, num_tokens=256)
    topk = inp.topk_idx.numpy()
    lay = oracle.layout(topk, wk.num_experts, wk.num_ranks)
    d = oracle.dispatch(_bits(inp.x), topk, None, wk.num_experts, wk.num_ranks,
                        lay["token_dst_row"], lay["num_recv"])
    out, _ = oracle.combine(d["recv_x"], lay["token_dst_row"])
    D = torch.from_numpy(lay["is_token_in_rank"].sum(axis=1).astype(np.float32))
    ref = (inp.x.float() * D[:, None]).to(torch.bfloat16)
    np.testing.assert_array_equal(out, _bits(ref))


def test_oracle_identity_expert_returns_x():
    # expert = identity scaled by the row's local weights; weights sum to 1 per token,
    # so combine returns x up to two bf16 roundings (unit roundoff 2^-8 each -> 2^-7)
    wk = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(wk, with_partial=False, num_tokens=256)
    topk = inp.topk_idx.numpy()
    lay = oracle.layout(topk, wk.num_experts, wk.num_ranks)
    d = oracle.dispatch(_bits(inp.x), topk, inp.topk_weights.numpy(), wk.num_experts, wk.num_ranks,
                        lay["token_dst_row"], lay["num_recv"])
    wrow = d["recv_topk_weights"].sum(axis=1)
    partial = bf.f32_to_bf16_bits(bf.bf16_bits_to_f32(d["recv_x"]) * wrow[:, None])
    out, _ = oracle.combine(partial, lay["token_dst_row"])
    got = bf.bf16_bits_to_f32(out).astype(np.float64)
    x = inp.x.float().numpy().astype(np.float64)
    assert np.all(np.abs(got - x) <= 2.0 ** -7 * np.abs(x) * 1.01 + 1e-30)


def test_oracle_combine_token_without_rows_is_zero():
    topk = np.array([[-1, -1], [0, 1]], np.int64)
    lay = oracle.layout(topk, 2, 2)
    partial = bf.f32_to_bf16_bits(np.ones((2, 16), np.float32))
    out, _ = oracle.combine(partial, lay["token_dst_row"])
    assert np.all(out[0] == 0) and np.all(bf.bf16_bits_to_f32(out[1]) == 2.0)


# ---------------------------------------------------------------- dispatch of E4M3 input

def test_oracle_fp8_input_dispatch_matches_quantised_dispatch():
    # quantising inside dispatch and dispatching already-quantised rows with their
    # scales must land the same bytes in the same receive rows
    wk = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(wk, with_partial=False, num_tokens=300)
    topk = inp.topk_idx.numpy()
    lay = oracle.layout(topk, wk.num_experts, wk.num_ranks)
    N = lay["num_recv"]
    q = oracle.dispatch(_bits(inp.x), topk, inp.topk_weights.numpy(), wk.num_experts, wk.num_ranks,
                        lay["token_dst_row"], N, fp8=True)
    # the source rows' codes: each token's codes appear in every one of its receive rows
    src = q["recv_src_idx"]
    codes = np.zeros((300, wk.hidden), np.uint8)
    codes[src] = q["recv_x"]
    c = oracle.dispatch_fp8_input(codes, q["x_scales"], topk, inp.topk_weights.numpy(), wk.num_experts,
                                  wk.num_ranks, lay["token_dst_row"], N)
    assert c["flags"] == 0
    for key in ("recv_x", "recv_topk_idx", "recv_src_idx"):
        np.testing.assert_array_equal(c[key], q[key], err_msg=key)
    np.testing.assert_array_equal(c["recv_x_scales"].view(np.uint32), q["recv_x_scales"].view(np.uint32))


def test_oracle_fp8_input_dispatch_copies_bytes():
    g = np.random.default_rng(3)
    T, H, E, R, k = 64, 256, 16, 4, 3
    topk = wl.make_topk_uniform(torch.Generator().manual_seed(3), T, E, k).numpy()
    codes = g.integers(0, 256, (T, H), dtype=np.uint8)
    scales = g.standard_normal((T, H // 128)).astype(np.float32)
    lay = oracle.layout(topk, E, R)
    d = oracle.dispatch_fp8_input(codes, scales, topk, None, E, R, lay["token_dst_row"], lay["num_recv"])
    src = d["recv_src_idx"]
    np.testing.assert_array_equal(d["recv_x"], codes[src])
    np.testing.assert_array_equal(d["recv_x_scales"], scales[src])
    assert np.all(d["recv_topk_weights"] == 0)


# ---------------------------------------------------------------- weighted combine

def _rn32(v):
    from fractions import Fraction
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    q = Fraction(2) ** (max(e, -126) - 23)
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * q


def test_oracle_weighted_combine_vs_exact_fma():
    # acc = fma(w, x, acc): the exact product plus acc, rounded once to fp32, emulated with rationals
    from fractions import Fraction
    g = torch.Generator().manual_seed(4)
    T, E, R, k, H = 24, 16, 8, 4, 16
    topk = wl.make_topk_uniform(g, T, E, k)
    lay = oracle.layout(topk.numpy(), E, R)
    N = lay["num_recv"]
    partial = _bits(wl.make_partial(g, N, H))
    w = (torch.rand(N, generator=g) * 3 - 1).numpy().astype(np.float32)
    out, _, flags = oracle.combine_weighted(partial, lay["token_dst_row"], w)
    assert flags == 0
    pf = bf.bf16_bits_to_f32(partial)
    ref = np.zeros((T, H), np.float32)
    for t in range(T):
        rows = sorted(int(r) for r in lay["token_dst_row"][t] if r >= 0)
        for h in range(H):
            acc = Fraction(0)
            for r in rows:
                acc = _rn32(Fraction(float(w[r])) * Fraction(float(pf[r, h])) + acc)
            ref[t, h] = float(acc)
    np.testing.assert_array_equal(out, bf.f32_to_bf16_bits(ref))


def test_oracle_weighted_combine_unit_weights_is_plain_combine():
    wk = wl.CONFIGS["tiny"]
    inp = wl.make_inputs(wk)
    lay = oracle.layout(inp.topk_idx.numpy(), wk.num_experts, wk.num_ranks)
    partial = _bits(inp.partial)
    a, _, _ = oracle.combine_weighted(partial, lay["token_dst_row"], np.ones(partial.shape[0], np.float32))
    b, _ = oracle.combine(partial, lay["token_dst_row"])
    np.testing.assert_array_equal(a, b)


def test_oracle_combined_topk_weights_return_the_routing_weights():
    # each weight travels in exactly one receive row (its expert's rank), zeros elsewhere,
    # so reducing the received weights gives the token's weights back
    wk = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(wk, with_partial=False, num_tokens=256)
    topk = wl.mask_random_lanes(torch.Generator().manual_seed(9), inp.topk_idx, 0.2).numpy()
    lay = oracle.layout(topk, wk.num_experts, wk.num_ranks)
    d = oracle.dispatch(_bits(inp.x), topk, inp.topk_weights.numpy(), wk.num_experts, wk.num_ranks,
                        lay["token_dst_row"], lay["num_recv"])
    _, cw, _ = oracle.combine_weighted(d["recv_x"], lay["token_dst_row"], None, d["recv_topk_weights"])
    expect = np.where(topk >= 0, inp.topk_weights.numpy(), 0.0).astype(np.float32)
    np.testing.assert_array_equal(cw, expect)


def test_oracle_weighted_combine_is_fused():
    # two rows of one token: acc = wA * 1 exactly, then wB * xB has an inexact fp32
    # product whose lost part (2^-30) is all that is left after cancellation --
    # a fused multiply-add keeps it, multiply-then-add loses it
    topk = np.array([[0, 1]], np.int64)
    lay = oracle.layout(topk, 2, 2)                     # rows 0 and 1
    wA = np.float32(-(1 + 2.0 ** -7 + 2.0 ** -23))
    wB = np.float32(1 + 2.0 ** -23)
    partial = bf.f32_to_bf16_bits(np.array([[1.0], [1 + 2.0 ** -7]], np.float32))
    assert float(wA) == -(1 + 2.0 ** -7 + 2.0 ** -23) and float(wB) == 1 + 2.0 ** -23
    out, _, _ = oracle.combine_weighted(partial, lay["token_dst_row"], np.array([wA, wB], np.float32))
    assert bf.bf16_bits_to_f32(out)[0, 0] == np.float32(2.0 ** -30)


# ---------------------------------------------------------------- expand mode (one row per valid entry)

def _cmp_expand(a, b):
    np.testing.assert_array_equal(a["expert_prefix"], b["expert_prefix"])
    np.testing.assert_array_equal(a["token_expert_row"], b["token_expert_row"])
    assert a["num_recv"] == b["num_recv"]


@pytest.mark.parametrize("seed", range(30))
def test_oracle_expand_layout_vs_bruteforce_random_small(seed):
    topk, _, _, E, R = _random_small_case(seed)
    a = oracle.expand_layout(topk.numpy(), E)
    assert a["flags"] == 0
    _cmp_expand(a, bf.expand_layout(topk.numpy(), E))


def test_oracle_expand_layout_duplicates_and_bad_entries():
    # a token naming one expert twice gets two rows; entries outside [-1, E) are flagged and get no row
    topk = np.array([[1, 1, -1], [0, 7, 1], [-5, 0, 2], [2, 2, 2]], np.int64)
    a = oracle.expand_layout(topk, 4)
    assert a["flags"] == oracle.ORACLE_BAD_TOPK
    _cmp_expand(a, bf.expand_layout(topk, 4))
    np.testing.assert_array_equal(a["expert_prefix"], [0, 2, 5, 9, 9])
    np.testing.assert_array_equal(a["token_expert_row"], [[2, 3, -1], [0, -1, 4], [-1, 1, 5], [6, 7, 8]])


def test_oracle_expand_layout_empty():
    a = oracle.expand_layout(np.zeros((0, 4), np.int64), 8)
    assert a["flags"] == 0 and a["num_recv"] == 0
    np.testing.assert_array_equal(a["expert_prefix"], np.zeros(9, np.int32))


@pytest.mark.parametrize("name", ["dsv3", "skewed", "decode"])
def test_oracle_expand_layout_invariants_full_configs(name):
    wk = wl.CONFIGS[name]
    topk = wl.make_inputs(wk, with_partial=False, num_tokens=min(wk.num_tokens, 2048)).topk_idx.numpy()
    E = wk.num_experts
    a = oracle.expand_layout(topk, E)
    rows = a["token_expert_row"]
    valid = topk >= 0
    # one row per valid entry, rows a permutation of [0, number of valid entries)
    assert np.all((rows >= 0) == valid)
    np.testing.assert_array_equal(np.sort(rows[valid]), np.arange(int(valid.sum())))
    # the per-expert prefix is the rank-mode layout's expert_prefix
    np.testing.assert_array_equal(a["expert_prefix"], oracle.layout(topk, E, wk.num_ranks)["expert_prefix"])
    # each expert's rows fill its region, in ascending (token, choice) order
    t_idx, j_idx = np.nonzero(valid)
    e = topk[t_idx, j_idx]
    r = rows[t_idx, j_idx]
    assert np.all(r >= a["expert_prefix"][e]) and np.all(r < a["expert_prefix"][e + 1])
    order = np.lexsort((j_idx, t_idx, e))
    np.testing.assert_array_equal(r[order], np.arange(len(r)))


def _distinct_topk(seed, T, E, k):
    return wl.make_topk_uniform(torch.Generator().manual_seed(seed), T, E, k)


@pytest.mark.parametrize("mode", [0, 1])
def test_oracle_expand_reduces_to_rank_mode_with_one_expert_per_rank(mode):
    # with one expert per rank (E == R) and distinct experts per token, every entry is its
    # rank's only entry: the expand rows, the copies and the metadata are those of rank mode
    T, E, k, H = 96, 16, 4, 256
    topk = wl.mask_random_lanes(torch.Generator().manual_seed(3), _distinct_topk(2, T, E, k), 0.2).numpy()
    w = wl.make_weights(torch.Generator().manual_seed(4), T, k).numpy()
    x = _bits(wl.make_x(torch.Generator().manual_seed(5), T, H))
    lay = oracle.layout(topk, E, E)
    ex = oracle.expand_layout(topk, E)
    np.testing.assert_array_equal(ex["token_expert_row"], lay["token_dst_row"])
    N = lay["num_recv"]
    a = oracle.dispatch(x, topk, w, E, E, lay["token_dst_row"], N, fp8=mode == 1)
    b = oracle.dispatch_expand(mode, x, topk, w, E, E, ex["token_expert_row"], N)
    for key in ("recv_x", "recv_topk_idx", "recv_src_idx"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    np.testing.assert_array_equal(a["recv_topk_weights"].view(np.uint32), b["recv_topk_weights"].view(np.uint32))
    if mode == 1:
        np.testing.assert_array_equal(a["recv_x_scales"].view(np.uint32), b["recv_x_scales"].view(np.uint32))
        np.testing.assert_array_equal(a["x_scales"].view(np.uint32), b["x_scales"].view(np.uint32))


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("seed", range(12))
def test_oracle_dispatch_expand_vs_bruteforce_random_small(seed, fp8):
    topk, w, x, E, R = _random_small_case(seed)
    ex = oracle.expand_layout(topk.numpy(), E)
    a = oracle.dispatch_expand(1 if fp8 else 0, _bits(x), topk.numpy(), w.numpy(), E, R, ex["token_expert_row"],
                               ex["num_recv"])
    b = bf.dispatch_expand(_bits(x), topk.numpy(), w.numpy(), E, R, fp8=fp8)
    assert a["flags"] == 0
    for key in ("recv_x", "recv_src_idx", "recv_topk_idx"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    np.testing.assert_array_equal(a["recv_topk_weights"].view(np.uint32), b["recv_topk_weights"].view(np.uint32))
    if fp8:
        np.testing.assert_array_equal(a["recv_x_scales"].view(np.uint32), b["recv_x_scales"].view(np.uint32))


def test_oracle_dispatch_expand_fp8_input_matches_quantised():
    # E4M3 rows dispatched with their scales land the same bytes as quantising inside dispatch
    wk = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(wk, with_partial=False, num_tokens=64)
    topk = inp.topk_idx.numpy()
    ex = oracle.expand_layout(topk, wk.num_experts)
    N = ex["num_recv"]
    q = oracle.dispatch_expand(1, _bits(inp.x), topk, inp.topk_weights.numpy(), wk.num_experts, wk.num_ranks,
                               ex["token_expert_row"], N)
    # the token's codes: any of its expand rows
    first = np.array([ex["token_expert_row"][t][ex["token_expert_row"][t] >= 0][0] for t in range(64)])
    codes, scales = q["recv_x"][first], q["recv_x_scales"][first]
    np.testing.assert_array_equal(scales.view(np.uint32), q["x_scales"].view(np.uint32))
    p = oracle.dispatch_expand(2, codes, topk, inp.topk_weights.numpy(), wk.num_experts, wk.num_ranks,
                               ex["token_expert_row"], N, x_scales=scales)
    for key in ("recv_x", "recv_topk_idx", "recv_src_idx"):
        np.testing.assert_array_equal(p[key], q[key], err_msg=key)
    np.testing.assert_array_equal(p["recv_x_scales"].view(np.uint32), q["recv_x_scales"].view(np.uint32))


def test_oracle_expand_dispatch_then_combine_is_count_times_x():
    # identity experts on the expand rows: every valid entry sends x_t back once, so the
    # combine returns bf16(n_t * x_t); with k = 4 all valid, n_t = 4 and the sum is exact
    wk = wl.CONFIGS["dsv3"]
    T, E, k = 128, wk.num_experts, 4
    topk = _distinct_topk(7, T, E, k).numpy()
    x = wl.make_x(torch.Generator().manual_seed(8), T, 256)
    ex = oracle.expand_layout(topk, E)
    d = oracle.dispatch_expand(0, _bits(x), topk, None, E, wk.num_ranks, ex["token_expert_row"], ex["num_recv"])
    out, flags = oracle.combine(d["recv_x"], ex["token_expert_row"])
    assert flags == 0
    np.testing.assert_array_equal(out, _bits((x.float() * 4).to(torch.bfloat16)))


def test_oracle_expand_weighted_combine_returns_weights_and_mixture():
    # each entry's weight travels in its own row only, so the reduced weights are the routing
    # weights; weighting each identity-expert row by its entry weight gives sum_j w_j * x_t
    wk = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(wk, with_partial=False, num_tokens=128)
    topk = wl.mask_random_lanes(torch.Generator().manual_seed(11), inp.topk_idx, 0.2).numpy()
    w = inp.topk_weights.numpy()
    ex = oracle.expand_layout(topk, wk.num_experts)
    d = oracle.dispatch_expand(0, _bits(inp.x), topk, w, wk.num_experts, wk.num_ranks, ex["token_expert_row"],
                               ex["num_recv"])
    row_w = d["recv_topk_weights"].sum(axis=1).astype(np.float32)     # one non-zero entry per row
    out, cw, _ = oracle.combine_weighted(d["recv_x"], ex["token_expert_row"], row_w, d["recv_topk_weights"])
    np.testing.assert_array_equal(cw, np.where(topk >= 0, w, 0.0).astype(np.float32))
    wsum = np.where(topk >= 0, w, 0.0).astype(np.float64).sum(axis=1)
    x = inp.x.float().numpy().astype(np.float64)
    got = bf.bf16_bits_to_f32(out).astype(np.float64)
    # fp32 fma chain of <= 8 terms then one bf16 rounding
    assert np.all(np.abs(got - wsum[:, None] * x) <= 2.0 ** -8 * np.abs(wsum[:, None] * x) * 1.01 + 8 * 2.0 ** -24 * np.abs(x))


# ---------------------------------------------------------------- combine of E4M3 partial rows

def _random_fp8_rows(seed, rows, H):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, (rows, H), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38          # no NaN codes
    scales = (rng.standard_normal((rows, H // 128)) * 2.0 ** rng.integers(-8, 8, (rows, H // 128))).astype(np.float32)
    return codes, scales


@pytest.mark.parametrize("seed", range(10))
def test_oracle_combine_fp8_vs_bruteforce(seed):
    topk, _, _, E, R = _random_small_case(seed)
    lay = oracle.layout(topk.numpy(), E, R)
    H = 256
    codes, scales = _random_fp8_rows(seed, max(lay["num_recv"], 1), H)
    a, flags = oracle.combine_fp8(codes, scales, lay["token_dst_row"])
    assert flags == 0
    np.testing.assert_array_equal(a, bf.combine_fp8(codes, scales, lay["token_dst_row"]))


def test_oracle_combine_fp8_single_row_is_the_e4m3_value():
    # one row per token with scale 1: every E4M3 value is a bf16 value, so the output is the table value exactly
    codes = np.arange(256, dtype=np.uint8).reshape(2, 128)
    codes[(codes & 0x7F) == 0x7F] = 0
    dst = np.array([[0, -1], [-1, 1]], np.int32)
    out, _ = oracle.combine_fp8(codes, np.ones((2, 1), np.float32), dst)
    np.testing.assert_array_equal(bf.bf16_bits_to_f32(out), bf.e4m3_decode(codes).astype(np.float32))


def test_oracle_combine_fp8_rounds_product_then_sum():
    # row 0: -1.0 * (1.125 + 2^-23) is exact; row 1: 1.125 * (1 + 2^-23) = 1.125 + 2^-23 + 2^-26 rounds to
    # 1.125 + 2^-23, so the ascending sum is exactly 0; a fused multiply-add would keep 2^-26
    codes = np.array([[0xB8] * 128, [0x39] * 128], np.uint8)
    assert bf.e4m3_decode(codes[:, :1]).ravel().tolist() == [-1.0, 1.125]
    scales = np.array([[1.125 + 2.0 ** -23], [1 + 2.0 ** -23]], np.float32)
    out, _ = oracle.combine_fp8(codes, scales, np.array([[0, 1]], np.int32))
    assert np.all(out == 0)


def test_oracle_dispatch_fp8_then_combine_fp8_is_d_times_dequantised_x():
    # identity experts on FP8 rows: every row of a token carries the same codes and scales, so the combine
    # returns the D-fold sum of the dequantised token, within one bf16 rounding plus the fp32 sum's roundings
    wk = wl.CONFIGS["dsv3"]
    inp = wl.make_inputs(wk, with_partial=False, num_tokens=128)
    topk = inp.topk_idx.numpy()
    lay = oracle.layout(topk, wk.num_experts, wk.num_ranks)
    d = oracle.dispatch(_bits(inp.x), topk, None, wk.num_experts, wk.num_ranks, lay["token_dst_row"], lay["num_recv"],
                        fp8=True)
    out, flags = oracle.combine_fp8(d["recv_x"], d["recv_x_scales"], lay["token_dst_row"])
    assert flags == 0
    deq = bf.e4m3_decode(d["recv_x"]).astype(np.float64) * np.repeat(d["recv_x_scales"].astype(np.float64), 128, axis=1)
    D = lay["is_token_in_rank"].sum(axis=1).astype(np.float64)
    first = np.array([lay["token_dst_row"][t][lay["token_dst_row"][t] >= 0].min() for t in range(128)])
    ref = D[:, None] * deq[first]
    got = bf.bf16_bits_to_f32(out).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) * 1.01 + 1e-30)
