"""Second, independent CPU implementation for tiny inputs (pure Python + numpy).

TEST INFRASTRUCTURE ONLY (part of the oracle package). It pins the C oracle:
each function reaches the same result as ``moe_oracle.c`` by a different
route, so a slip in either shows up as a mismatch.

* Layout: collect every (rank, token) pair once, keeping the lowest choice
  index, then sort the pairs by (rank, token): a pair's index in that sorted
  list is its global receive row. (The C oracle uses counts, exclusive prefix
  sums and running per-rank positions instead.)
* E4M3: enumerate the 127 non-negative finite codes from the format
  definition and pick the nearest value, ties to the code with an even last
  bit, saturating above 448. (The C oracle counts quanta per binade.)
* bf16 rounding: torch's float32 -> bfloat16 cast (round to nearest even).
* fp32 sums: numpy float32 element-wise adds, one row at a time.
* Expand layout: list every valid (expert, token, choice) triple and sort it;
  a triple's index in the sorted list is its row. (The C oracle uses counts,
  prefix sums and a running counter per expert.)
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch


def layout(topk_idx, num_experts: int, num_ranks: int) -> dict:
    topk = [list(map(int, row)) for row in np.asarray(topk_idx)]
    T = len(topk)
    k = len(topk[0]) if T else 0
    m = num_experts // num_ranks
    bad = False
    expert_count = [0] * num_experts
    pairs = []                                  # (rank, token, first choice index)
    for t, row in enumerate(topk):
        owner = {}
        for j, e in enumerate(row):
            if e == -1:
                continue
            if not (0 <= e < num_experts):
                bad = True
                continue
            expert_count[e] += 1
            owner.setdefault(e // m, j)
        pairs.extend((r, t, j) for r, j in owner.items())
    pairs.sort()
    dst = np.full((T, k), -1, np.int32)
    in_rank = np.zeros((T, num_ranks), np.uint8)
    rank_count = [0] * num_ranks
    for row, (r, t, j) in enumerate(pairs):
        dst[t, j] = row
        in_rank[t, r] = 1
        rank_count[r] += 1
    rank_prefix = np.array([sum(rank_count[:r]) for r in range(num_ranks + 1)], np.int32)
    expert_prefix = np.array([sum(expert_count[:e]) for e in range(num_experts + 1)], np.int32)
    return dict(num_tokens_per_rank=np.array(rank_count, np.int32),
                num_tokens_per_expert=np.array(expert_count, np.int32),
                is_token_in_rank=in_rank, rank_prefix=rank_prefix, expert_prefix=expert_prefix,
                token_dst_row=dst, bad_topk=bad, num_recv=len(pairs))


def _e4m3_table() -> np.ndarray:
    vals = []
    for code in range(127):                     # 0x00..0x7E, 0x7F is NaN
        ex, man = code >> 3, code & 7
        if ex == 0:
            vals.append(man / 8.0 * 2.0 ** -6)
        else:
            vals.append((1.0 + man / 8.0) * 2.0 ** (ex - 7))
    return np.array(vals, np.float64)


_E4M3 = _e4m3_table()


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code by table search (finite inputs)."""
    v = np.asarray(v, np.float32).astype(np.float64)
    sign = np.signbit(v).astype(np.uint8) << 7
    a = np.abs(v)
    hi = np.clip(np.searchsorted(_E4M3, a, side="left"), 0, 126)   # first table value >= a
    lo = np.clip(hi - 1, 0, 126)
    d_hi = np.abs(_E4M3[hi] - a)
    d_lo = np.abs(a - _E4M3[lo])
    pick = np.where(d_lo < d_hi, lo, hi)
    tie = (d_lo == d_hi) & (lo != hi)
    pick = np.where(tie, np.where(lo % 2 == 0, lo, hi), pick)
    pick = np.where(a > 448.0, 126, pick)
    return (pick.astype(np.uint8) | sign).astype(np.uint8)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, np.uint8)
    mag = _E4M3[np.minimum(c & 0x7F, 126)]
    return np.where(c & 0x80, -mag, mag)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def dispatch(x_bits: np.ndarray, topk_idx, topk_weights: Optional[np.ndarray], num_experts: int,
             num_ranks: int, fp8: bool = False) -> dict:
    """Receive buffers of exactly N rows (N = number of (token, rank) pairs)."""
    lay = layout(topk_idx, num_experts, num_ranks)
    topk = np.asarray(topk_idx)
    T, k = topk.shape
    H = x_bits.shape[1]
    m = num_experts // num_ranks
    N = lay["num_recv"]
    dst = lay["token_dst_row"]
    recv_src = np.zeros(N, np.int32)
    recv_idx = np.zeros((N, k), np.int64)
    recv_w = np.zeros((N, k), np.float32)
    if fp8:
        nb = H // 128
        q = np.zeros((T, H), np.uint8)
        s = np.zeros((T, nb), np.float32)
        xf = bf16_bits_to_f32(x_bits)
        for t in range(T):
            for b in range(nb):
                blk = xf[t, b * 128:(b + 1) * 128]
                amax = np.float32(np.max(np.abs(blk)))
                sc = np.float32(amax / np.float32(448.0))
                s[t, b] = sc
                if sc != 0:
                    q[t, b * 128:(b + 1) * 128] = e4m3_encode((blk / sc).astype(np.float32))
        recv_x = np.zeros((N, H), np.uint8)
        recv_scales = np.zeros((N, nb), np.float32)
    else:
        recv_x = np.zeros((N, H), np.uint16)
    for t in range(T):
        for j in range(k):
            row = int(dst[t, j])
            if row < 0:
                continue
            r = int(topk[t, j]) // m
            recv_src[row] = t
            if fp8:
                recv_x[row] = q[t]
                recv_scales[row] = s[t]
            else:
                recv_x[row] = x_bits[t]
            for jj in range(k):
                e = int(topk[t, jj])
                if 0 <= e < num_experts and e // m == r:
                    recv_idx[row, jj] = e - r * m
                    recv_w[row, jj] = 0.0 if topk_weights is None else topk_weights[t, jj]
                else:
                    recv_idx[row, jj] = -1
                    recv_w[row, jj] = 0.0
    out = dict(layout=lay, recv_x=recv_x, recv_src_idx=recv_src, recv_topk_idx=recv_idx,
               recv_topk_weights=recv_w)
    if fp8:
        out["recv_x_scales"] = recv_scales
        out["x_scales"] = s
    return out


def combine(partial_bits: np.ndarray, token_dst_row: np.ndarray) -> np.ndarray:
    T, k = token_dst_row.shape
    H = partial_bits.shape[1]
    pf = bf16_bits_to_f32(partial_bits)
    out = np.zeros((T, H), np.float32)
    for t in range(T):
        acc = np.zeros(H, np.float32)
        for row in sorted(int(v) for v in token_dst_row[t] if v >= 0):
            acc = (acc + pf[row]).astype(np.float32)
        out[t] = acc
    return f32_to_bf16_bits(out)


def expand_layout(topk_idx, num_experts: int) -> dict:
    topk = np.asarray(topk_idx, np.int64)
    T, k = topk.shape if topk.ndim == 2 else (0, 1)
    triples = sorted((int(topk[t, j]), t, j) for t in range(T) for j in range(k)
                     if 0 <= int(topk[t, j]) < num_experts)
    rows = np.full((T, k), -1, np.int32)
    for row, (_, t, j) in enumerate(triples):
        rows[t, j] = row
    prefix = np.zeros(num_experts + 1, np.int32)
    for e, _, _ in triples:
        prefix[e + 1:] += 1
    bad = bool(np.any((topk != -1) & ((topk < 0) | (topk >= num_experts))))
    return dict(expert_prefix=prefix, token_expert_row=rows, num_recv=len(triples), bad_topk=bad)


def dispatch_expand(x_bits: np.ndarray, topk_idx, topk_weights: Optional[np.ndarray], num_experts: int,
                    num_ranks: int, fp8: bool = False) -> dict:
    """Expand-mode receive buffers of exactly one row per valid entry."""
    lay = expand_layout(topk_idx, num_experts)
    topk = np.asarray(topk_idx)
    T, k = topk.shape
    H = x_bits.shape[1]
    m = num_experts // num_ranks
    N = lay["num_recv"]
    rows = lay["token_expert_row"]
    if fp8:
        # the token's codes and scales are those of the rank-mode brute force
        ref = dispatch(x_bits, topk_idx, topk_weights, num_experts, num_ranks, fp8=True)
        src_rows = layout(topk_idx, num_experts, num_ranks)["token_dst_row"]
        recv_x = np.zeros((N, H), np.uint8)
        recv_scales = np.zeros((N, H // 128), np.float32)
    else:
        recv_x = np.zeros((N, H), np.uint16)
    recv_src = np.zeros(N, np.int32)
    recv_idx = np.full((N, k), -1, np.int64)
    recv_w = np.zeros((N, k), np.float32)
    for t in range(T):
        for j in range(k):
            row = int(rows[t, j])
            if row < 0:
                continue
            e = int(topk[t, j])
            recv_src[row] = t
            recv_idx[row, j] = e % m
            recv_w[row, j] = 0.0 if topk_weights is None else topk_weights[t, j]
            if fp8:
                # any rank-mode row of token t holds its codes
                r_row = max(int(v) for v in src_rows[t])
                recv_x[row] = ref["recv_x"][r_row]
                recv_scales[row] = ref["recv_x_scales"][r_row]
            else:
                recv_x[row] = x_bits[t]
    out = dict(layout=lay, recv_x=recv_x, recv_src_idx=recv_src, recv_topk_idx=recv_idx, recv_topk_weights=recv_w)
    if fp8:
        out["recv_x_scales"] = recv_scales
        out["x_scales"] = ref["x_scales"]
    return out


def combine_fp8(codes: np.ndarray, scales: np.ndarray, token_dst_row: np.ndarray) -> np.ndarray:
    """Dequantise by table lookup times the block scale (numpy float32), then
    add the token's rows in ascending row order; bf16 by torch's cast."""
    T, k = token_dst_row.shape
    H = codes.shape[1]
    deq = (e4m3_decode(codes).astype(np.float32) * np.repeat(np.asarray(scales, np.float32), 128, axis=1)).astype(np.float32)
    out = np.zeros((T, H), np.float32)
    for t in range(T):
        acc = np.zeros(H, np.float32)
        for row in sorted(int(v) for v in token_dst_row[t] if v >= 0):
            acc = (acc + deq[row]).astype(np.float32)
        out[t] = acc
    return f32_to_bf16_bits(out)
