"""CPU oracle for MoE layout / dispatch / combine on logical ranks.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(``combine_moe_get_gb300``) never imports it, and the two share no code.

``liboracle.so`` (from ``moe_oracle.c``) holds the scalar definitions; this
module only marshals numpy arrays into it. ``bruteforce.py`` is a second,
pure-Python implementation used to pin the C oracle on tiny inputs, and
``expected_topk.py`` holds the closed form for the expected number of distinct
destination ranks per token.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from .build import build as _build

ORACLE_BAD_TOPK = 1
ORACLE_CAPACITY = 2
ORACLE_BAD_ARG = 4

_lib = None


def lib():
    global _lib
    if _lib is None:
        # MOE_ORACLE_LIB points the pins at a deliberately broken copy of the
        # oracle (the mutation test); normally the library is built in place.
        _lib = ctypes.CDLL(os.environ.get("MOE_ORACLE_LIB") or _build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        _lib.oracle_layout.argtypes = [P, I, I, I, I, P, P, P, P, P, P]
        _lib.oracle_dispatch_bf16.argtypes = [P, I, I, P, P, I, I, I, P, I, P, P, P, P]
        _lib.oracle_dispatch_fp8.argtypes = [P, I, I, P, P, I, I, I, P, I, P, P, P, P, P, P]
        _lib.oracle_combine.argtypes = [P, I, I, I, I, P, P]
        _lib.oracle_dispatch_fp8_input.argtypes = [P, P, I, I, P, P, I, I, I, P, I, P, P, P, P, P]
        _lib.oracle_dispatch_fp8_input.restype = I
        _lib.oracle_combine_weighted.argtypes = [P, I, I, I, I, P, P, P, P, P]
        _lib.oracle_combine_weighted.restype = I
        _lib.oracle_expand_layout.argtypes = [P, I, I, I, P, P]
        _lib.oracle_expand_layout.restype = I
        _lib.oracle_dispatch_expand.argtypes = [I, P, P, I, I, P, P, I, I, I, P, I, P, P, P, P, P, P]
        _lib.oracle_dispatch_expand.restype = I
        _lib.oracle_combine_fp8.argtypes = [P, P, I, I, I, I, P, P]
        _lib.oracle_combine_fp8.restype = I
        _lib.oracle_dispatch_bf16_mt.argtypes = [P, I, I, P, P, I, I, I, P, I, P, P, P, P, I]
        _lib.oracle_dispatch_bf16_mt.restype = I
        _lib.oracle_combine_mt.argtypes = [P, I, I, I, I, P, P, I]
        _lib.oracle_combine_mt.restype = I
        for f in ("oracle_layout", "oracle_dispatch_bf16", "oracle_dispatch_fp8", "oracle_combine"):
            getattr(_lib, f).restype = I
        _lib.oracle_bf16_from_float.argtypes = [ctypes.c_float]
        _lib.oracle_bf16_from_float.restype = ctypes.c_uint16
        _lib.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
        _lib.oracle_bf16_to_float.restype = ctypes.c_float
        _lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        _lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
        _lib.oracle_e4m3_to_float.argtypes = [ctypes.c_uint8]
        _lib.oracle_e4m3_to_float.restype = ctypes.c_float
        _lib.oracle_bf16_from_float_n.argtypes = [P, P, ctypes.c_int64]
        _lib.oracle_e4m3_from_float_n.argtypes = [P, P, ctypes.c_int64]
    return _lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def layout(topk_idx: np.ndarray, num_experts: int, num_ranks: int) -> dict:
    """Counts, membership bitmap, prefixes and global receive rows."""
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, k = topk_idx.shape
    out = dict(
        num_tokens_per_rank=np.zeros(num_ranks, np.int32),
        num_tokens_per_expert=np.zeros(num_experts, np.int32),
        is_token_in_rank=np.zeros((T, num_ranks), np.uint8),
        rank_prefix=np.zeros(num_ranks + 1, np.int32),
        expert_prefix=np.zeros(num_experts + 1, np.int32),
        token_dst_row=np.zeros((T, k), np.int32),
    )
    flags = lib().oracle_layout(_ptr(topk_idx), T, k, num_experts, num_ranks,
                                _ptr(out["num_tokens_per_rank"]), _ptr(out["num_tokens_per_expert"]),
                                _ptr(out["is_token_in_rank"]), _ptr(out["rank_prefix"]),
                                _ptr(out["expert_prefix"]), _ptr(out["token_dst_row"]))
    out["flags"] = flags
    out["num_recv"] = int(out["rank_prefix"][-1])
    return out


def dispatch(x_bits: np.ndarray, topk_idx: np.ndarray, topk_weights: Optional[np.ndarray],
             num_experts: int, num_ranks: int, token_dst_row: np.ndarray, recv_capacity: int,
             fp8: bool = False, fill_x: int = 0, fill_meta: int = 0, threads: int = 1) -> dict:
    """Row copies (bf16 bit patterns, or E4M3 codes plus per-128 scales) and
    per-row metadata. ``x_bits`` holds bf16 bit patterns as uint16 [T, H].
    Unwritten receive rows keep the fill values, so callers can compare
    poisoned buffers byte for byte. ``threads`` > 1 runs the bf16 copy over
    token ranges on that many threads (same results; for timing)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    token_dst_row = np.ascontiguousarray(token_dst_row, dtype=np.int32)
    w = None if topk_weights is None else np.ascontiguousarray(topk_weights, dtype=np.float32)
    T, H = x_bits.shape
    k = topk_idx.shape[1]
    cap = recv_capacity
    out = dict(
        recv_topk_idx=np.full((cap, k), fill_meta, np.int64),
        recv_topk_weights=np.full((cap, k), fill_meta, np.int32).view(np.float32),
        recv_src_idx=np.full(cap, fill_meta, np.int32),
    )
    L = lib()
    if fp8:
        nb = H // 128
        out["recv_x"] = np.full((cap, H), fill_x & 0xFF, np.uint8)
        out["recv_x_scales"] = np.full((cap, nb), fill_meta, np.int32).view(np.float32)
        out["x_scales"] = np.zeros((T, nb), np.float32)
        flags = L.oracle_dispatch_fp8(_ptr(x_bits), T, H, _ptr(topk_idx), _ptr(w), k, num_experts, num_ranks,
                                      _ptr(token_dst_row), cap, _ptr(out["recv_x"]), _ptr(out["recv_x_scales"]),
                                      _ptr(out["recv_topk_idx"]), _ptr(out["recv_topk_weights"]),
                                      _ptr(out["recv_src_idx"]), _ptr(out["x_scales"]))
    elif threads > 1:
        out["recv_x"] = np.full((cap, H), fill_x & 0xFFFF, np.uint16)
        flags = L.oracle_dispatch_bf16_mt(_ptr(x_bits), T, H, _ptr(topk_idx), _ptr(w), k, num_experts, num_ranks,
                                          _ptr(token_dst_row), cap, _ptr(out["recv_x"]),
                                          _ptr(out["recv_topk_idx"]), _ptr(out["recv_topk_weights"]),
                                          _ptr(out["recv_src_idx"]), int(threads))
    else:
        out["recv_x"] = np.full((cap, H), fill_x & 0xFFFF, np.uint16)
        flags = L.oracle_dispatch_bf16(_ptr(x_bits), T, H, _ptr(topk_idx), _ptr(w), k, num_experts, num_ranks,
                                       _ptr(token_dst_row), cap, _ptr(out["recv_x"]),
                                       _ptr(out["recv_topk_idx"]), _ptr(out["recv_topk_weights"]),
                                       _ptr(out["recv_src_idx"]))
    out["flags"] = flags
    return out


def dispatch_fp8_input(codes: np.ndarray, scales: np.ndarray, topk_idx: np.ndarray,
                       topk_weights: Optional[np.ndarray], num_experts: int, num_ranks: int,
                       token_dst_row: np.ndarray, recv_capacity: int) -> dict:
    """Copies of E4M3 rows [T, H] (uint8) and their scales [T, H/128] per destination."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    token_dst_row = np.ascontiguousarray(token_dst_row, dtype=np.int32)
    w = None if topk_weights is None else np.ascontiguousarray(topk_weights, dtype=np.float32)
    T, H = codes.shape
    k = topk_idx.shape[1]
    cap = recv_capacity
    out = dict(recv_x=np.zeros((cap, H), np.uint8), recv_x_scales=np.zeros((cap, H // 128), np.float32),
               recv_topk_idx=np.zeros((cap, k), np.int64), recv_topk_weights=np.zeros((cap, k), np.float32),
               recv_src_idx=np.zeros(cap, np.int32))
    out["flags"] = lib().oracle_dispatch_fp8_input(
        _ptr(codes), _ptr(scales), T, H, _ptr(topk_idx), _ptr(w), k, num_experts, num_ranks, _ptr(token_dst_row),
        cap, _ptr(out["recv_x"]), _ptr(out["recv_x_scales"]), _ptr(out["recv_topk_idx"]),
        _ptr(out["recv_topk_weights"]), _ptr(out["recv_src_idx"]))
    return out


def combine(partial_bits: np.ndarray, token_dst_row: np.ndarray, threads: int = 1) -> tuple[np.ndarray, int]:
    """bf16 bit patterns [T, H] of the fp32 ascending-rank sums. ``threads`` > 1
    runs it over token ranges on that many threads (same results; for timing)."""
    partial_bits = np.ascontiguousarray(partial_bits, dtype=np.uint16)
    token_dst_row = np.ascontiguousarray(token_dst_row, dtype=np.int32)
    num_rows, H = partial_bits.shape
    T, k = token_dst_row.shape
    out = np.zeros((T, H), np.uint16)
    if threads > 1:
        flags = lib().oracle_combine_mt(_ptr(partial_bits), num_rows, T, H, k, _ptr(token_dst_row), _ptr(out),
                                        int(threads))
    else:
        flags = lib().oracle_combine(_ptr(partial_bits), num_rows, T, H, k, _ptr(token_dst_row), _ptr(out))
    return out, flags


def combine_weighted(partial_bits: np.ndarray, token_dst_row: np.ndarray, row_weights: Optional[np.ndarray],
                     recv_topk_weights: Optional[np.ndarray] = None) -> tuple[np.ndarray, Optional[np.ndarray], int]:
    """(out bf16 bits [T, H], combined top-k weights [T, k] or None, flags)."""
    partial_bits = np.ascontiguousarray(partial_bits, dtype=np.uint16)
    token_dst_row = np.ascontiguousarray(token_dst_row, dtype=np.int32)
    rw = None if row_weights is None else np.ascontiguousarray(row_weights, dtype=np.float32)
    rtw = None if recv_topk_weights is None else np.ascontiguousarray(recv_topk_weights, dtype=np.float32)
    num_rows, H = partial_bits.shape
    T, k = token_dst_row.shape
    out = np.zeros((T, H), np.uint16)
    cw = None if rtw is None else np.zeros((T, k), np.float32)
    flags = lib().oracle_combine_weighted(_ptr(partial_bits), num_rows, T, H, k, _ptr(token_dst_row), _ptr(rw),
                                          _ptr(rtw), _ptr(out), _ptr(cw))
    return out, cw, flags


def expand_layout(topk_idx: np.ndarray, num_experts: int) -> dict:
    """Expand mode: expert_prefix [E+1] and token_expert_row [T, k], one row
    per valid entry, expert regions in expert order, source order inside."""
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, k = topk_idx.shape
    out = dict(expert_prefix=np.zeros(num_experts + 1, np.int32), token_expert_row=np.zeros((T, k), np.int32))
    out["flags"] = lib().oracle_expand_layout(_ptr(topk_idx), T, k, num_experts, _ptr(out["expert_prefix"]),
                                              _ptr(out["token_expert_row"]))
    out["num_recv"] = int(out["expert_prefix"][-1])
    return out


EXPAND_BF16, EXPAND_QUANTIZE_FP8, EXPAND_FP8 = 0, 1, 2


def dispatch_expand(mode: int, x: np.ndarray, topk_idx: np.ndarray, topk_weights: Optional[np.ndarray],
                    num_experts: int, num_ranks: int, token_expert_row: np.ndarray, recv_capacity: int,
                    x_scales: Optional[np.ndarray] = None, fill_x: int = 0, fill_meta: int = 0) -> dict:
    """Expand-mode dispatch. ``x`` is bf16 bit patterns (uint16 [T, H]) for
    modes 0 and 1, E4M3 codes (uint8 [T, H]) with ``x_scales`` for mode 2."""
    x = np.ascontiguousarray(x, dtype=np.uint8 if mode == EXPAND_FP8 else np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    token_expert_row = np.ascontiguousarray(token_expert_row, dtype=np.int32)
    w = None if topk_weights is None else np.ascontiguousarray(topk_weights, dtype=np.float32)
    xs = None if x_scales is None else np.ascontiguousarray(x_scales, dtype=np.float32)
    T, H = x.shape
    k = topk_idx.shape[1]
    cap = recv_capacity
    nb = H // 128
    fp8 = mode != EXPAND_BF16
    out = dict(
        recv_x=(np.full((cap, H), fill_x & 0xFF, np.uint8) if fp8 else np.full((cap, H), fill_x & 0xFFFF, np.uint16)),
        recv_x_scales=np.full((cap, max(nb, 1)), fill_meta, np.int32).view(np.float32) if fp8 else None,
        recv_topk_idx=np.full((cap, k), fill_meta, np.int64),
        recv_topk_weights=np.full((cap, k), fill_meta, np.int32).view(np.float32),
        recv_src_idx=np.full(cap, fill_meta, np.int32),
        x_scales=np.zeros((T, nb), np.float32) if mode == EXPAND_QUANTIZE_FP8 else None,
    )
    out["flags"] = lib().oracle_dispatch_expand(
        mode, _ptr(x), _ptr(xs), T, H, _ptr(topk_idx), _ptr(w), k, num_experts, num_ranks, _ptr(token_expert_row),
        cap, _ptr(out["recv_x"]), _ptr(out["recv_x_scales"]), _ptr(out["recv_topk_idx"]),
        _ptr(out["recv_topk_weights"]), _ptr(out["recv_src_idx"]), _ptr(out["x_scales"]))
    return out


def combine_fp8(codes: np.ndarray, scales: np.ndarray, token_dst_row: np.ndarray) -> tuple[np.ndarray, int]:
    """bf16 bit patterns [T, H] of the ascending fp32 sums of the dequantised
    E4M3 rows (codes uint8 [rows, H], scales fp32 [rows, H/128])."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    token_dst_row = np.ascontiguousarray(token_dst_row, dtype=np.int32)
    num_rows, H = codes.shape
    T, k = token_dst_row.shape
    out = np.zeros((T, H), np.uint16)
    flags = lib().oracle_combine_fp8(_ptr(codes), _ptr(scales), num_rows, T, H, k, _ptr(token_dst_row), _ptr(out))
    return out, flags


def bf16_from_float(v: float) -> int:
    return int(lib().oracle_bf16_from_float(float(v)))


def bf16_to_float(h: int) -> float:
    return float(lib().oracle_bf16_to_float(int(h)))


def e4m3_from_float(v: float) -> int:
    return int(lib().oracle_e4m3_from_float(float(v)))


def e4m3_to_float(c: int) -> float:
    return float(lib().oracle_e4m3_to_float(int(c)))


def bf16_from_float_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint16)
    lib().oracle_bf16_from_float_n(_ptr(v), _ptr(out), v.size)
    return out


def e4m3_from_float_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().oracle_e4m3_from_float_n(_ptr(v), _ptr(out), v.size)
    return out
