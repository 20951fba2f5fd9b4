"""Thin Python binding of ``libmoe_get.so`` (the C ABI in ``include/moe_get.h``).

Argument marshalling only: every function takes CUDA tensors, allocates the
outputs it is not given with torch (device memory is torch's job here), and
passes raw pointers, sizes and the current CUDA stream to the C entry point
of the same name. All computation runs in the library's CUDA kernels; there
is no CPU path. If the library cannot be built or loaded, import fails.

Errors the host detects come back as ``MoeError``. Errors that depend on the
data land in the int32 ``status`` tensor (first error wins; never cleared by
the library): call ``check_status`` after synchronising.
"""
from __future__ import annotations

import contextlib
import ctypes
import dataclasses
import os
from typing import Optional

import numpy as np

import torch

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_MISALIGNED = 2
MOE_ERR_CAPACITY = 3
MOE_ERR_BAD_TOPK = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_CUDA = 6
MOE_ERR_WORKSPACE = 7

_P = ctypes.c_void_p
_I = ctypes.c_int


class MoeLayoutC(ctypes.Structure):
    _fields_ = [("num_tokens_per_rank", _P), ("num_tokens_per_expert", _P), ("is_token_in_rank", _P),
                ("rank_prefix", _P), ("expert_prefix", _P), ("token_dst_row", _P)]


class MoeLayoutOptionsC(ctypes.Structure):
    _fields_ = [("wait_timeout_ns", ctypes.c_int64), ("test_unpublished_tile", ctypes.c_int32),
                ("layout_mode", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


def library_path() -> str:
    return _build.LIB


def _load():
    if not os.path.exists(_build.LIB) or not _build.up_to_date():
        _build.build()
    return _configure(ctypes.CDLL(_build.LIB))


def load_library(path: str):
    """A configured handle of another build of the library at `path` (e.g. the
    tracing build, build.TRACE_LIB); route the functions below through it with
    `using(handle)`."""
    return _configure(ctypes.CDLL(path))


def _configure(lib):
    lib.moe_get_version.restype = _I
    lib.moe_trace_enable.argtypes = [_P, _I, _P, _I]
    lib.moe_trace_enable.restype = _I
    lib.moe_status_string.argtypes = [_I]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_get_layout_workspace_size.argtypes = [_I, _I, _I]
    lib.moe_get_layout_workspace_size.restype = ctypes.c_size_t
    lib.moe_get_layout.argtypes = [_P, _I, _I, _I, _I, MoeLayoutC, _P, ctypes.c_size_t, _P, _P]
    lib.moe_get_layout.restype = _I
    lib.moe_get_layout_ex.argtypes = [_P, _I, _I, _I, _I, MoeLayoutC, _P, ctypes.c_size_t, _P, _P,
                                      ctypes.POINTER(MoeLayoutOptionsC)]
    lib.moe_get_layout_ex.restype = _I
    lib.moe_get_expand_layout_workspace_size.argtypes = [_I, _I]
    lib.moe_get_expand_layout_workspace_size.restype = ctypes.c_size_t
    lib.moe_get_expand_layout.argtypes = [_P, _I, _I, _I, _P, _P, _P, ctypes.c_size_t, _P, _P,
                                          ctypes.POINTER(MoeLayoutOptionsC)]
    lib.moe_get_expand_layout.restype = _I
    lib.moe_dispatch.argtypes = [_P, _I, _I, _P, _P, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]
    lib.moe_dispatch.restype = _I
    lib.moe_dispatch_ex.argtypes = [_P, _I, _I, _P, _P, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    lib.moe_dispatch_ex.restype = _I
    lib.moe_layout_dispatch.argtypes = [_P, _I, _I, _P, _P, _I, _I, _I, MoeLayoutC, _P, ctypes.c_size_t, _I, _I, _P,
                                        _P, _P, _P, _P, _P, _P, _P]
    lib.moe_layout_dispatch.restype = _I
    lib.moe_combine.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P]
    lib.moe_combine.restype = _I
    lib.moe_combine_fp8.argtypes = [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P]
    lib.moe_combine_fp8.restype = _I
    lib.moe_combine_fp8_ex.argtypes = [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]
    lib.moe_combine_fp8_ex.restype = _I
    lib.moe_combine_ex.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]
    lib.moe_combine_ex.restype = _I
    return lib


LIB = _load()


@contextlib.contextmanager
def using(lib):
    """Within the block, every function of this module calls `lib` (a handle from
    load_library) instead of the default build."""
    global LIB
    old, LIB = LIB, lib
    try:
        yield lib
    finally:
        LIB = old


# moe_trace_record_t, as written by a build with MOE_PROFILE
TRACE_RECORD = np.dtype([("kernel", "<u4"), ("cta", "<u4"), ("warp", "<u4"), ("sm", "<u4"),
                         ("start_ns", "<u8"), ("end_ns", "<u8")])
TRACE_KERNELS = {1: "layout_tiles", 2: "layout_direct", 3: "layout_cluster", 4: "layout_count", 5: "layout_scan",
                 6: "layout_rows_scan", 7: "expand_layout", 8: "expand_layout_cluster", 9: "dispatch",
                 10: "dispatch_fp8_rows", 11: "combine", 12: "layout_rows"}
TRACE_PHASE = 0x10000   # warp field of a per-CTA phase record: TRACE_PHASE + phase (1, 2, ...)
TRACE_PHASE_NAMES = {3: ("dependency wait", "top-k tile loaded", "bitmap and expert histogram",
                         "tile counts and first cluster barrier", "exchange and second barrier",
                         "prefixes and count writes", "receive rows", "is_token_in_rank rows"),
                     9: ("set-up (behind the layout: first loads, L2 prefetch)", "dependency wait",
                         "fused small-batch layout", "the rest"),
                     10: ("set-up", "dependency wait", "the rest"),
                     11: ("set-up", "dependency wait", "the rest")}


TRACE_WARPS, TRACE_PHASES = 1, 2


def trace_enable(records: Optional[torch.Tensor], count: Optional[torch.Tensor],
                 what: int = TRACE_WARPS | TRACE_PHASES) -> None:
    """Send the records of later launches (`what`: TRACE_WARPS, a record per
    warp; TRACE_PHASES, per-CTA phases) to `records` (a CUDA uint8 tensor of
    n * TRACE_RECORD.itemsize bytes) and count them in `count` (a zeroed CUDA
    int32 tensor of one element); None stops. Needs a build with MOE_PROFILE."""
    if records is None:
        _check(LIB.moe_trace_enable(None, 0, None, 0), "moe_trace_enable")
        return
    cap = records.numel() // TRACE_RECORD.itemsize
    _check(LIB.moe_trace_enable(_ptr(records), cap, _ptr(count), int(what)), "moe_trace_enable")


def trace_read(records: torch.Tensor, count: torch.Tensor) -> np.ndarray:
    """The records written so far (after the stream has synchronised)."""
    n = min(int(count.item()), records.numel() // TRACE_RECORD.itemsize)
    return records[: n * TRACE_RECORD.itemsize].cpu().numpy().view(TRACE_RECORD)


def trace_split(rec: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(per-warp records, per-CTA phase records) of trace_read's result."""
    phase = rec["warp"] >= TRACE_PHASE
    return rec[~phase], rec[phase]


def status_string(code: int) -> str:
    return LIB.moe_status_string(int(code)).decode()


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmoe_get takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("libmoe_get takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(code: int, where: str) -> None:
    if code != MOE_OK:
        raise MoeError(code, where)


def new_status(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def new_balance_counter(device=None) -> torch.Tensor:
    """Two zeroed uint32 (as int32) for the combine's tail balancing; each call leaves them zero."""
    return torch.zeros(2, dtype=torch.int32, device=device or "cuda")


def check_status(status: torch.Tensor, where: str = "kernel") -> None:
    code = int(status.item())
    if code != MOE_OK:
        raise MoeError(code, where)


@dataclasses.dataclass
class Layout:
    num_tokens_per_rank: torch.Tensor     # [R] int32
    num_tokens_per_expert: torch.Tensor   # [E] int32
    is_token_in_rank: torch.Tensor        # [T, R] uint8
    rank_prefix: torch.Tensor             # [R+1] int32
    expert_prefix: torch.Tensor           # [E+1] int32
    token_dst_row: torch.Tensor           # [T, k] int32

    @staticmethod
    def empty(num_tokens: int, num_topk: int, num_experts: int, num_ranks: int, device) -> "Layout":
        i32 = dict(dtype=torch.int32, device=device)
        return Layout(torch.empty(num_ranks, **i32), torch.empty(num_experts, **i32),
                      torch.empty(num_tokens, num_ranks, dtype=torch.uint8, device=device),
                      torch.empty(num_ranks + 1, **i32), torch.empty(num_experts + 1, **i32),
                      torch.empty(num_tokens, num_topk, **i32))

    def c(self) -> MoeLayoutC:
        return MoeLayoutC(*(_ptr(getattr(self, f.name)) for f in dataclasses.fields(self)))


def moe_get_layout_workspace_size(num_tokens: int, num_experts: int, num_ranks: int) -> int:
    return int(LIB.moe_get_layout_workspace_size(num_tokens, num_experts, num_ranks))


def moe_get_layout(topk_idx: torch.Tensor, num_experts: int, num_ranks: int, *,
                   out: Optional[Layout] = None, workspace: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None, stream=None,
                   wait_timeout_ns: int = 0, test_unpublished_tile: int = -1, layout_mode: int = 0) -> Layout:
    """Counts, membership, prefixes and receive rows of ``topk_idx`` [T, k] int64.
    ``layout_mode`` 1 keeps the call off the cluster mode, 2 on the lookback modes (same outputs)."""
    T, k = topk_idx.shape
    dev = topk_idx.device
    out = out or Layout.empty(T, k, num_experts, num_ranks, dev)
    ws_bytes = moe_get_layout_workspace_size(T, num_experts, num_ranks)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    status = new_status(dev) if status is None else status
    opts = MoeLayoutOptionsC(int(wait_timeout_ns), int(test_unpublished_tile), int(layout_mode))
    code = LIB.moe_get_layout_ex(_ptr(topk_idx), T, k, num_experts, num_ranks, out.c(), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream),
                                 ctypes.byref(opts))
    _check(code, "moe_get_layout")
    return out


def moe_get_expand_layout_workspace_size(num_tokens: int, num_experts: int) -> int:
    return int(LIB.moe_get_expand_layout_workspace_size(num_tokens, num_experts))


def moe_get_expand_layout(topk_idx: torch.Tensor, expert_prefix: torch.Tensor, num_experts: int, *,
                          out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                          status: Optional[torch.Tensor] = None, stream=None, wait_timeout_ns: int = 0,
                          test_unpublished_tile: int = -1, layout_mode: int = 0) -> torch.Tensor:
    """Expand-mode receive rows [T, k] int32 (one per valid entry, grouped by
    expert); ``expert_prefix`` is the layout's [E+1] prefix for ``topk_idx``."""
    T, k = topk_idx.shape
    dev = topk_idx.device
    out = torch.empty(T, k, dtype=torch.int32, device=dev) if out is None else out
    ws_bytes = moe_get_expand_layout_workspace_size(T, num_experts)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    status = new_status(dev) if status is None else status
    opts = MoeLayoutOptionsC(int(wait_timeout_ns), int(test_unpublished_tile), int(layout_mode))
    code = LIB.moe_get_expand_layout(_ptr(topk_idx), T, k, num_experts, _ptr(expert_prefix), _ptr(out),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
                                     _stream(stream), ctypes.byref(opts))
    _check(code, "moe_get_expand_layout")
    return out


@dataclasses.dataclass
class Dispatched:
    recv_x: torch.Tensor                      # [capacity, H] bf16 or uint8 (E4M3 codes)
    recv_x_scales: Optional[torch.Tensor]     # [capacity, H/128] fp32 (FP8)
    recv_topk_idx: Optional[torch.Tensor]     # [capacity, k] int64
    recv_topk_weights: Optional[torch.Tensor] # [capacity, k] fp32
    recv_src_idx: Optional[torch.Tensor]      # [capacity] int32
    x_scales: Optional[torch.Tensor]          # [T, H/128] fp32 (FP8)


MOE_DISPATCH_BF16 = 0
MOE_DISPATCH_QUANTIZE_FP8 = 1
MOE_DISPATCH_FP8 = 2
MOE_DISPATCH_EXPAND = 0x100


def moe_dispatch(x: torch.Tensor, topk_idx: torch.Tensor, topk_weights: Optional[torch.Tensor],
                 num_experts: int, num_ranks: int, token_dst_row: torch.Tensor, recv_capacity: int, *,
                 quantize_fp8: bool = False, x_scales: Optional[torch.Tensor] = None, expand: bool = False,
                 out: Optional[Dispatched] = None, with_metadata: bool = True,
                 balance: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                 stream=None) -> Dispatched:
    """Row copies and per-row metadata. ``x`` bf16 is copied as is, or quantised
    to E4M3 with per-128 scales when ``quantize_fp8``; ``x`` uint8 (E4M3 codes)
    is copied together with its ``x_scales`` [T, H/128]. With ``expand``,
    ``token_dst_row`` is the expand layout's token_expert_row. ``balance``
    (new_balance_counter()) calls moe_dispatch_ex, which spreads the last units
    over the SMs."""
    T, H = x.shape
    k = topk_idx.shape[1]
    dev = x.device
    fp8_in = x.dtype == torch.uint8
    mode = MOE_DISPATCH_FP8 if fp8_in else (MOE_DISPATCH_QUANTIZE_FP8 if quantize_fp8 else MOE_DISPATCH_BF16)
    fp8_out = mode != MOE_DISPATCH_BF16
    if fp8_in and x_scales is None:
        raise ValueError("E4M3 input needs its x_scales")
    if out is None:
        nb = H // 128
        out = Dispatched(
            recv_x=torch.empty(recv_capacity, H, dtype=torch.uint8 if fp8_out else torch.bfloat16, device=dev),
            recv_x_scales=torch.empty(recv_capacity, nb, dtype=torch.float32, device=dev) if fp8_out else None,
            recv_topk_idx=torch.empty(recv_capacity, k, dtype=torch.int64, device=dev) if with_metadata else None,
            recv_topk_weights=(torch.empty(recv_capacity, k, dtype=torch.float32, device=dev)
                               if with_metadata else None),
            recv_src_idx=torch.empty(recv_capacity, dtype=torch.int32, device=dev) if with_metadata else None,
            x_scales=(x_scales if fp8_in else
                      (torch.empty(T, nb, dtype=torch.float32, device=dev) if quantize_fp8 else None)))
    status = new_status(dev) if status is None else status
    scales_arg = x_scales if fp8_in else out.x_scales
    args = (_ptr(x), T, H, _ptr(topk_idx), _ptr(topk_weights), k, num_experts, num_ranks, _ptr(token_dst_row),
            recv_capacity, mode | (MOE_DISPATCH_EXPAND if expand else 0), _ptr(out.recv_x), _ptr(out.recv_x_scales),
            _ptr(out.recv_topk_idx), _ptr(out.recv_topk_weights), _ptr(out.recv_src_idx), _ptr(scales_arg))
    if balance is None:
        code = LIB.moe_dispatch(*args, _ptr(status), _stream(stream))
    else:
        code = LIB.moe_dispatch_ex(*args, _ptr(balance), _ptr(status), _stream(stream))
    _check(code, "moe_dispatch")
    return out


def moe_layout_dispatch(x: torch.Tensor, topk_idx: torch.Tensor, topk_weights: Optional[torch.Tensor],
                        num_experts: int, num_ranks: int, recv_capacity: int, *, quantize_fp8: bool = False,
                        x_scales: Optional[torch.Tensor] = None, layout: Optional[Layout] = None,
                        workspace: Optional[torch.Tensor] = None, out: Optional[Dispatched] = None,
                        with_metadata: bool = True, status: Optional[torch.Tensor] = None,
                        stream=None) -> tuple[Layout, Dispatched]:
    """moe_get_layout + moe_dispatch in one call (one launch for small batches)."""
    T, H = x.shape
    k = topk_idx.shape[1]
    dev = x.device
    fp8_in = x.dtype == torch.uint8
    mode = MOE_DISPATCH_FP8 if fp8_in else (MOE_DISPATCH_QUANTIZE_FP8 if quantize_fp8 else MOE_DISPATCH_BF16)
    fp8_out = mode != MOE_DISPATCH_BF16
    if fp8_in and x_scales is None:
        raise ValueError("E4M3 input needs its x_scales")
    layout = layout or Layout.empty(T, k, num_experts, num_ranks, dev)
    ws_bytes = moe_get_layout_workspace_size(T, num_experts, num_ranks)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    if out is None:
        nb = H // 128
        out = Dispatched(
            recv_x=torch.empty(recv_capacity, H, dtype=torch.uint8 if fp8_out else torch.bfloat16, device=dev),
            recv_x_scales=torch.empty(recv_capacity, nb, dtype=torch.float32, device=dev) if fp8_out else None,
            recv_topk_idx=torch.empty(recv_capacity, k, dtype=torch.int64, device=dev) if with_metadata else None,
            recv_topk_weights=(torch.empty(recv_capacity, k, dtype=torch.float32, device=dev)
                               if with_metadata else None),
            recv_src_idx=torch.empty(recv_capacity, dtype=torch.int32, device=dev) if with_metadata else None,
            x_scales=(x_scales if fp8_in else
                      (torch.empty(T, nb, dtype=torch.float32, device=dev) if quantize_fp8 else None)))
    status = new_status(dev) if status is None else status
    scales_arg = x_scales if fp8_in else out.x_scales
    code = LIB.moe_layout_dispatch(_ptr(x), T, H, _ptr(topk_idx), _ptr(topk_weights), k, num_experts, num_ranks,
                                   layout.c(), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   recv_capacity, mode, _ptr(out.recv_x), _ptr(out.recv_x_scales),
                                   _ptr(out.recv_topk_idx), _ptr(out.recv_topk_weights), _ptr(out.recv_src_idx),
                                   _ptr(scales_arg), _ptr(status), _stream(stream))
    _check(code, "moe_layout_dispatch")
    return layout, out


def moe_combine(partial: torch.Tensor, token_dst_row: torch.Tensor, *, out: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[t] = bf16(fp32 sum of partial rows of token t in ascending rank order)."""
    rows, H = partial.shape
    T, k = token_dst_row.shape
    dev = partial.device
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev) if out is None else out
    status = new_status(dev) if status is None else status
    code = LIB.moe_combine(_ptr(partial), rows, T, H, k, _ptr(token_dst_row), _ptr(out), _ptr(status),
                           _stream(stream))
    _check(code, "moe_combine")
    return out


def moe_combine_fp8(partial_codes: torch.Tensor, partial_scales: torch.Tensor, token_dst_row: torch.Tensor, *,
                    out: Optional[torch.Tensor] = None, balance: Optional[torch.Tensor] = None,
                    status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[t] = bf16(fp32 ascending sum over the rows of t of RN(e4m3(code) * scale)).
    With `balance` (new_balance_counter()) this calls moe_combine_fp8_ex."""
    rows, H = partial_codes.shape
    T, k = token_dst_row.shape
    dev = partial_codes.device
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev) if out is None else out
    status = new_status(dev) if status is None else status
    if balance is None:
        code = LIB.moe_combine_fp8(_ptr(partial_codes), _ptr(partial_scales), rows, T, H, k, _ptr(token_dst_row),
                                   _ptr(out), _ptr(status), _stream(stream))
        _check(code, "moe_combine_fp8")
    else:
        code = LIB.moe_combine_fp8_ex(_ptr(partial_codes), _ptr(partial_scales), rows, T, H, k,
                                      _ptr(token_dst_row), _ptr(out), _ptr(balance), _ptr(status), _stream(stream))
        _check(code, "moe_combine_fp8_ex")
    return out


def moe_combine_ex(partial: torch.Tensor, token_dst_row: torch.Tensor, *, row_weights: Optional[torch.Tensor] = None,
                   recv_topk_weights: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                   combined_topk_weights: Optional[torch.Tensor] = None, balance: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None,
                   stream=None) -> tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Combine with per-row weights (fma per term) and/or the reduction of the
    received top-k weights back to [T, k], and optionally a balance counter
    (new_balance_counter()) that spreads the last tokens over the SMs.
    Returns (out, combined_topk_weights)."""
    rows, H = partial.shape
    T, k = token_dst_row.shape
    dev = partial.device
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev) if out is None else out
    if recv_topk_weights is not None and combined_topk_weights is None:
        combined_topk_weights = torch.empty(T, k, dtype=torch.float32, device=dev)
    status = new_status(dev) if status is None else status
    code = LIB.moe_combine_ex(_ptr(partial), rows, T, H, k, _ptr(token_dst_row), _ptr(row_weights),
                              _ptr(recv_topk_weights), _ptr(combined_topk_weights), _ptr(out), _ptr(balance),
                              _ptr(status), _stream(stream))
    _check(code, "moe_combine_ex")
    return out, combined_topk_weights
