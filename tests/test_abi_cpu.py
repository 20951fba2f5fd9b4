"""The C-ABI library builds, loads, exports every symbol its header declares,
and rejects bad arguments on the host before touching CUDA (so these run on a
machine without a GPU; every call below fails validation by design)."""
from __future__ import annotations

import ctypes
import glob
import os
import re

import pytest

from combine_moe_get_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = cuda_build.build()
    from combine_moe_get_gb300 import binding
    assert binding.library_path() == path
    return binding


def _declared_symbols():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = "\n".join(line for line in text.splitlines() if not line.lstrip().startswith("#"))
        names += re.findall(r"MOE_API\s+[^;{]*?\b(\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = _declared_symbols()
    for required in ("moe_get_layout", "moe_dispatch", "moe_combine", "moe_get_layout_workspace_size"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib.library_path())
    for name in _declared_symbols():
        assert hasattr(raw, name), f"{name} declared in include/ but not exported"


def test_version_and_status_strings(lib):
    assert lib.LIB.moe_get_version() >= 100
    for code, name in [(0, "MOE_OK"), (1, "MOE_ERR_INVALID_ARG"), (2, "MOE_ERR_MISALIGNED"),
                       (3, "MOE_ERR_CAPACITY"), (4, "MOE_ERR_BAD_TOPK"), (5, "MOE_ERR_TIMEOUT"),
                       (6, "MOE_ERR_CUDA"), (7, "MOE_ERR_WORKSPACE")]:
        assert lib.status_string(code) == name
    assert lib.status_string(99) == "MOE_ERR_UNKNOWN"


def test_workspace_size(lib):
    ws = lib.moe_get_layout_workspace_size
    assert ws(4096, 256, 8) > 0
    assert ws(0, 256, 8) > 0
    assert ws(1 << 20, 2048, 256) >= (1 << 20) // 128 * 256 * 8
    assert ws(4096, 255, 8) == 0          # E % R != 0
    assert ws(4096, 256, 2048) == 0       # too many ranks
    assert ws(-1, 256, 8) == 0


# Fake device addresses: validation rejects the call before any is dereferenced.
A = 0x7F0000000000          # 256-byte aligned
MIS = A + 2                 # misaligned for anything wider than 2 bytes


def _layout_struct(lib, base=A):
    return lib.MoeLayoutC(base, base + 0x1000, base + 0x2000, base + 0x3000, base + 0x4000, base + 0x5000)


def _layout(lib, T=128, k=2, E=16, R=4, topk=A, ws=A + 0x100000, ws_bytes=1 << 30, status=A + 0x200000, lay=None):
    return lib.LIB.moe_get_layout(topk, T, k, E, R, lay or _layout_struct(lib), ws, ws_bytes, status, None)


@pytest.mark.parametrize("kw,code", [
    (dict(k=0), 1), (dict(k=33), 1), (dict(E=15), 1), (dict(R=0), 1), (dict(R=2048, E=2048), 1),
    (dict(E=16384, R=4), 1), (dict(T=-1), 1), (dict(status=None), 1), (dict(topk=None), 1),
    (dict(ws=None), 1), (dict(topk=MIS), 2), (dict(ws=MIS), 2), (dict(status=MIS), 2),
    (dict(ws_bytes=16), 7),
])
def test_layout_rejects_bad_arguments(lib, kw, code):
    assert _layout(lib, **kw) == code


def test_layout_rejects_null_or_misaligned_outputs(lib):
    s = _layout_struct(lib)
    s.token_dst_row = None
    assert _layout(lib, lay=s) == 1
    s = _layout_struct(lib)
    s.rank_prefix = MIS
    assert _layout(lib, lay=s) == 2


def _dispatch(lib, x=A, T=128, H=256, topk=A + 0x10000, w=None, k=2, E=16, R=4, dst=A + 0x20000, cap=256,
              fp8=0, recv=A + 0x100000, scales=None, status=A + 0x300000):
    return lib.LIB.moe_dispatch(x, T, H, topk, w, k, E, R, dst, cap, fp8, recv, scales, None, None, None, None,
                                status, None)


@pytest.mark.parametrize("kw,code", [
    (dict(H=12), 1), (dict(H=0), 1), (dict(fp8=1, H=264, scales=A + 0x400000), 1), (dict(fp8=1), 1),
    (dict(k=40), 1), (dict(E=17), 1), (dict(cap=-1), 1), (dict(x=None), 1), (dict(recv=None), 1),
    (dict(status=None), 1), (dict(x=A + 8), 2), (dict(recv=A + 8), 2), (dict(dst=MIS), 2),
    (dict(fp8=3), 1), (dict(fp8=2, scales=A + 0x400000), 1), (dict(fp8=-1), 1),
    (dict(fp8=0x103), 1), (dict(fp8=0x200), 1), (dict(fp8=0x102), 1), (dict(fp8=0x101, H=264), 1),
    (dict(fp8=0x100, dst=MIS), 2),
])
def test_dispatch_rejects_bad_arguments(lib, kw, code):
    assert _dispatch(lib, **kw) == code


def _combine(lib, partial=A, rows=256, T=128, H=256, k=2, dst=A + 0x10000, out=A + 0x100000, status=A + 0x200000):
    return lib.LIB.moe_combine(partial, rows, T, H, k, dst, out, status, None)


@pytest.mark.parametrize("kw,code", [
    (dict(H=4), 1), (dict(k=0), 1), (dict(rows=-1), 1), (dict(T=-5), 1), (dict(out=None), 1),
    (dict(partial=None), 1), (dict(dst=None), 1), (dict(status=None), 1), (dict(partial=A + 4), 2),
    (dict(out=A + 8), 2),
])
def test_combine_rejects_bad_arguments(lib, kw, code):
    assert _combine(lib, **kw) == code


def test_expand_workspace_size(lib):
    ws = lib.moe_get_expand_layout_workspace_size
    assert ws(4096, 256) >= 4096 // 256 * 256 * 8
    assert ws(0, 256) > 0
    assert ws(4096, 0) == 0 and ws(4096, 8193) == 0 and ws(-1, 16) == 0


def _expand(lib, T=128, k=2, E=16, topk=A, prefix=A + 0x10000, rows=A + 0x20000, ws=A + 0x100000,
            ws_bytes=1 << 30, status=A + 0x200000):
    return lib.LIB.moe_get_expand_layout(topk, T, k, E, prefix, rows, ws, ws_bytes, status, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(k=0), 1), (dict(k=33), 1), (dict(E=0), 1), (dict(E=8193), 1), (dict(T=-1), 1),
    (dict(status=None), 1), (dict(topk=None), 1), (dict(prefix=None), 1), (dict(rows=None), 1),
    (dict(ws=None), 1), (dict(topk=MIS), 2), (dict(prefix=MIS), 2), (dict(rows=MIS), 2), (dict(ws=A + 8), 2),
    (dict(status=MIS), 2), (dict(ws_bytes=64), 7),
])
def test_expand_layout_rejects_bad_arguments(lib, kw, code):
    assert _expand(lib, **kw) == code


def _layout_dispatch(lib, x=A, T=128, H=256, topk=A + 0x10000, k=2, E=16, R=4, ws=A + 0x300000, ws_bytes=1 << 30,
                     cap=256, mode=0, recv=A + 0x100000, status=A + 0x200000):
    return lib.LIB.moe_layout_dispatch(x, T, H, topk, None, k, E, R, _layout_struct(lib, A + 0x400000), ws, ws_bytes,
                                       cap, mode, recv, None, None, None, None, None, status, None)


@pytest.mark.parametrize("kw,code", [
    (dict(mode=0x100), 1), (dict(mode=3), 1), (dict(H=12), 1), (dict(k=33), 1), (dict(E=15), 1),
    (dict(ws=None), 1), (dict(ws_bytes=16), 7), (dict(x=A + 8), 2), (dict(topk=MIS), 2), (dict(status=None), 1),
    (dict(recv=None), 1), (dict(cap=-1), 1),
])
def test_layout_dispatch_rejects_bad_arguments(lib, kw, code):
    assert _layout_dispatch(lib, **kw) == code


def _combine_fp8(lib, codes=A, scales=A + 0x80000, rows=256, T=128, H=1024, k=2, dst=A + 0x10000, out=A + 0x100000,
                 status=A + 0x200000):
    return lib.LIB.moe_combine_fp8(codes, scales, rows, T, H, k, dst, out, status, None)


@pytest.mark.parametrize("kw,code", [
    (dict(H=256), 1), (dict(H=640), 1), (dict(k=0), 1), (dict(rows=-1), 1), (dict(scales=None), 1),
    (dict(codes=None), 1), (dict(out=None), 1), (dict(status=None), 1), (dict(scales=A + 4), 2),
    (dict(codes=A + 8), 2), (dict(out=A + 8), 2),
])
def test_combine_fp8_rejects_bad_arguments(lib, kw, code):
    assert _combine_fp8(lib, **kw) == code


def _combine_fp8_ex(lib, balance=A + 0x500000, **kw):
    d = dict(codes=A, scales=A + 0x80000, rows=256, T=128, H=1024, k=2, dst=A + 0x10000, out=A + 0x100000,
             status=A + 0x200000)
    d.update(kw)
    return lib.LIB.moe_combine_fp8_ex(d["codes"], d["scales"], d["rows"], d["T"], d["H"], d["k"], d["dst"], d["out"],
                                      balance, d["status"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(balance=A + 4), 2), (dict(H=640), 1), (dict(k=0), 1), (dict(scales=None), 1), (dict(status=None), 1),
    (dict(codes=A + 8), 2), (dict(out=A + 8), 2),
])
def test_combine_fp8_ex_rejects_bad_arguments(lib, kw, code):
    # the same checks as moe_combine_fp8, plus the balance counter's alignment; nothing is launched
    assert _combine_fp8_ex(lib, **kw) == code


def _combine_ex(lib, partial=A, rows=256, T=128, H=256, k=2, dst=A + 0x10000, roww=None, rtw=None, cw=None,
                out=A + 0x100000, balance=None, status=A + 0x200000):
    return lib.LIB.moe_combine_ex(partial, rows, T, H, k, dst, roww, rtw, cw, out, balance, status, None)


@pytest.mark.parametrize("kw,code", [
    (dict(H=4), 1), (dict(k=0), 1), (dict(status=None), 1), (dict(rtw=A + 0x300000), 1), (dict(cw=A + 0x300000), 1),
    (dict(balance=A + 4), 2), (dict(roww=A + 2), 2), (dict(partial=A + 4), 2),
])
def test_combine_ex_rejects_bad_arguments(lib, kw, code):
    assert _combine_ex(lib, **kw) == code


def _dispatch_ex(lib, balance=A + 0x500000, **kw):
    d = dict(x=A, T=128, H=256, topk=A + 0x10000, w=None, k=2, E=16, R=4, dst=A + 0x20000, cap=256, fp8=0,
             recv=A + 0x100000, scales=None, status=A + 0x300000)
    d.update(kw)
    return lib.LIB.moe_dispatch_ex(d["x"], d["T"], d["H"], d["topk"], d["w"], d["k"], d["E"], d["R"], d["dst"],
                                   d["cap"], d["fp8"], d["recv"], d["scales"], None, None, None, None, balance,
                                   d["status"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(balance=A + 4), 2), (dict(H=12), 1), (dict(x=A + 8), 2), (dict(status=None), 1), (dict(fp8=3), 1),
])
def test_dispatch_ex_rejects_bad_arguments(lib, kw, code):
    assert _dispatch_ex(lib, **kw) == code


def test_layout_ex_rejects_unknown_mode(lib):
    opts = lib.MoeLayoutOptionsC(0, -1, 3)
    code = lib.LIB.moe_get_layout_ex(A, 128, 2, 16, 4, _layout_struct(lib), A + 0x100000, 1 << 30, A + 0x200000, None,
                                     ctypes.byref(opts))
    assert code == 1


def test_default_build_records_no_trace(lib):
    # only a build compiled with MOE_PROFILE records; the default one refuses, enabling or not
    assert lib.LIB.moe_trace_enable(None, 0, None, 0) == lib.MOE_ERR_INVALID_ARG


def test_trace_build_exports_the_same_abi(lib):
    from combine_moe_get_gb300 import build
    path = build.build_trace()
    raw = ctypes.CDLL(path)
    for name in _declared_symbols():
        assert hasattr(raw, name), f"{name} missing from the tracing build"
    tl = lib.load_library(path)
    assert tl.moe_get_version() == lib.LIB.moe_get_version()
    assert tl.moe_trace_enable(None, 0, None, 0) == lib.MOE_OK           # stop: accepted with no buffer
    bad = ctypes.c_void_p(8)
    assert tl.moe_trace_enable(bad, 4, None, 3) == lib.MOE_ERR_INVALID_ARG  # a buffer needs a counter
    assert tl.moe_trace_enable(bad, -1, bad, 3) == lib.MOE_ERR_INVALID_ARG
    assert tl.moe_trace_enable(bad, 4, bad, 0) == lib.MOE_ERR_INVALID_ARG   # nothing to record
    assert tl.moe_trace_enable(bad, 4, bad, 4) == lib.MOE_ERR_INVALID_ARG   # unknown bit
    assert tl.moe_trace_enable(None, 0, None, 0) == lib.MOE_OK


def test_trace_record_layout_matches_header(lib):
    text = open(os.path.join(ROOT, "include", "moe_get.h")).read()
    body = re.search(r"typedef struct\s*\{([^}]*)\}\s*moe_trace_record_t;", text, flags=re.S).group(1)
    fields = re.findall(r"\b(uint32_t|uint64_t)\s+(\w+)\s*;", body)
    np_code = {"uint32_t": "<u4", "uint64_t": "<u8"}
    assert [(n, np_code[t]) for t, n in fields] == [(n, lib.TRACE_RECORD[n].str) for n in lib.TRACE_RECORD.names]
    assert lib.TRACE_RECORD.itemsize == 32
    named = {k: int(v, 0) for k, v in re.findall(r"\b(MOE_TRACE_\w+)\s*=\s*(0x[0-9a-fA-F]+|\d+)", text)}
    assert named.pop("MOE_TRACE_PHASE") == lib.TRACE_PHASE
    assert (named.pop("MOE_TRACE_WARPS"), named.pop("MOE_TRACE_PHASES")) == (lib.TRACE_WARPS, lib.TRACE_PHASES)
    assert sorted(named.values()) == sorted(lib.TRACE_KERNELS)
    assert set(lib.TRACE_PHASE_NAMES) <= set(lib.TRACE_KERNELS)
