"""The oracle's thread-parallel forms (used only to time the oracle on every
host core) give the single-threaded results byte for byte: receive rows,
metadata, combine outputs and result flags, for thread counts that do and do
not divide the token count, more threads than tokens, and inputs with masked,
duplicate and invalid entries and a capacity overflow."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_moe_get_gb300 import workloads as wl


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _case(seed, T, H, k, E, R, mask=0.2):
    g = torch.Generator().manual_seed(seed)
    topk = wl.mask_random_lanes(g, wl.make_topk_uniform(g, T, E, k), mask)
    x = _bits(wl.make_x(g, T, H))
    w = wl.make_weights(g, T, k).numpy()
    partial = _bits(wl.make_partial(g, max(wl.recv_capacity(T, k, R), 1), H))
    return topk.numpy(), x, w, partial


@pytest.mark.parametrize("threads", [2, 3, 7, 16, 300])
@pytest.mark.parametrize("T,H,k,E,R", [(257, 96, 8, 256, 8), (100, 64, 6, 48, 3), (5, 32, 4, 16, 16)])
def test_threaded_dispatch_and_combine_equal_single_thread(threads, T, H, k, E, R):
    topk, x, w, partial = _case(T * 31 + threads, T, H, k, E, R)
    lay = oracle.layout(topk, E, R)
    cap = wl.recv_capacity(T, k, R)
    one = oracle.dispatch(x, topk, w, E, R, lay["token_dst_row"], cap, fill_x=0x7FBF, fill_meta=-7)
    many = oracle.dispatch(x, topk, w, E, R, lay["token_dst_row"], cap, fill_x=0x7FBF, fill_meta=-7,
                           threads=threads)
    for key in ("recv_x", "recv_topk_idx", "recv_src_idx"):
        np.testing.assert_array_equal(many[key], one[key], err_msg=key)
    np.testing.assert_array_equal(many["recv_topk_weights"].view(np.uint32), one["recv_topk_weights"].view(np.uint32))
    assert many["flags"] == one["flags"]
    c1, f1 = oracle.combine(partial, lay["token_dst_row"])
    cn, fn = oracle.combine(partial, lay["token_dst_row"], threads=threads)
    np.testing.assert_array_equal(cn, c1)
    assert fn == f1


def test_threaded_forms_flag_bad_entries_and_capacity():
    T, H, k, E, R = 300, 64, 8, 64, 8
    g = torch.Generator().manual_seed(3)
    topk = torch.randint(0, E, (T, k), generator=g)      # duplicates inside rows
    topk[::9] = -1
    topk[5, 3] = E + 2                                   # invalid entry
    topk = topk.numpy()
    x = _bits(wl.make_x(g, T, H))
    lay = oracle.layout(topk, E, R)
    cap = lay["num_recv"] - 13                           # the last rows overflow the capacity
    one = oracle.dispatch(x, topk, None, E, R, lay["token_dst_row"], cap)
    many = oracle.dispatch(x, topk, None, E, R, lay["token_dst_row"], cap, threads=5)
    assert one["flags"] & oracle.ORACLE_CAPACITY
    assert many["flags"] == one["flags"]
    np.testing.assert_array_equal(many["recv_x"], one["recv_x"])
    partial = _bits(wl.make_partial(g, cap, H))          # fewer partial rows than the layout names
    c1, f1 = oracle.combine(partial, lay["token_dst_row"])
    cn, fn = oracle.combine(partial, lay["token_dst_row"], threads=5)
    assert f1 & oracle.ORACLE_CAPACITY and fn == f1
    np.testing.assert_array_equal(cn, c1)


def test_threaded_forms_empty_batch():
    topk = np.zeros((0, 8), np.int64)
    lay = oracle.layout(topk, 256, 8)
    d = oracle.dispatch(np.zeros((0, 64), np.uint16), topk, None, 256, 8, lay["token_dst_row"], 0, threads=4)
    assert d["flags"] == 0
    out, flags = oracle.combine(np.zeros((1, 64), np.uint16), lay["token_dst_row"], threads=4)
    assert out.shape == (0, 64) and flags == 0
