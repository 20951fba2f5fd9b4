"""moe_get_layout_noalloc: the layout entry point for callers that cannot
allocate device memory (for instance a plugin inside a host framework that
owns all device allocations and hands out no workspace). It keeps its scratch
in the library's own device array instead of a caller workspace.

Checked through the C ABI against the CPU oracle's layout, on two calls in a
row with different routings (the second call finds the first call's contents
in the scratch), in every layout mode the scratch serves: the cluster mode
(DeepSeek-V3 shape), the direct mode (skewed shape), a single tile (decode and
tiny), the cooperative lookback (16,384 and 65,536 tokens) and the scan
mode (2^20 tokens over 8 ranks, whose 0.5 MiB workspace still fits); and on
its size limit. The file name sorts last so that a run stopping at the
first failure has already run every other test; it also passes alone in a
fresh process (the first call performs the per-device set-up).
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_moe_get_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

KEYS = ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "rank_prefix", "expert_prefix",
        "token_dst_row")
SCRATCH_BYTES = 1 << 20


@pytest.fixture(scope="module")
def moe():
    from combine_moe_get_gb300 import binding
    f = binding.LIB.moe_get_layout_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, binding.MoeLayoutC,
                  ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return binding


def noalloc_layout(moe, topk: torch.Tensor, E: int, R: int):
    T, k = topk.shape
    lay = moe.Layout.empty(T, k, E, R, topk.device)
    for t in (lay.token_dst_row, lay.is_token_in_rank, lay.num_tokens_per_rank, lay.num_tokens_per_expert,
              lay.rank_prefix, lay.expert_prefix):
        t.fill_(0x5A)           # poison: everything must be written by the call
    status = moe.new_status(topk.device)
    code = moe.LIB.moe_get_layout_noalloc(ctypes.c_void_p(topk.data_ptr()), T, k, E, R, lay.c(),
                                          ctypes.c_void_p(status.data_ptr()),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return code, lay, status


def check_twice(moe, routings, E, R):
    for topk in routings:
        ref = oracle.layout(topk.numpy(), E, R)
        assert ref["flags"] == 0
        code, lay, status = noalloc_layout(moe, topk.cuda(), E, R)
        assert code == moe.MOE_OK, moe.status_string(code)
        torch.cuda.synchronize()
        assert int(status.item()) == moe.MOE_OK
        for key in KEYS:
            np.testing.assert_array_equal(getattr(lay, key).cpu().numpy(), ref[key], err_msg=key)


@pytest.mark.parametrize("name", ["skewed", "dsv3", "decode", "tiny"])
def test_noalloc_layout_matches_oracle_twice(moe, name):
    w = wl.CONFIGS[name]
    first = wl.make_inputs(w, with_partial=False).topk_idx
    g = torch.Generator().manual_seed(99)
    second = wl.make_topk_uniform(g, w.num_tokens, w.num_experts, w.num_topk)
    check_twice(moe, [first, second], w.num_experts, w.num_ranks)


@pytest.mark.parametrize("T,E,R", [(16384, 256, 8), (65536, 256, 64), (1 << 20, 256, 8)])
def test_noalloc_layout_lookback_modes_match_oracle_twice(moe, T, E, R):
    # beyond the cluster and direct modes: the lookback kernels and the scan mode,
    # whose tile words live in the scratch, cleared by each call
    assert moe.moe_get_layout_workspace_size(T, E, R) <= SCRATCH_BYTES
    routings = []
    for seed in (T + R, T + R + 1):
        g = torch.Generator().manual_seed(seed)
        routings.append(wl.mask_random_lanes(g, wl.make_topk_uniform(g, T, E, 8), 0.1))
    check_twice(moe, routings, E, R)


def test_noalloc_layout_rejects_sizes_beyond_scratch(moe):
    # 2^20 tokens over 256 ranks needs a 16 MiB lookback workspace, beyond the 1 MiB scratch
    T, k, E, R = 1 << 20, 8, 2048, 256
    assert moe.moe_get_layout_workspace_size(T, E, R) > SCRATCH_BYTES
    topk = torch.zeros(T, k, dtype=torch.int64, device="cuda")
    code, _, status = noalloc_layout(moe, topk, E, R)
    assert code == moe.MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(status.item()) == 0
