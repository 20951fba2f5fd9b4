"""moe_get_layout_noalloc: the layout entry point for callers that cannot
allocate device memory (for instance a plugin inside a host framework that
owns all device allocations and hands out no workspace). It keeps its scratch
in the library's own device array instead of a caller workspace.

Checked through the C ABI against moe_get_layout on the same inputs, on two
calls in a row (the second call reuses the scratch left by the first), and
on its size limit. The file name sorts last so that a run stopping at the
first failure has already run every other test; it also passes alone in a
fresh process (the first call performs the per-device set-up).
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from combine_moe_get_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

KEYS = ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "rank_prefix", "expert_prefix",
        "token_dst_row")


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
    for t in (lay.token_dst_row, lay.is_token_in_rank):
        t.fill_(0x5A)           # poison: everything must be written by the call
    status = moe.new_status(topk.device)
    code = moe.LIB.moe_get_layout_noalloc(ctypes.c_void_p(topk.data_ptr()), T, k, E, R, lay.c(),
                                          ctypes.c_void_p(status.data_ptr()),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return code, lay, status


@pytest.mark.parametrize("name", ["skewed", "dsv3", "decode", "tiny"])
def test_noalloc_layout_matches_layout_twice(moe, name):
    w = wl.CONFIGS[name]
    topk = wl.make_inputs(w, with_partial=False).topk_idx.cuda()
    ref = moe.moe_get_layout(topk, w.num_experts, w.num_ranks)
    torch.cuda.synchronize()
    for _ in range(2):
        code, lay, status = noalloc_layout(moe, topk, w.num_experts, w.num_ranks)
        assert code == moe.MOE_OK, moe.status_string(code)
        torch.cuda.synchronize()
        assert int(status.item()) == moe.MOE_OK
        for key in KEYS:
            np.testing.assert_array_equal(getattr(lay, key).cpu().numpy(), getattr(ref, key).cpu().numpy(),
                                          err_msg=key)


def test_noalloc_layout_rejects_sizes_beyond_scratch(moe):
    # 2^20 tokens over 256 ranks needs a 16 MiB lookback workspace, beyond the 1 MiB scratch
    T, k, E, R = 1 << 20, 8, 2048, 256
    assert moe.moe_get_layout_workspace_size(T, E, R) > (1 << 20)
    topk = torch.zeros(T, k, dtype=torch.int64, device="cuda")
    code, _, status = noalloc_layout(moe, topk, E, R)
    assert code == moe.MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(status.item()) == 0
