"""moe_permute_noalloc: the permutation for callers that cannot allocate device memory.

Such callers (code running under CUDA graph capture, serving loops that must
never call cudaMalloc, plugins whose host framework owns all device memory)
get the permutation without a workspace: the library uses its own fixed
device scratch. This file checks, through the C ABI, that two calls in a row
give exactly what moe_permute gives with a workspace, and that sizes beyond
the scratch are refused. It is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workload as W
import sparse_moe_layer_14_b300 as bm
from sparse_moe_layer_14_b300 import _native as N

pytestmark = pytest.mark.gpu


def _permute_both(T, E, K, d, seed, hot=0):
    idx_h = W.random_topk(seed, T, E, K, hot_count=hot, hot_prob=0.5 if hot else 0.0)
    x = torch.from_numpy(W.normal_bf16(seed, W.TID_X, 0, T * d, 1.0).reshape(T, d)).view(torch.int16)
    x = x.view(torch.bfloat16).cuda()
    idx = torch.from_numpy(idx_h).cuda()
    dims = bm.Dims(T, d, E, 1, 1, K, 64)
    R = T * K

    def outputs():
        return (torch.full((E,), -1, dtype=torch.int32, device="cuda"),
                torch.full((E + 1,), -1, dtype=torch.int32, device="cuda"),
                torch.full((R,), -1, dtype=torch.int32, device="cuda"),
                torch.full((R,), -1, dtype=torch.int32, device="cuda"),
                torch.zeros((R, d), dtype=torch.bfloat16, device="cuda"))

    ref = outputs()
    ws = bm.allocate_workspace(dims)
    bm.moe_permute(dims, x, idx, *ref, ws)

    got = outputs()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    lib = N.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.moe_permute_noalloc(ctypes.byref(dims.c()), ctypes.c_void_p(x.data_ptr()),
                                 ctypes.c_void_p(idx.data_ptr()), *[ctypes.c_void_p(t.data_ptr()) for t in got],
                                 ctypes.c_void_p(status.data_ptr()), stream)
    assert rc == N.MOE_OK
    torch.cuda.synchronize()
    assert int(status.item()) == bm.MOE_DEV_OK
    for a, b in zip(ref[:4], got[:4]):
        assert torch.equal(a, b)
    assert torch.equal(ref[4].view(torch.int16), got[4].view(torch.int16))


def test_noalloc_matches_permute_on_two_calls_in_a_row():
    # the larger batch first: the second call must not see the first call's bitmap
    _permute_both(T=3000, E=256, K=8, d=128, seed=41, hot=16)
    _permute_both(T=77, E=16, K=4, d=64, seed=42)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    lib = N.load()
    fake = ctypes.c_void_p(1 << 20)
    dims = N.MoeDims(16385, 128, 16, 1, 1, 4, 64, 2.5, 0)
    rc = lib.moe_permute_noalloc(ctypes.byref(dims), fake, fake, fake, fake, fake, fake, fake, None, None)
    assert rc == N.MOE_ERR_SCRATCH_LIMIT


def test_noalloc_empty_call_reports_ok():
    """T = 0 permutes nothing but still writes MOE_DEV_OK to the caller's status word."""
    lib = N.load()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    dims = N.MoeDims(0, 128, 16, 1, 1, 4, 64, 2.5, 0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.moe_permute_noalloc(ctypes.byref(dims), None, None, None, None, None, None, None,
                                 ctypes.c_void_p(status.data_ptr()), stream)
    assert rc == N.MOE_OK
    torch.cuda.synchronize()
    assert int(status.item()) == bm.MOE_DEV_OK
