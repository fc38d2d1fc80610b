"""Failure detection on the GPU without a GPU fault.

Every pipeline wait in the expert GEMM kernels and in the tensor-core router is
bounded. Forcing the bound to one poll makes the waits expire: the kernels must
latch MOE_DEV_TIMEOUT, drain their own copies and MMAs, free TMEM and return,
leaving the context usable.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
import sparse_moe_layer_14_b300 as bm
from support import DeviceWeights, compare_routing, dev, host_bits

pytestmark = pytest.mark.gpu


def _forward(cfg, inp, dw, ws):
    dims = bm.Dims.from_config(cfg)
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    bm.moe_forward(dims, dev(inp["x"]), dev(inp["w_r"]), dw.dev, out, ws)
    torch.cuda.synchronize()
    return out


def test_wait_timeout_is_reported_and_the_context_recovers():
    cfg = W.MoEConfig("t", T=64, d=1024, E=32, n_groups=8, topk_groups=4, top_k=8, inter=512)
    inp = {"x": W.gen_x(cfg, 3), "w_r": W.gen_wr(cfg, 3)}
    dw = DeviceWeights(cfg, 3, keep_host=False)
    ws = bm.allocate_workspace(bm.Dims.from_config(cfg))
    good = _forward(cfg, inp, dw, ws)
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    bm.moe_set_wait_bound(1)
    try:
        _forward(cfg, inp, dw, ws)
        code = bm.moe_get_device_status(ws, clear=True)
    finally:
        bm.moe_set_wait_bound(0)
    assert code == bm.MOE_DEV_TIMEOUT
    again = _forward(cfg, inp, dw, ws)
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    assert np.array_equal(host_bits(good), host_bits(again))


def test_router_wait_timeout_is_reported_and_the_context_recovers():
    """T = 1100 takes the tensor-core router (mbarrier pipeline, then the bulk-copy ring of the FP32
    recompute): with one poll per wait it latches MOE_DEV_TIMEOUT and returns; the next call on the
    same workspace routes exactly like the oracle."""
    cfg = W.CONFIGS["decode"].with_tokens(1100)
    x_h, wr_h = W.gen_x(cfg, 7), W.gen_wr(cfg, 7)
    dims = bm.Dims.from_config(cfg)
    ws = bm.allocate_workspace(dims)
    x, w_r = dev(x_h), dev(wr_h)
    idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.top_k), dtype=torch.float32, device="cuda")
    bm.moe_set_wait_bound(1)
    try:
        bm.moe_route(dims, x, w_r, idx, w, ws)
        torch.cuda.synchronize()
        code = bm.moe_get_device_status(ws, clear=True)
    finally:
        bm.moe_set_wait_bound(0)
    assert code == bm.MOE_DEV_TIMEOUT
    bm.moe_route(dims, x, w_r, idx, w, ws)
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    compare_routing(cfg, idx.cpu().numpy(), w.cpu().numpy(), O.route(cfg, x_h, wr_h), label="router after timeout")


def test_simt_router_wait_timeout_is_reported_and_the_context_recovers():
    """T = 64 takes the SIMT router (a TMA ring per CTA, clusters of 8 CTAs): with one poll per wait
    it latches MOE_DEV_TIMEOUT, still meets every cluster barrier and counts itself in the
    selection tickets, and returns; the next call on the same workspace routes like the oracle."""
    cfg = W.CONFIGS["decode"].with_tokens(64)
    x_h, wr_h = W.gen_x(cfg, 8), W.gen_wr(cfg, 8)
    dims = bm.Dims.from_config(cfg)
    ws = bm.allocate_workspace(dims)
    x, w_r = dev(x_h), dev(wr_h)
    idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.top_k), dtype=torch.float32, device="cuda")
    bm.moe_set_wait_bound(1)
    try:
        bm.moe_route(dims, x, w_r, idx, w, ws)
        torch.cuda.synchronize()
        code = bm.moe_get_device_status(ws, clear=True)
    finally:
        bm.moe_set_wait_bound(0)
    assert code == bm.MOE_DEV_TIMEOUT
    bm.moe_route(dims, x, w_r, idx, w, ws)
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    compare_routing(cfg, idx.cpu().numpy(), w.cpu().numpy(), O.route(cfg, x_h, wr_h), label="SIMT router after timeout")
