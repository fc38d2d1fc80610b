"""GPU parity: every step of the CUDA path, through the C ABI, against the CPU oracle
on the same seeded inputs.

Bars: routing bit-exact (expert sets, slot order, per-expert counts) outside
near-ties (margin < 1e-6, excluded and checked for validity), permutation
bit-exact, layer outputs within max|err| <= 2e-2 * RMS(oracle) for bf16 weights (5e-2 for NVFP4 and
FP8 weights).
Full-size cases run in the launch configuration the benchmark times
(moe_forward on the whole batch) and compare sampled tokens one by one.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import workload as W
import sparse_moe_layer_14_b300 as bm
from support import (RMS_BAR, TOL, TOL_BF16, TOL_FP8, TOL_NVFP4, DeviceWeights, bf16_to_f64, check_output,
                     compare_routing, dev, host_bits, plan_n_max, report, work_item_rows)

pytestmark = pytest.mark.gpu

TINY = W.CONFIGS["tiny"]


def run_forward(cfg, x, w_r, weights, T=None):
    dims = bm.Dims.from_config(cfg, T)
    ws = bm.allocate_workspace(dims)
    out = torch.empty((dims.T, dims.d), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((dims.T, dims.top_k), dtype=torch.int32, device="cuda")
    counts = torch.empty((dims.E,), dtype=torch.int32, device="cuda")
    bm.moe_forward(dims, x, w_r, weights, out, ws, topk_idx=idx, counts=counts)
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    return out, idx, counts, ws


def route_only(cfg, x_h, wr_h):
    dims = bm.Dims.from_config(cfg, x_h.shape[0])
    ws = bm.allocate_workspace(dims)
    idx = torch.empty((dims.T, dims.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((dims.T, dims.top_k), dtype=torch.float32, device="cuda")
    bm.moe_route(dims, dev(x_h), dev(wr_h), idx, w, ws)
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    return idx.cpu().numpy(), w.cpu().numpy()


# ---------------------------------------------------------------------------------------- router

@pytest.mark.parametrize("name,T,seed", [("tiny", 64, 0), ("tiny", 77, 1), ("tiny", 1, 2), ("decode", 64, 0),
                                         ("decode", 1000, 3), ("prefill", 4096, 0),
                                         # batches of >= 1024 tokens take the tensor-core router
                                         ("tiny", 1500, 8), ("decode", 1100, 9), ("skewed", 2048, 10)])
def test_route_parity(name, T, seed):
    cfg = W.CONFIGS[name].with_tokens(T)
    x_h, wr_h = W.gen_x(cfg, seed), W.gen_wr(cfg, seed)
    gi, gw = route_only(cfg, x_h, wr_h)
    orc = O.route(cfg, x_h, wr_h)
    excluded, _, _ = compare_routing(cfg, gi, gw, orc)
    assert excluded.size <= max(2, T // 200)


@pytest.mark.parametrize("name,T,seed", [("tiny", 64, 21), ("decode", 64, 22), ("decode", 1100, 23),
                                         ("prefill", 2048, 24)])
def test_route_parity_selection_bias(name, T, seed):
    """Per-expert selection bias (DeepSeek-V3-style balancing): choice on s + b, weights on s;
    SIMT router (T < 1024) and tensor-core router with its fp32 recompute (T >= 1024)."""
    cfg = W.CONFIGS[name].with_tokens(T)
    x_h, wr_h = W.gen_x(cfg, seed), W.gen_wr(cfg, seed)
    bias = (0.1 * (W.uniform_f64(seed, W.TID_AUX + 7, 0, cfg.E) - 0.5)).astype(np.float32)
    dims = bm.Dims.from_config(cfg)
    ws = bm.allocate_workspace(dims)
    idx = torch.empty((T, cfg.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.top_k), dtype=torch.float32, device="cuda")
    bm.moe_route(dims, dev(x_h), dev(wr_h), idx, w, ws, sel_bias=dev(bias))
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    gi, gw = idx.cpu().numpy(), w.cpu().numpy()
    orc = O.route(cfg, x_h, wr_h, bias=bias)
    excluded, _, _ = compare_routing(cfg, gi, gw, orc, bias=bias)
    assert excluded.size <= max(2, T // 200)
    # the bias changes the choice of some tokens, so the biased path is the one tested
    assert np.any(np.sort(orc["idx"], 1) != np.sort(O.route(cfg, x_h, wr_h)["idx"], 1))


def test_forward_selection_bias():
    cfg = TINY.with_tokens(96)
    inp = W.make_host_inputs(cfg, 25)
    bias = (0.2 * (W.uniform_f64(25, W.TID_AUX + 7, 0, cfg.E) - 0.5)).astype(np.float32)
    dw = DeviceWeights(cfg, 25)
    dims = bm.Dims.from_config(cfg)
    ws = bm.allocate_workspace(dims)
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    bm.moe_forward(dims, dev(inp["x"]), dev(inp["w_r"]), dw.dev, out, ws, topk_idx=idx, sel_bias=dev(bias))
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    orc = O.route(cfg, inp["x"], inp["w_r"], bias=bias)
    gi = idx.cpu().numpy()
    s = orc["scores"].astype(np.float64)
    sv = np.take_along_axis(s, gi.astype(np.int64), 1)
    w_like = (cfg.routed_scale * sv / sv.sum(1, keepdims=True)).astype(np.float32)  # unbiased weights
    _, ref_idx, ref_w = compare_routing(cfg, gi, w_like, orc, bias=bias)
    ref = O.forward_tokens(cfg, inp["x"], ref_idx, ref_w, np.arange(cfg.T), dw.host)
    check_output(host_bits(out), ref, TOL_BF16)


@pytest.mark.parametrize("case", ["x16", "wr4", "bias", "outliers", "aligned"])
def test_route_tensor_core_guard(case):
    """The tensor-core router keeps its decision only where every margin exceeds a logit-error bound
    that scales with |x_t| and the column norms of W_r; it must still route like the oracle on
    inputs far from the Beam-shape ones: activations x16 (logits saturate the sigmoid: many exact
    ties, checked for validity), router weights x4, a strong selection bias, outlier channels
    (1 % of the hidden dimension at 20x), and router columns aligned with the token mean (large
    logits)."""
    cfg = W.CONFIGS["prefill"].with_tokens(2048)
    seed = 50 + ["x16", "wr4", "bias", "outliers", "aligned"].index(case)
    x_h, wr_h = W.gen_x(cfg, seed), W.gen_wr(cfg, seed)
    xf = W.bf16_to_f32(x_h)
    bias = None
    if case == "x16":
        xf = xf * 16
    elif case == "wr4":
        wr_h = wr_h * np.float32(4)
    elif case == "bias":
        bias = (0.5 * (W.uniform_f64(seed, W.TID_AUX + 7, 0, cfg.E) - 0.5)).astype(np.float32)
    elif case == "outliers":
        xf[:, ::100] *= 20
    else:
        m = xf.mean(0) + 0.5
        wr_h = (wr_h + 0.05 * (m / np.linalg.norm(m))[:, None]).astype(np.float32)
        xf = xf + 0.5
    x_h = torch.from_numpy(np.ascontiguousarray(xf, np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    x_h = x_h.view(np.uint16)
    dims = bm.Dims.from_config(cfg)
    ws = bm.allocate_workspace(dims)
    idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.top_k), dtype=torch.float32, device="cuda")
    bm.moe_route(dims, dev(x_h), dev(wr_h), idx, w, ws, sel_bias=None if bias is None else dev(bias))
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    flagged = int(ws[16:20].view(torch.int32).item())
    orc = O.route(cfg, x_h, wr_h, bias=bias)
    ex, _, _ = compare_routing(cfg, idx.cpu().numpy(), w.cpu().numpy(), orc, bias=bias,
                               label=f"tensor-core guard {case} T={cfg.T} ({flagged} tokens recomputed in fp32)")


def test_route_uniform_scores():
    """W_r = 0: every score is 0.5, lowest-index groups/experts win, w = 2.5/8 = 0.3125."""
    cfg = W.CONFIGS["decode"].with_tokens(40)
    x_h = W.gen_x(cfg, 1)
    gi, gw = route_only(cfg, x_h, np.zeros((cfg.d, cfg.E), np.float32))
    assert np.array_equal(gi, np.tile(np.arange(8, dtype=np.int32), (40, 1)))
    assert np.all(gw == np.float32(0.3125))


@pytest.mark.parametrize("name,T,seed", [("tiny", 77, 31), ("decode", 64, 32), ("decode", 1100, 33)])
def test_route_strong_selection_bias(name, T, seed):
    """A selection bias of a few units (most selection scores s + b negative, some below -1):
    the selection works on exact order keys of s + b, so no sentinel value can collide with a real
    score; SIMT (T < 1024) and tensor-core (T >= 1024) routers."""
    cfg = W.CONFIGS[name].with_tokens(T)
    x_h, wr_h = W.gen_x(cfg, seed), W.gen_wr(cfg, seed)
    bias = (6.0 * (W.uniform_f64(seed, W.TID_AUX + 7, 0, cfg.E) - 0.7)).astype(np.float32)
    dims = bm.Dims.from_config(cfg)
    ws = bm.allocate_workspace(dims)
    idx = torch.empty((T, cfg.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.top_k), dtype=torch.float32, device="cuda")
    bm.moe_route(dims, dev(x_h), dev(wr_h), idx, w, ws, sel_bias=dev(bias))
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    orc = O.route(cfg, x_h, wr_h, bias=bias)
    assert np.mean(orc["scores"] + bias < -1.0) > 0.2
    excluded, _, _ = compare_routing(cfg, idx.cpu().numpy(), w.cpu().numpy(), orc, bias=bias,
                                     label=f"strong bias {name} T={T}")
    assert excluded.size <= max(2, T // 200)


@pytest.mark.parametrize("E,G,Gk,K,T,d", [(18, 6, 3, 4, 50, 192),   # E not a multiple of 4: padded W_r copy
                                          (7, 1, 1, 3, 9, 64),       # one group
                                          (8, 8, 4, 2, 130, 128),    # one expert per group
                                          (96, 32, 8, 20, 65, 256),  # 32 groups, 20 slots
                                          (16, 4, 2, 4, 1536, 192),  # the largest batch the logits kernel selects in
                                          (16, 4, 2, 4, 1600, 192)]) # selection in a kernel of its own
def test_route_simt_shapes(E, G, Gk, K, T, d):
    """SIMT router over shapes away from the Beam one: expert counts that are not a multiple of
    the 16-expert tile or of 4, one group, one expert per group, 32 groups, a hidden dimension
    shorter than the 8-way split (d = 64: some CTAs of a cluster add nothing), and batches on
    either side of the largest one whose selection runs inside the logits kernel (d = 192 keeps
    T >= 1024 off the tensor-core router)."""
    cfg = W.MoEConfig("simt", T=T, d=d, E=E, n_groups=G, topk_groups=Gk, top_k=K, inter=64)
    x_h, wr_h = W.gen_x(cfg, 40 + E), W.gen_wr(cfg, 40 + E)
    gi, gw = route_only(cfg, x_h, wr_h)
    excluded, _, _ = compare_routing(cfg, gi, gw, O.route(cfg, x_h, wr_h), label=f"SIMT E={E} G={G} T={T} d={d}")
    assert excluded.size <= max(2, T // 200)


@pytest.mark.parametrize("T,d,E,G,Gk,K", [(100, 16384, 64, 8, 4, 8),   # 32 slices per CTA: the ring wraps 4 times
                                           (1, 5120, 256, 8, 4, 8),     # one token: 63 rows of the tile read as zero
                                           (1024, 256, 48, 6, 3, 4)])   # tensor-core router, clusters of 2 (E_pad 48)
def test_route_edges(T, d, E, G, Gk, K):
    """Router shapes at the edges of the two kernels: the widest hidden dimension (d = 16384) on
    the SIMT router, a single token (a nearly empty tile and one selecting warp), and the
    tensor-core router with an expert count whose padded rows split into halves (clusters of 2)
    at the smallest tensor-core batch."""
    cfg = W.MoEConfig("edge", T=T, d=d, E=E, n_groups=G, topk_groups=Gk, top_k=K, inter=64)
    x_h, wr_h = W.gen_x(cfg, 70 + T), W.gen_wr(cfg, 70 + T)
    gi, gw = route_only(cfg, x_h, wr_h)
    excluded, _, _ = compare_routing(cfg, gi, gw, O.route(cfg, x_h, wr_h), label=f"router edge T={T} d={d} E={E}")
    assert excluded.size <= max(2, T // 200)


def test_route_simt_repeated_calls_reuse_tickets():
    """The fused selection counts finished CTAs in the workspace header and returns the counts to
    zero: many calls on one workspace, with different batch sizes, route like the oracle."""
    cfg = W.CONFIGS["decode"]
    dims_max = bm.Dims.from_config(cfg.with_tokens(200))
    ws = bm.allocate_workspace(dims_max)
    wr_h = W.gen_wr(cfg, 61)
    w_r = dev(wr_h)
    for i, T in enumerate([64, 200, 1, 64, 130, 200, 7]):
        c = cfg.with_tokens(T)
        x_h = W.gen_x(c, 61 + i)
        dims = bm.Dims.from_config(c)
        idx = torch.empty((T, c.top_k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, c.top_k), dtype=torch.float32, device="cuda")
        bm.moe_route(dims, dev(x_h), w_r, idx, w, ws)
        torch.cuda.synchronize()
        assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
        compare_routing(c, idx.cpu().numpy(), w.cpu().numpy(), O.route(c, x_h, wr_h), label=f"repeated call {i} T={T}")
    assert int(ws[:1024].view(torch.int32)[13:13 + 192].abs().sum().item()) == 0


# ---------------------------------------------------------------------------------------- permute

@pytest.mark.parametrize("T,E,K,hot", [(64, 16, 4, 0), (77, 16, 4, 3), (1, 256, 8, 0), (4096, 256, 8, 0),
                                       (3000, 256, 8, 16), (33, 32, 32, 0)])
def test_permute_parity(T, E, K, hot):
    d = 128
    idx_h = W.random_topk(11, T, E, K, hot_count=hot, hot_prob=0.5 if hot else 0.0)
    x_h = W.normal_bf16(11, W.TID_X, 0, T * d, 1.0).reshape(T, d)
    dims = bm.Dims(T, d, E, 1, 1, K, 64)
    ws = bm.allocate_workspace(dims)
    R = T * K
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    row_token = torch.empty(R, dtype=torch.int32, device="cuda")
    inv_row = torch.empty(R, dtype=torch.int32, device="cuda")
    x_perm = torch.empty((R, d), dtype=torch.bfloat16, device="cuda")
    bm.moe_permute(dims, dev(x_h), dev(idx_h), counts, offsets, row_token, inv_row, x_perm, ws)
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    c, o, rt, ir = O.permute(idx_h, E)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(row_token.cpu().numpy(), rt)
    assert np.array_equal(inv_row.cpu().numpy(), ir)
    assert np.array_equal(host_bits(x_perm), x_h[rt])


def test_permute_bad_expert_latched():
    """An out-of-range expert id is dropped and latched, never faults."""
    T, E, K, d = 40, 16, 4, 64
    idx_h = W.random_topk(12, T, E, K)
    idx_h[5, 2] = E + 3
    idx_h[9, 0] = -1
    x_h = W.normal_bf16(12, W.TID_X, 0, T * d, 1.0).reshape(T, d)
    dims = bm.Dims(T, d, E, 1, 1, K, 64)
    ws = bm.allocate_workspace(dims)
    R = T * K
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    row_token = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    inv_row = torch.empty(R, dtype=torch.int32, device="cuda")
    x_perm = torch.zeros((R, d), dtype=torch.bfloat16, device="cuda")
    bm.moe_permute(dims, dev(x_h), dev(idx_h), counts, offsets, row_token, inv_row, x_perm, ws)
    assert bm.moe_get_device_status(ws, clear=True) == bm.MOE_DEV_BAD_EXPERT
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    ir = inv_row.cpu().numpy().reshape(T, K)
    assert ir[5, 2] == -1 and ir[9, 0] == -1
    assert counts.cpu().numpy().sum() == R - 2
    assert offsets.cpu().numpy()[-1] == R - 2


def test_permute_duplicate_expert_latched():
    """A token that names one expert in two slots latches MOE_DEV_DUP_EXPERT; both slots share
    one row, the counts take the token once, and every other row is still exact."""
    T, E, K, d = 40, 16, 4, 64
    idx_h = W.random_topk(13, T, E, K)
    idx_h[7, 3] = idx_h[7, 1]
    x_h = W.normal_bf16(13, W.TID_X, 0, T * d, 1.0).reshape(T, d)
    dims = bm.Dims(T, d, E, 1, 1, K, 64)
    ws = bm.allocate_workspace(dims)
    R = T * K
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    row_token = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    inv_row = torch.empty(R, dtype=torch.int32, device="cuda")
    x_perm = torch.zeros((R, d), dtype=torch.bfloat16, device="cuda")
    bm.moe_permute(dims, dev(x_h), dev(idx_h), counts, offsets, row_token, inv_row, x_perm, ws)
    assert bm.moe_get_device_status(ws, clear=True) == bm.MOE_DEV_DUP_EXPERT
    ir = inv_row.cpu().numpy().reshape(T, K)
    assert ir[7, 1] == ir[7, 3] >= 0
    assert offsets.cpu().numpy()[-1] == R - 1
    # the routing with the repeat removed (slot 3 of token 7 dropped) gives the same rows
    c = np.bincount(np.delete(idx_h.ravel(), 7 * K + 3), minlength=E)
    assert np.array_equal(counts.cpu().numpy(), c)
    pairs = sorted({(int(e), t) for t in range(T) for e in idx_h[t]})  # rows ordered by (expert, token)
    rt = np.array([t for _, t in pairs], np.int32)
    assert np.array_equal(row_token.cpu().numpy()[:R - 1], rt)
    assert np.array_equal(host_bits(x_perm)[:R - 1], x_h[rt])


# ---------------------------------------------------------------------------------------- experts

def _ffn_case(d, inter, E, T, K, counts_list, seed, wfmt="bf16"):
    R = T * K
    counts_h = np.array(counts_list, np.int64)
    assert counts_h.size == E and counts_h.sum() <= R
    offsets_h = np.concatenate([[0], np.cumsum(counts_h)]).astype(np.int32)
    cfg = W.MoEConfig("ffn", T=T, d=d, E=E, n_groups=1, topk_groups=1, top_k=K, inter=inter, wfmt=wfmt)
    dw = DeviceWeights(cfg, seed)
    x_perm_h = W.normal_bf16(seed, W.TID_X, 0, R * d, 1.0).reshape(R, d)
    dims = bm.Dims.from_config(cfg)
    ws = bm.allocate_workspace(dims)
    y = torch.full((R, d), float("nan"), dtype=torch.float32, device="cuda")
    bm.moe_expert_ffn(dims, dev(x_perm_h), dev(offsets_h), dw.dev, y, ws)
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    n = int(offsets_h[-1])
    row_expert = np.repeat(np.arange(E, dtype=np.int32), counts_h)
    ref = O.ffn_rows(row_expert, x_perm_h[:n], dw.host, d, inter, wfmt)
    got = y[:n].float().cpu().numpy().astype(np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    report(f"expert ffn d={d} inter={inter} E={E} {wfmt}", f"{err.size} elements: max|err|/RMS = "
           f"{err.max() / rms:.3e} (bar {TOL[wfmt]:g}), RMS(err)/RMS = {np.sqrt(np.mean(err ** 2)) / rms:.3e}")
    assert err.max() <= TOL[wfmt] * rms, (err.max(), rms)
    # the typical error is far below the bar: fp32 accumulation order, 1-ulp flips of the
    # bf16 h and output, and for FP8 the bf16 rounding of the dequantised weights
    assert np.sqrt(np.mean(err ** 2)) <= RMS_BAR[wfmt] * rms
    return got, ref


def test_expert_ffn_tiles_and_ragged_tails():
    """Empty expert, one row, 17, exactly 256 (one full tile), 257, 600 (three tiles), 33;
    three 128-row weight tiles in GEMM1 and two in GEMM2."""
    _ffn_case(d=256, inter=384, E=8, T=710, K=2, counts_list=[0, 1, 17, 256, 257, 255, 600, 33], seed=21)


def test_expert_ffn_intermediate_below_tile():
    """inter = 64 < 128: the weight tile spans two experts; rows past inter are masked."""
    _ffn_case(d=128, inter=64, E=16, T=64, K=4, counts_list=[16] * 16, seed=22)


def test_expert_ffn_beam_shape_few_rows():
    """d=5120, inter=2560: the full 80-step K loop, 20 + 40 weight tiles per expert."""
    _ffn_case(d=5120, inter=2560, E=4, T=16, K=2, counts_list=[3, 1, 0, 12], seed=23)


def test_expert_ffn_nvfp4_tiles_and_ragged_tails():
    """NVFP4 weights decoded on chip: same tile/ragged coverage as the bf16 case."""
    _ffn_case(d=256, inter=256, E=8, T=710, K=2, counts_list=[0, 1, 17, 256, 257, 255, 600, 33], seed=24,
              wfmt="nvfp4")


def test_expert_ffn_nvfp4_beam_shape_few_rows():
    _ffn_case(d=5120, inter=2560, E=4, T=16, K=2, counts_list=[3, 1, 0, 12], seed=25, wfmt="nvfp4")


def test_expert_ffn_fp8_tiles_and_ragged_tails():
    """FP8 weights decoded on chip; d = 384 leaves the last 256-row down tile half past the
    expert (its rows take scale 0 and are dropped), inter = 384 gives three GEMM1 tiles."""
    _ffn_case(d=384, inter=384, E=8, T=710, K=2, counts_list=[0, 1, 17, 256, 257, 255, 600, 33], seed=26,
              wfmt="fp8")


def test_expert_ffn_fp8_beam_shape_few_rows():
    """d=5120, inter=2560: 40 and 20 scale blocks along K, every block scale distinct."""
    _ffn_case(d=5120, inter=2560, E=4, T=16, K=2, counts_list=[3, 1, 0, 12], seed=27, wfmt="fp8")


def test_fp8_needs_multiples_of_128():
    E, d, inter = 4, 192, 128
    dims = bm.Dims(16, d, E, 1, 1, 2, inter, 1.0, bm.MOE_W_FP8)
    w = bm.ExpertWeights(
        torch.zeros((E, inter, d), dtype=torch.uint8, device="cuda"),
        torch.zeros((E, inter, d), dtype=torch.uint8, device="cuda"),
        torch.zeros((E, d, inter), dtype=torch.uint8, device="cuda"),
        gate_sf=torch.ones((E, inter // 128, d // 128), dtype=torch.float32, device="cuda"),
        up_sf=torch.ones((E, inter // 128, d // 128), dtype=torch.float32, device="cuda"),
        down_sf=torch.ones((E, d // 128, inter // 128), dtype=torch.float32, device="cuda"))
    ws = bm.allocate_workspace(dims)
    x = torch.zeros((16, d), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((d, E), dtype=torch.float32, device="cuda")
    out = torch.empty((16, d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bm.MoEError, match="UNSUPPORTED"):
        bm.moe_forward(dims, x, wr, w, out, ws)
    torch.cuda.synchronize()


def test_nvfp4_needs_multiples_of_256():
    cfg = W.MoEConfig("q", T=16, d=128, E=4, n_groups=1, topk_groups=1, top_k=2, inter=64, wfmt="nvfp4")
    dw = DeviceWeights(cfg, 1, keep_host=False)
    dims = bm.Dims.from_config(cfg)
    ws = bm.allocate_workspace(dims)
    x = torch.zeros((16, 128), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((128, 4), dtype=torch.float32, device="cuda")
    out = torch.empty((16, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bm.MoEError, match="UNSUPPORTED"):
        bm.moe_forward(dims, x, wr, dw.dev, out, ws)
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------------------- combine

@pytest.mark.parametrize("T,K,d", [(64, 4, 128), (33, 8, 5120), (1, 1, 64), (7, 20, 192)])
def test_combine_parity(T, K, d):
    E = max(K, 16)
    idx_h = W.random_topk(31, T, E, K)
    _, _, _, inv_row_h = O.permute(idx_h, E)
    y_h = W.normal_f32(31, W.TID_AUX, 0, T * K * d, 1.0).reshape(T * K, d)
    w_h = (2.5 * W.uniform_f64(31, W.TID_AUX + 1, 0, T * K)).astype(np.float32).reshape(T, K)
    dims = bm.Dims(T, d, E, 1, 1, K, 64)
    out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    bm.moe_combine(dims, dev(y_h), dev(inv_row_h), dev(w_h), out)
    torch.cuda.synchronize()
    ref = O.combine(y_h, inv_row_h, w_h.astype(np.float64))
    got = bf16_to_f64(host_bits(out))
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * np.sqrt(np.mean(ref ** 2)))


# ---------------------------------------------------------------------------------------- block

@pytest.mark.parametrize("T,seed", [(64, 0), (77, 5), (1, 6), (256, 7)])
def test_forward_tiny_full_parity(T, seed):
    cfg = TINY.with_tokens(T)
    inp = W.make_host_inputs(cfg, seed)
    dw = DeviceWeights(cfg, seed)
    out, idx, counts, _ = run_forward(cfg, dev(inp["x"]), dev(inp["w_r"]), dw.dev)
    orc = O.route(cfg, inp["x"], inp["w_r"])
    gi = idx.cpu().numpy()
    # the forward pass keeps its weights in the workspace; moe_route tests check them
    excluded, ref_idx, ref_w = compare_routing_idx_only(cfg, gi, orc)
    assert np.array_equal(counts.cpu().numpy(), np.bincount(gi.ravel(), minlength=cfg.E))
    ref = O.forward_tokens(cfg, inp["x"], ref_idx, ref_w, np.arange(T), dw.host)
    check_output(host_bits(out), ref, TOL_BF16)


def compare_routing_idx_only(cfg, gi, orc):
    """compare_routing with the oracle's own weights standing in for the GPU's (the
    forward pass keeps its weights in the workspace; moe_route tests check them)."""
    w_like = np.zeros(gi.shape, np.float32)
    s = orc["scores"].astype(np.float64)
    sv = np.take_along_axis(s, gi.astype(np.int64), 1)
    w_like[:] = cfg.routed_scale * sv / sv.sum(1, keepdims=True)
    return compare_routing(cfg, gi, w_like, orc)


SMALL_NVFP4 = W.MoEConfig("small_nvfp4", T=64, d=256, E=16, n_groups=4, topk_groups=2, top_k=4, inter=256,
                          wfmt="nvfp4")


@pytest.mark.parametrize("wfmt", ["nvfp4", "fp8"])
@pytest.mark.parametrize("T,seed", [(64, 0), (100, 4)])
def test_forward_quantised_full_parity(T, seed, wfmt):
    cfg = dataclasses.replace(SMALL_NVFP4.with_tokens(T), wfmt=wfmt)
    x_h, wr_h = W.gen_x(cfg, seed), W.gen_wr(cfg, seed)
    dw = DeviceWeights(cfg, seed)
    out, idx, counts, _ = run_forward(cfg, dev(x_h), dev(wr_h), dw.dev)
    orc = O.route(cfg, x_h, wr_h)
    excluded, ref_idx, ref_w = compare_routing_idx_only(cfg, idx.cpu().numpy(), orc)
    ref = O.forward_tokens(cfg, x_h, ref_idx, ref_w, np.arange(T), dw.host)
    check_output(host_bits(out), ref, TOL[wfmt], label=f"forward 16 experts T={T} {wfmt}")


# E = 40 (not a multiple of 16: padded to 48 on the tensor-core router), groups of 8 (the generic
# group-score path), top-6 of 2 kept groups, intermediate 192 (a ragged 64-row second weight tile)
ODD = W.MoEConfig("odd", T=1200, d=256, E=40, n_groups=5, topk_groups=2, top_k=6, inter=192)


def test_forward_odd_shape_tensor_core_router():
    """T = 1200 >= 1024 takes the tensor-core router (hidden split in 8 for the fp32 recompute)."""
    cfg = ODD
    x_h, wr_h = W.gen_x(cfg, 3), W.gen_wr(cfg, 3)
    gi_route, gw_route = route_only(cfg, x_h, wr_h)
    orc = O.route(cfg, x_h, wr_h)
    compare_routing(cfg, gi_route, gw_route, orc)
    dw = DeviceWeights(cfg, 3)
    out, idx, counts, _ = run_forward(cfg, dev(x_h), dev(wr_h), dw.dev)
    gi = idx.cpu().numpy()
    excluded, ref_idx, ref_w = compare_routing_idx_only(cfg, gi, orc)
    assert np.array_equal(counts.cpu().numpy(), np.bincount(gi.ravel(), minlength=cfg.E))
    rows = np.arange(0, cfg.T, 7)
    ref = O.forward_tokens(cfg, x_h, ref_idx, ref_w, rows, dw.host)
    check_output(host_bits(out)[rows], ref, TOL_BF16)


def test_forward_deterministic():
    cfg = TINY.with_tokens(200)
    inp = W.make_host_inputs(cfg, 9)
    dw = DeviceWeights(cfg, 9, keep_host=False)
    a, _, _, _ = run_forward(cfg, dev(inp["x"]), dev(inp["w_r"]), dw.dev)
    b, _, _, _ = run_forward(cfg, dev(inp["x"]), dev(inp["w_r"]), dw.dev)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_forward_empty_batch_is_noop():
    cfg = TINY
    dims = bm.Dims.from_config(cfg, 0)
    dw = DeviceWeights(cfg, 0, keep_host=False)
    ws = bm.allocate_workspace(bm.Dims.from_config(cfg, 1))
    out = torch.empty((0, cfg.d), dtype=torch.bfloat16, device="cuda")
    x = torch.empty((0, cfg.d), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((cfg.d, cfg.E), dtype=torch.float32, device="cuda")
    bm.moe_forward(dims, x, wr, dw.dev, out, ws)
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------------------- full size

@pytest.fixture(scope="module")
def beam_weights():
    """The Beam-shape layer (256 experts, d=5120, inter=2560, ~20 GB bf16), shared by the
    decode, prefill and skewed workloads."""
    dw = DeviceWeights(W.CONFIGS["decode"], 0)
    yield dw
    del dw
    torch.cuda.empty_cache()


def _sample_tokens(T, gi, n=48, seed=0):
    rng = np.random.default_rng(seed)
    picks = set(rng.choice(T, size=min(n, T), replace=False).tolist()) | {0, T - 1}
    counts = np.bincount(gi.ravel(), minlength=256)
    hot = int(np.argmax(counts))
    hot_tokens = np.nonzero((gi == hot).any(1))[0]
    picks |= set(hot_tokens[:4].tolist()) | set(hot_tokens[-4:].tolist())
    return np.array(sorted(picks), np.int32)


def _full_size_parity(cfg, dw, label):
    """One full-size batch in the launch configuration the benchmark times (moe_forward on the
    whole batch), and the same batch through the four staged calls, which run the same kernels
    with the same plan; the two outputs must agree bit for bit. Then, against the oracle:
    routing on every token (weights included), the permutation bit-exact, the expert output
    of at least one row in every work item of the expert GEMMs (every expert, weight tile and
    token tile of this launch), and the block output on sampled tokens."""
    tol = TOL[cfg.wfmt]
    x_h, wr_h = W.gen_x(cfg, 0), W.gen_wr(cfg, 0)
    x, w_r = dev(x_h), dev(wr_h)
    out, idx_f, counts_f, ws = run_forward(cfg, x, w_r, dw.dev)
    T, K, E, d = cfg.T, cfg.top_k, cfg.E, cfg.d
    R = T * K
    dims = bm.Dims.from_config(cfg)
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    row_token = torch.empty(R, dtype=torch.int32, device="cuda")
    inv_row = torch.empty(R, dtype=torch.int32, device="cuda")
    x_perm = torch.empty((R, d), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((R, d), dtype=torch.float32, device="cuda")
    out_s = torch.empty_like(out)
    bm.moe_route(dims, x, w_r, idx, w, ws)
    bm.moe_permute(dims, x, idx, counts, offsets, row_token, inv_row, x_perm, ws)
    bm.moe_expert_ffn(dims, x_perm, offsets, dw.dev, y, ws)
    bm.moe_combine(dims, y, inv_row, w, out_s, ws)
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    assert torch.equal(idx, idx_f) and torch.equal(counts, counts_f)
    assert torch.equal(out_s.view(torch.int16), out.view(torch.int16))

    gi, gw = idx.cpu().numpy(), w.cpu().numpy()
    orc = O.route(cfg, x_h, wr_h)
    excluded, ref_idx, ref_w = compare_routing(cfg, gi, gw, orc, label=label)
    assert excluded.size <= max(2, T // 200)
    c, o, rt, ir = O.permute(ref_idx, E)
    assert np.array_equal(counts.cpu().numpy(), c) and np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(row_token.cpu().numpy(), rt)
    # inv_row follows each token's slot order, which may differ from the oracle's where two chosen
    # experts score within a rounding of each other (both orders are valid): compare each token's
    # set of rows, and check every slot's row belongs to the slot's expert
    gir = inv_row.cpu().numpy().reshape(T, K)
    assert np.array_equal(np.sort(gir, 1), np.sort(ir.reshape(T, K), 1))
    row_expert = np.repeat(np.arange(E, dtype=np.int32), c)
    assert np.array_equal(row_expert[gir], gi)
    rt_dev = torch.from_numpy(rt.astype(np.int64)).cuda()
    assert torch.equal(x_perm.view(torch.int16), x.view(torch.int16)[rt_dev])
    del rt_dev

    n_max = plan_n_max(T, E, K, cfg.wfmt != "bf16")
    rows, n_tiles = work_item_rows(c, n_max, np.random.default_rng(1))
    row_e = np.repeat(np.arange(E, dtype=np.int32), c)[rows]
    ref_y = O.ffn_rows(row_e, x_h[rt[rows]], dw.host, d, cfg.inter, cfg.wfmt)
    got_y = y[torch.from_numpy(rows).cuda()].cpu().numpy()
    check_output(got_y, ref_y, tol, rms_bar=RMS_BAR[cfg.wfmt],
                 label=f"{label} expert rows ({rows.size} rows covering all {n_tiles} token tiles, n_max {n_max})")
    toks = np.arange(T, dtype=np.int32) if T <= 64 else _sample_tokens(T, gi)
    ref = O.forward_tokens(cfg, x_h, ref_idx, ref_w, toks, dw.host)
    check_output(host_bits(out)[toks], ref, tol, label=f"{label} block output ({toks.size} tokens)")
    return c


@pytest.mark.slow
@pytest.mark.parametrize("wfmt", ["nvfp4", "fp8"])
def test_forward_full_size_quantised(wfmt):
    """The NVFP4 and FP8 prefill workloads (T=4096, Beam shape, weights quantised from the same
    seeded bf16)."""
    cfg = W.CONFIGS[wfmt]
    dw = DeviceWeights(cfg, 0)
    _full_size_parity(cfg, dw, f"{wfmt} T={cfg.T}")
    del dw
    torch.cuda.empty_cache()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode", "prefill", "skewed"])
def test_forward_full_size(name, beam_weights):
    cfg = W.CONFIGS[name]
    c = _full_size_parity(cfg, beam_weights, f"{name} T={cfg.T}")
    if cfg.skew:
        ratio = c[list(cfg.hot_experts)].mean() / (cfg.T * cfg.top_k / cfg.E)
        assert 3.5 < ratio < 4.5


@pytest.mark.slow
@pytest.mark.parametrize("name,seed", [("prefill", 1), ("prefill", 2), ("prefill", 3), ("prefill", 4),
                                       ("skewed", 5)])
def test_route_stress_32k(name, seed):
    """Routing of 32,768 tokens on both router paths against the oracle: the tensor-core router
    on the whole batch, and the FP32 SIMT router on the same tokens in batches of 1,000 (below
    the tensor-core threshold)."""
    cfg = W.CONFIGS[name].with_tokens(32768)
    x_h, wr_h = W.gen_x(cfg, seed), W.gen_wr(cfg, seed)
    orc = O.route(cfg, x_h, wr_h)
    gi, gw = route_only(cfg, x_h, wr_h)
    ex, _, _ = compare_routing(cfg, gi, gw, orc, label=f"{name} T=32768 seed {seed}, tensor-core router")
    assert ex.size <= cfg.T // 200
    parts = [route_only(cfg, np.ascontiguousarray(x_h[a:a + 1000]), wr_h) for a in range(0, cfg.T, 1000)]
    gi2, gw2 = np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])
    compare_routing(cfg, gi2, gw2, orc, label=f"{name} T=32768 seed {seed}, SIMT router in batches of 1000")


# ---------------------------------------------------------------------------------------- residual

@pytest.mark.parametrize("T,K,d,step", [(33, 8, 5120, 2), (64, 4, 128, 1), (5, 8, 5120, 37), (1, 20, 192, 3)])
def test_combine_residual_parity(T, K, d, step):
    """Combine + RMSNorm post-norm + depth-scaled residual update (release article, section
    "Residual stream"), against the oracle's exact combine and residual update."""
    E = max(K, 16)
    idx_h = W.random_topk(41, T, E, K)
    _, _, _, inv_row_h = O.permute(idx_h, E)
    y_h = W.normal_f32(41, W.TID_AUX, 0, T * K * d, 1.0).reshape(T * K, d)
    w_h = (2.5 * W.uniform_f64(41, W.TID_AUX + 1, 0, T * K)).astype(np.float32).reshape(T, K)
    gain_h = W.normal_bf16(41, W.TID_AUX + 2, 0, d, 0.1)
    gain_h = (W.bf16_to_f32(gain_h) + 1.0).astype(np.float32)
    gain_bits = torch.from_numpy(gain_h).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    h_old = W.normal_bf16(41, W.TID_AUX + 3, 0, T * d, 1.0).reshape(T, d)
    dims = bm.Dims(T, d, E, 1, 1, K, 64)
    resid = dev(h_old)
    bm.moe_combine_residual(dims, dev(y_h), dev(inv_row_h), dev(w_h), dev(gain_bits), 1e-6, step, resid)
    torch.cuda.synchronize()
    out = O.combine(y_h, inv_row_h, w_h.astype(np.float64))
    ref = O.residual_update(out, h_old, gain_bits, 1e-6, step)
    check_output(host_bits(resid), ref, TOL_BF16)
    # the only roundings: FP32 combine and norm, and the bf16 result (<= 2^-9 relative)
    err = np.abs(bf16_to_f64(host_bits(resid)) - ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-5 * np.sqrt(np.mean(ref ** 2)))


def test_forward_residual_parity():
    cfg = TINY.with_tokens(80)
    inp = W.make_host_inputs(cfg, 27)
    dw = DeviceWeights(cfg, 27)
    dims = bm.Dims.from_config(cfg)
    ws = bm.allocate_workspace(dims)
    h_old = W.normal_bf16(27, W.TID_AUX + 3, 0, cfg.T * cfg.d, 1.0).reshape(cfg.T, cfg.d)
    gain_bits = W.normal_bf16(27, W.TID_AUX + 2, 0, cfg.d, 0.05)
    gain_bits = torch.from_numpy(W.bf16_to_f32(gain_bits) + 1.0).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    resid = dev(h_old)
    idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    bm.moe_forward_residual(dims, dev(inp["x"]), dev(inp["w_r"]), dw.dev, dev(gain_bits), 1e-6, 7, resid, ws,
                            topk_idx=idx)
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    orc = O.route(cfg, inp["x"], inp["w_r"])
    _, ref_idx, ref_w = compare_routing_idx_only(cfg, idx.cpu().numpy(), orc)
    out = O.forward_tokens(cfg, inp["x"], ref_idx, ref_w, np.arange(cfg.T), dw.host)
    ref = O.residual_update(out, h_old, gain_bits, 1e-6, 7)
    check_output(host_bits(resid), ref, TOL_BF16)


@pytest.mark.parametrize("T,d", [(7, 64), (300, 5120), (1, 16384)])
def test_pre_norm_parity(T, d):
    """Pre-norm of the sublayer input (release article, section "Residual stream"): the FP32
    kernel against the oracle's exact value rounded to FP32 and then bf16. Reduction order can
    move an element across a bf16 rounding boundary, so a few elements may differ by one ulp."""
    h = W.normal_bf16(61, W.TID_AUX, 0, T * d, 2.0).reshape(T, d)
    gain = W.normal_bf16(61, W.TID_AUX + 1, 0, d, 0.1)
    gain = torch.from_numpy(W.bf16_to_f32(gain) + 1.0).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    x = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    bm.moe_pre_norm(bm.Dims(T, d, 1, 1, 1, 1, 64), dev(h), dev(gain), 1e-6, x)
    torch.cuda.synchronize()
    got = host_bits(x).astype(np.int32)
    ref = O.pre_norm(h, gain, 1e-6).astype(np.int32)
    diff = np.abs(got - ref)  # same-sign bf16 patterns: one ulp = 1
    assert diff.max() <= 1
    assert np.count_nonzero(diff) <= max(2, diff.size // 1000)


def test_sublayer_parity():
    """Pre-norm, block forward and post-norm residual update in one call, against the oracle's
    pre_norm -> route -> forward_tokens -> residual_update on the x the kernel produced."""
    cfg = TINY.with_tokens(80)
    inp = W.make_host_inputs(cfg, 29)
    dw = DeviceWeights(cfg, 29)
    dims = bm.Dims.from_config(cfg)
    ws = bm.allocate_workspace(dims)
    h_old = W.normal_bf16(29, W.TID_AUX + 3, 0, cfg.T * cfg.d, 1.0).reshape(cfg.T, cfg.d)

    def gain(tid):
        g = W.normal_bf16(29, tid, 0, cfg.d, 0.05)
        return torch.from_numpy(W.bf16_to_f32(g) + 1.0).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    pre, post = gain(W.TID_AUX + 4), gain(W.TID_AUX + 5)
    resid = dev(h_old)
    x = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    bm.moe_sublayer(dims, resid, dev(pre), dev(post), 1e-6, 5, dev(inp["w_r"]), dw.dev, x, ws, topk_idx=idx)
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    x_h = host_bits(x)
    ref_x = O.pre_norm(h_old, pre, 1e-6)
    assert np.abs(x_h.astype(np.int32) - ref_x.astype(np.int32)).max() <= 1
    orc = O.route(cfg, x_h, inp["w_r"])
    _, ref_idx, ref_w = compare_routing_idx_only(cfg, idx.cpu().numpy(), orc)
    out = O.forward_tokens(cfg, x_h, ref_idx, ref_w, np.arange(cfg.T), dw.host)
    ref = O.residual_update(out, h_old, post, 1e-6, 5)
    check_output(host_bits(resid), ref, TOL_BF16)


def test_sublayer_fp8_selection_bias():
    """Every optional piece at once: FP8 expert weights, a selection bias, the pre-norm and the
    post-norm residual update, on a 16-expert block with 4 groups (T = 100, ragged tiles)."""
    cfg = dataclasses.replace(SMALL_NVFP4.with_tokens(100), wfmt="fp8")
    seed = 33
    wr_h = W.gen_wr(cfg, seed)
    bias = (0.2 * (W.uniform_f64(seed, W.TID_AUX + 7, 0, cfg.E) - 0.5)).astype(np.float32)
    dw = DeviceWeights(cfg, seed)
    dims = bm.Dims.from_config(cfg)
    ws = bm.allocate_workspace(dims)
    h_old = W.normal_bf16(seed, W.TID_AUX + 3, 0, cfg.T * cfg.d, 1.0).reshape(cfg.T, cfg.d)

    def gain(tid):
        g = W.normal_bf16(seed, tid, 0, cfg.d, 0.05)
        return torch.from_numpy(W.bf16_to_f32(g) + 1.0).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    pre, post = gain(W.TID_AUX + 4), gain(W.TID_AUX + 5)
    resid = dev(h_old)
    x = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    bm.moe_sublayer(dims, resid, dev(pre), dev(post), 1e-6, 3, dev(wr_h), dw.dev, x, ws, topk_idx=idx,
                    sel_bias=dev(bias))
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    x_h = host_bits(x)
    assert np.abs(x_h.astype(np.int32) - O.pre_norm(h_old, pre, 1e-6).astype(np.int32)).max() <= 1
    orc = O.route(cfg, x_h, wr_h, bias=bias)
    gi = idx.cpu().numpy()
    sv = np.take_along_axis(orc["scores"].astype(np.float64), gi.astype(np.int64), 1)
    w_like = (cfg.routed_scale * sv / sv.sum(1, keepdims=True)).astype(np.float32)
    _, ref_idx, ref_w = compare_routing(cfg, gi, w_like, orc, bias=bias)
    out = O.forward_tokens(cfg, x_h, ref_idx, ref_w, np.arange(cfg.T), dw.host)
    ref = O.residual_update(out, h_old, post, 1e-6, 3)
    check_output(host_bits(resid), ref, TOL_FP8)


@pytest.mark.parametrize("wfmt", ["bf16", "nvfp4", "fp8"])
def test_forward_single_token(wfmt):
    """T = 1: one token, 4 experts of 16 touched, one 16-row token tile per expert."""
    cfg = dataclasses.replace(SMALL_NVFP4.with_tokens(1), wfmt=wfmt)
    x_h, wr_h = W.gen_x(cfg, 35), W.gen_wr(cfg, 35)
    dw = DeviceWeights(cfg, 35)
    out, idx, counts, _ = run_forward(cfg, dev(x_h), dev(wr_h), dw.dev)
    orc = O.route(cfg, x_h, wr_h)
    _, ref_idx, ref_w = compare_routing_idx_only(cfg, idx.cpu().numpy(), orc)
    assert counts.cpu().numpy().sum() == cfg.top_k
    ref = O.forward_tokens(cfg, x_h, ref_idx, ref_w, np.arange(1), dw.host)
    check_output(host_bits(out), ref, TOL[wfmt])
