"""GPU parity of the dense SwiGLU MLP (the first decoder layers; release article, section
"Architecture") through the C ABI, against the oracle's single-expert SwiGLU rows."""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
import sparse_moe_layer_14_b300 as bm
from support import TOL, DeviceWeights, check_output, dev, host_bits

pytestmark = pytest.mark.gpu


def _dense_cfg(T, d, inter, wfmt="bf16"):
    return W.MoEConfig("dense", T=T, d=d, E=1, n_groups=1, topk_groups=1, top_k=1, inter=inter, wfmt=wfmt)


def _run(cfg, seed, rows=None):
    dw = DeviceWeights(cfg, seed)
    x_h = W.gen_x(cfg, seed)
    dims = bm.Dims.from_config(cfg)
    ws = bm.allocate_dense_workspace(dims)
    out = torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    bm.moe_dense_mlp(dims, dev(x_h), dw.dev, out, ws)
    torch.cuda.synchronize()
    assert bm.moe_get_device_status(ws) == bm.MOE_DEV_OK
    rows = np.arange(cfg.T) if rows is None else rows
    ref = O.ffn_rows(np.zeros(rows.size, np.int32), x_h[rows], dw.host, cfg.d, cfg.inter, cfg.wfmt)
    got = host_bits(out)[rows]
    err, rms = check_output(got, ref, TOL[cfg.wfmt])
    return got, ref


@pytest.mark.parametrize("T,d,inter,seed", [(100, 256, 384, 1),   # three 128-row weight tiles, one token tile
                                            (600, 128, 64, 2),    # inter below one weight tile; three token tiles
                                            (1, 192, 128, 3)])    # a single token
def test_dense_mlp_parity(T, d, inter, seed):
    got, ref = _run(_dense_cfg(T, d, inter), seed)
    # bf16 h and bf16 output are the only roundings beyond accumulation order
    assert np.sqrt(np.mean((W.bf16_to_f32(got).astype(np.float64) - ref) ** 2)) <= 2e-3 * np.sqrt(np.mean(ref ** 2))


@pytest.mark.parametrize("wfmt", ["nvfp4", "fp8"])
def test_dense_mlp_quantised_parity(wfmt):
    _run(_dense_cfg(100, 256, 512, wfmt), 4)


def test_dense_mlp_beam_width_sampled_rows():
    """d = 5120 with a wide intermediate (20480: 160 weight tiles, the full 80-step K loop)."""
    _run(_dense_cfg(64, 5120, 20480), 5, rows=np.array([0, 7, 31, 63]))


def test_dense_mlp_empty_and_unsupported():
    cfg = _dense_cfg(0, 256, 384)
    dw = DeviceWeights(cfg.with_tokens(1), 0, keep_host=False)
    dims = bm.Dims.from_config(cfg)
    ws = bm.allocate_dense_workspace(bm.Dims.from_config(cfg.with_tokens(1)))
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    bm.moe_dense_mlp(dims, x, dw.dev, torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda"), ws)
    # inter = 100 is not a multiple of 64: rejected on the host, nothing launched
    bad = bm.Dims.from_config(_dense_cfg(4, 256, 100))
    z = lambda *shape: torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    w_bad = bm.ExpertWeights(z(1, 100, 256), z(1, 100, 256), z(1, 256, 100))
    with pytest.raises(bm.MoEError, match="UNSUPPORTED"):
        bm.moe_dense_mlp(bad, z(4, 256), w_bad, z(4, 256), ws)
