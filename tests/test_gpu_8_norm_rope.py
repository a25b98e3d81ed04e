"""GPU parity of nvfp4_rmsnorm_rope_quantize (RMS norm -> RoPE -> NVFP4 in one
pass) against the fp64 oracle.

The f32 rows the kernel quantizes (its optional y_out) equal the oracle's fp64
rows within f32 rounding; the codes and scales equal the oracle quantizer
applied to those same f32 rows bit for bit (the quantization decision is taken
in f32 on both sides); against the oracle's own rows rounded to f32 they differ
only where the two f32 roundings land on opposite sides of a code boundary."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import cosine, sf_rows_index, sf_tiled_index
from nvfp4_block_scaled_05_gb300 import binding as B
from nvfp4_block_scaled_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(rows, D, R, P, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = (torch.randn(rows, D, generator=g) * 2.0).to(torch.bfloat16)
    gamma = 1.0 + 0.2 * torch.randn(D, generator=g)
    ang = torch.rand(P, max(R // 2, 1), generator=g) * (2 * np.pi)
    cos_t, sin_t = torch.cos(ang).float(), torch.sin(ang).float()
    pos = torch.randint(0, P, (rows,), generator=g, dtype=torch.int32)
    return x, gamma, cos_t, sin_t, pos


@pytest.mark.parametrize("rows,D,R,layout", [(300, 192, 64, B.NVFP4_SF_TILED), (257, 576, 64, B.NVFP4_SF_ROWMAJOR),
                                             (37, 7168, 0, B.NVFP4_SF_TILED), (1, 64, 64, B.NVFP4_SF_TILED),
                                             (300, 192, 64, B.NVFP4_SF_TILED_ROWS)])
def test_norm_rope_quantize_matches_oracle(rows, D, R, layout):
    P = 4096
    x, gamma, cos_t, sin_t, pos = _inputs(rows, D, R, P, rows + D)
    eps = 1e-6
    yref = O.rmsnorm_rope(W.bf16_bits(x), gamma.double().numpy(), eps, R, pos.numpy(),
                          cos_t.double().numpy(), sin_t.double().numpy())
    gs = O.global_scale(np.float32(np.abs(yref).max()))
    y_out = torch.empty((rows, D), dtype=torch.float32, device=DEV)
    codes, sf = B.nvfp4_rmsnorm_rope_quantize(
        x.to(DEV), gamma.to(DEV), eps, R, pos.to(DEV) if R else None, cos_t.to(DEV) if R else None,
        sin_t.to(DEV) if R else None, torch.tensor([gs], device=DEV), sf_layout=layout, y_out=y_out)
    assert B.nvfp4moe_last_device_status() == 0
    yg = y_out.cpu().numpy()
    scale = np.abs(yref).max()
    # f32 sum of D squares (one lane sums D/32 of them) then rsqrt: relative error of a
    # few 1e-6 at most on the whole row, plus the per-element f32 products
    assert np.all(np.abs(yg - yref) <= 1e-5 * np.abs(yref) + 1e-6 * scale)
    c = codes.cpu().numpy()
    s = sf.cpu().numpy()
    s_rm = (s[sf_tiled_index(rows, D)] if layout == B.NVFP4_SF_TILED
            else s[sf_rows_index(rows, D)] if layout == B.NVFP4_SF_TILED_ROWS
            else s.reshape(rows, D // 16))
    c_own, s_own = O.quantize_f32(yg, gs)
    assert np.array_equal(c, c_own) and np.array_equal(s_rm, s_own)
    c_ref, s_ref = O.quantize_f32(yref.astype(np.float32), gs)
    assert np.mean(c != c_ref) <= 0.01 and np.mean(s_rm != s_ref) <= 0.01
    assert cosine(O.dequantize_f64(c, s_rm, gs), yref) > 0.99


def test_position_out_of_range_zeroes_row_and_reports():
    rows, D, R, P = 64, 192, 64, 100
    x, gamma, cos_t, sin_t, pos = _inputs(rows, D, R, P, 3)
    pos[5] = -1
    pos[9] = P
    gs = torch.tensor([200.0], device=DEV)
    codes, sf = B.nvfp4_rmsnorm_rope_quantize(x.to(DEV), gamma.to(DEV), 1e-6, R, pos.to(DEV), cos_t.to(DEV),
                                              sin_t.to(DEV), gs, sf_layout=B.NVFP4_SF_ROWMAJOR)
    assert B.nvfp4moe_last_device_status() == -1
    c = codes.cpu().numpy()
    s = sf.cpu().numpy().reshape(rows, D // 16)
    assert not c[[5, 9]].any() and not s[[5, 9]].any()
    ok = [r for r in range(rows) if r not in (5, 9)]
    assert c[ok].any()
    assert B.nvfp4moe_last_device_status() == 0
