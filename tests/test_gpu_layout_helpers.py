"""GPU checks of the offline layout helpers (README "Bridge Layer":
assemble_scales_2d_side / _3d_side, interleave_l1_weights /
deinterleave_l1_weights), through the C ABI:

* nvfp4_sf_to_tiled writes every byte of both tiled layouts as the index maps
  written from the header's layout formulas (tests/helpers.py) place them,
  padding 0; nvfp4_sf_from_tiled gives the row-major bytes back;
* nvfp4_interleave_gate_up moves codes and scales the way the oracle's
  interleave does, its inverse undoes it, and quantize -> interleave -> tile
  gives the very bytes of the weight preparation the forward uses.
"""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import sf_rows_index, sf_tiled_index
from nvfp4_block_scaled_05_gb300 import binding as B
from nvfp4_block_scaled_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _tiled_ref(sf_rm, rows, cols, layout):
    """Tiled bytes of row-major scales (batch, rows, cols//16), padding 0."""
    per = B.nvfp4_sf_bytes(rows, cols, layout)
    idx = sf_tiled_index(rows, cols) if layout == B.NVFP4_SF_TILED else sf_rows_index(rows, cols)
    out = np.zeros((sf_rm.shape[0], per), np.uint8)
    for m in range(sf_rm.shape[0]):
        out[m][idx.reshape(-1)] = sf_rm[m].reshape(-1)
    return out.reshape(-1)


@pytest.mark.parametrize("layout", [B.NVFP4_SF_TILED, B.NVFP4_SF_TILED_ROWS])
@pytest.mark.parametrize("batch,rows,cols", [(1, 128, 64), (3, 300, 7168), (2, 4096, 2048), (1, 1, 16),
                                             (5, 129, 272)])
def test_sf_tiled_round_trip(layout, batch, rows, cols):
    rng = np.random.default_rng(rows + cols + layout)
    sf = rng.integers(1, 127, (batch, rows, cols // 16)).astype(np.uint8)
    t = B.nvfp4_sf_to_tiled(torch.from_numpy(sf).to(DEV), rows, cols, layout)
    back = B.nvfp4_sf_from_tiled(t, batch, rows, cols, layout)
    torch.cuda.synchronize()
    assert np.array_equal(t.cpu().numpy(), _tiled_ref(sf, rows, cols, layout))
    assert np.array_equal(back.cpu().numpy(), sf)


@pytest.mark.parametrize("K", [448, 48])
@pytest.mark.parametrize("layout", [B.NVFP4_SF_ROWMAJOR, B.NVFP4_SF_TILED, B.NVFP4_SF_TILED_ROWS])
def test_interleave_gate_up_matches_oracle(layout, K):
    """K=448: 16-byte code copies; K=48: 24-byte rows, copied byte by byte."""
    rng = np.random.default_rng(layout + K)
    batch, two_i = 3, 4096 + 16 * 3
    codes = rng.integers(0, 256, (batch, two_i, K // 2)).astype(np.uint8)
    sf_rm = rng.integers(1, 127, (batch, two_i, K // 16)).astype(np.uint8)
    sf_in = sf_rm.reshape(-1) if layout == B.NVFP4_SF_ROWMAJOR else _tiled_ref(sf_rm, two_i, K, layout)
    co, so = B.nvfp4_interleave_gate_up(torch.from_numpy(codes).to(DEV), torch.from_numpy(sf_in).to(DEV),
                                        two_i, K, layout)
    torch.cuda.synchronize()
    want_c = np.stack([O.interleave_rows(codes[m], 8) for m in range(batch)])
    want_s = np.stack([O.interleave_rows(sf_rm[m], 8) for m in range(batch)])
    assert np.array_equal(co.cpu().numpy(), want_c)
    want_s = want_s.reshape(-1) if layout == B.NVFP4_SF_ROWMAJOR else _tiled_ref(want_s, two_i, K, layout)
    assert np.array_equal(so.cpu().numpy(), want_s)
    ci, si = B.nvfp4_interleave_gate_up(co, so, two_i, K, layout, inverse=True)
    torch.cuda.synchronize()
    assert np.array_equal(ci.cpu().numpy(), codes)
    assert np.array_equal(si.cpu().numpy(), sf_in)


def test_interleave_then_tile_equals_weight_preparation():
    """W1 quantized in [gate | up] order with row-major scales, then
    interleaved and tiled by the helpers, is byte for byte the W1 the forward
    uses (prepare_moe_weights: the quantizer gathers interleaved rows and
    writes tiled scales directly)."""
    cfg = W.CONFIGS["tiny"]
    inp = W.moe_inputs(cfg, seed=3, device=DEV)
    w1 = inp["w1"]
    E, two_i, K = w1.shape
    prep = B.prepare_moe_weights(w1, inp["w2"])
    codes = torch.empty((E, two_i, K // 2), dtype=torch.uint8, device=DEV)
    sf = torch.empty((E, two_i, K // 16), dtype=torch.uint8, device=DEV)
    for e in range(E):
        B.nvfp4_quantize(w1[e], gs=prep["gs_w1"][e:e + 1], codes=codes[e], sf=sf[e], sf_layout=B.NVFP4_SF_ROWMAJOR)
    ci, si = B.nvfp4_interleave_gate_up(codes, sf, two_i, K, B.NVFP4_SF_ROWMAJOR)
    tiled = B.nvfp4_sf_to_tiled(si, two_i, K, B.NVFP4_SF_TILED)
    torch.cuda.synchronize()
    assert torch.equal(ci, prep["w1_codes"])
    per = B.nvfp4_sf_bytes(two_i, K, B.NVFP4_SF_TILED)
    # the quantizer leaves tiled padding unwritten; compare the valid bytes
    idx = torch.from_numpy(sf_tiled_index(two_i, K).reshape(-1)).to(DEV)
    for e in range(E):
        assert torch.equal(tiled[e * per:(e + 1) * per][idx], prep["w1_sf"][e * per:(e + 1) * per][idx])
