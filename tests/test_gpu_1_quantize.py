"""GPU parity of the BF16 -> NVFP4 quantizer: bit-exact against the oracle
(codes, scale bytes, global scale), through the C ABI."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import sf_rows_to_rowmajor, sf_tiled_to_rowmajor, padded_rows_of_compact
from nvfp4_block_scaled_05_gb300 import binding as B
from nvfp4_block_scaled_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _quant_check(x, gs_given=None, layout=B.NVFP4_SF_TILED):
    xb = W.bf16_bits(x)
    rows, cols = xb.shape
    gs_ref = O.global_scale(O.amax_bf16(xb)) if gs_given is None else np.float32(gs_given)
    gs_t = None if gs_given is None else torch.tensor([gs_given], dtype=torch.float32, device=DEV)
    codes, sf, gs = B.nvfp4_quantize(x.to(DEV), gs=gs_t, sf_layout=layout)
    torch.cuda.synchronize()
    assert gs.item() == gs_ref
    rc, rs = O.quantize_bf16(xb, gs_ref)
    got_c = codes.cpu().numpy()
    got_s = sf.cpu().numpy()
    got_s = (sf_tiled_to_rowmajor(got_s, rows, cols) if layout == B.NVFP4_SF_TILED
             else sf_rows_to_rowmajor(got_s, rows, cols) if layout == B.NVFP4_SF_TILED_ROWS
             else got_s.reshape(rows, cols // 16))
    assert np.array_equal(got_s, rs), "scale bytes differ at %s" % (np.argwhere(got_s != rs)[:5],)
    bad = np.argwhere(got_c != rc)
    assert bad.size == 0, "codes differ at %s: gpu %s oracle %s" % (
        bad[:5], got_c[tuple(bad[0])], rc[tuple(bad[0])])
    return got_c, got_s


def test_quantize_random_tiled():
    g = torch.Generator().manual_seed(11)
    _quant_check(torch.randn(300, 1024, generator=g).to(torch.bfloat16))


def test_quantize_activation_layout_and_ragged_cols():
    """The GEMMs' activation scale layout (NVFP4_SF_TILED_ROWS), with row and
    column counts that leave partial 128-row and 256-column tiles."""
    g = torch.Generator().manual_seed(14)
    _quant_check(torch.randn(300, 1024, generator=g).to(torch.bfloat16), layout=B.NVFP4_SF_TILED_ROWS)
    _quant_check(torch.randn(129, 592, generator=g).to(torch.bfloat16), layout=B.NVFP4_SF_TILED_ROWS)


def test_quantize_rowmajor_and_ragged_cols():
    g = torch.Generator().manual_seed(12)
    _quant_check(torch.randn(37, 80, generator=g).to(torch.bfloat16), layout=B.NVFP4_SF_ROWMAJOR)
    _quant_check(torch.randn(129, 592, generator=g).to(torch.bfloat16))


def test_quantize_global_scale_from_a_negative_extreme():
    g = torch.Generator().manual_seed(15)
    x = torch.randn(40, 256, generator=g)
    x[17, 100] = -23.5
    _quant_check(x.to(torch.bfloat16))


def test_quantize_precomputed_gs():
    g = torch.Generator().manual_seed(13)
    _quant_check((torch.randn(64, 512, generator=g) * 3).to(torch.bfloat16), gs_given=17.25)


def test_quantize_signed_zero_and_ties():
    # every E2M1 tie, tiny negatives rounding to -0, exact zeros, one zero block
    vals = np.array([6, -6, 3, -3, 1.5, 0.5, 0, -0.25, 0.75, 2.5, 5, 4, -1, 1, 2, -2,
                     6, -0.1, -0.0, 0.2, -0.01, 0.01, -0.2, 0.24, 0, 0, 0, 0, 0, 0, 0, 0,
                     0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0], np.float32)
    x = torch.from_numpy(np.tile(vals, (4, 1))).to(torch.bfloat16)
    codes, _ = _quant_check(x, gs_given=1.0)
    assert codes[0, 8] & 0xF0 == 0x80            # -0.1 -> code 0x8
    assert codes[0, 9] & 0x0F == 0x08            # -0.0 in a nonzero block -> code 0x8
    assert codes[0, 10] & 0x0F == 0x08           # -0.01 -> code 0x8


def test_quantize_linear_workload_edge_blocks():
    cfg = W.CONFIGS["linear"]
    inp = W.linear_inputs(cfg, seed=0)
    codes, sf = _quant_check(inp["x"])
    flat_sf = sf.reshape(-1)
    assert np.all(flat_sf[inp["zero_blocks"].numpy()] == 0)
    assert np.all(flat_sf[inp["underflow_blocks"].numpy()] == 0)
    assert np.all(flat_sf[inp["small_raw_blocks"].numpy()] != 0)
    cb = codes.reshape(-1, 8)
    assert not cb[inp["underflow_blocks"].numpy()].any()


def test_quantize_row_gather_and_zero_rows():
    g = torch.Generator().manual_seed(14)
    x = torch.randn(20, 256, generator=g).to(torch.bfloat16)
    src = torch.tensor([3, -1, 0, 19, 3, -1, 7], dtype=torch.int32)
    codes, sf, gs = B.nvfp4_quantize(x.to(DEV), row_src=src.to(DEV), sf_layout=B.NVFP4_SF_ROWMAJOR)
    torch.cuda.synchronize()
    xb = W.bf16_bits(x)
    used = xb[[3, 0, 19, 7]]
    gs_ref = O.global_scale(O.amax_bf16(used))
    assert gs.item() == gs_ref
    rc, rs = O.quantize_bf16(xb, gs_ref)
    gc = codes.cpu().numpy()
    gsf = sf.cpu().numpy().reshape(7, 16)
    for r, s in enumerate(src.tolist()):
        if s < 0:
            assert not gc[r].any() and not gsf[r].any()
        else:
            assert np.array_equal(gc[r], rc[s]) and np.array_equal(gsf[r], rs[s])


def test_weight_preparation_bit_exact_with_interleave():
    cfg = W.CONFIGS["tiny"]
    inp = W.moe_inputs(cfg, seed=0)
    wts = B.prepare_moe_weights(inp["w1"].to(DEV), inp["w2"].to(DEV))
    torch.cuda.synchronize()
    w1 = W.bf16_bits(inp["w1"])
    w2 = W.bf16_bits(inp["w2"])
    E, two_i, K = w1.shape
    I = two_i // 2
    sf1 = wts["w1_sf"].cpu().numpy().reshape(E, -1)
    sf2 = wts["w2_sf"].cpu().numpy().reshape(E, -1)
    for e in range(E):
        c, s, g = O.quantize_expert(w1[e])
        assert wts["gs_w1"][e].item() == g
        assert np.array_equal(wts["w1_codes"][e].cpu().numpy(), O.interleave_rows(c, 8))
        assert np.array_equal(sf_tiled_to_rowmajor(sf1[e], two_i, K), O.interleave_rows(s, 8))
        c, s, g = O.quantize_expert(w2[e])
        assert wts["gs_w2"][e].item() == g
        assert np.array_equal(wts["w2_codes"][e].cpu().numpy(), c)
        assert np.array_equal(sf_tiled_to_rowmajor(sf2[e], K, I), s)


def test_dispatch_quantize_padded_rows_bit_exact():
    cfg = W.CONFIGS["tiny"]
    inp = W.moe_inputs(cfg, seed=1, weights=False)
    x = inp["x"]
    ids, _ = O.route_topk(inp["logits"].numpy(), cfg.k)
    offsets, p2f, f2p = O.permute(ids, cfg.E)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    a_codes, a_sf, gs = B.moe_quantize_dispatch(x.to(DEV), d(ids), d(offsets), d(f2p), cfg.E)
    torch.cuda.synchronize()
    xb = W.bf16_bits(x)
    gs_ref = O.global_scale(O.amax_bf16(xb))
    assert gs.item() == gs_ref
    rc, rs = O.quantize_bf16(xb, gs_ref)
    prow = padded_rows_of_compact(offsets)
    a_rows = a_codes.shape[0]
    gsf = sf_rows_to_rowmajor(a_sf.cpu().numpy(), a_rows, cfg.K)
    gc = a_codes.cpu().numpy()
    for r in range(cfg.M):
        t = p2f[r] // cfg.k
        assert np.array_equal(gc[prow[r]], rc[t])
        assert np.array_equal(gsf[prow[r]], rs[t])


def test_quantize_underflow_boundary():
    """Blocks whose scaled maximum p = amax * gs sits exactly at 6 * 2^-9 (not an
    underflow block: the rule is strict), one BF16 step below it (underflow:
    scale 0, codes 0) and one step above."""
    thr_raw = 3.0 * 2.0 ** -10                    # * gs 4 = 6 * 2^-9, exact in BF16
    step = 2.0 ** -7 * 2.0 ** -9                  # one BF16 ulp at 1.5 * 2^-9
    rows = []
    for amax in (thr_raw, thr_raw - step, thr_raw + step):
        for sign in (1.0, -1.0):
            r = np.zeros(64, np.float32)
            r[5] = sign * amax
            r[9] = amax / 4
            r[16 + 2] = sign * amax                   # a second block in the row
            rows.append(r)
    x = torch.from_numpy(np.stack(rows)).to(torch.bfloat16)
    _, sf = _quant_check(x, gs_given=4.0, layout=B.NVFP4_SF_ROWMAJOR)
    assert np.all(sf[0:2, 0:2] == 1)                  # exactly at the threshold: 2^-9
    assert np.all(sf[2:4, 0:2] == 0)                  # below: underflow
    assert np.all(sf[4:6, 0:2] != 0)
