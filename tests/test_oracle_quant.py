"""Pins of the oracle's block quantizer, round trip and gate/up interleave.

Sources: "NVFP4 MegaMoE Kernel" README -- "What We Have" (16-element blocks,
E4M3 block scale, FP32 global scale), "Correctness Bugs Fixed" bugs 2
(dequantize -> requantize is byte-identical), 3 (all-zero block -> scale 0),
4 (underflow block -> zero codes), "Fused SwiGLU - How It Works" (gate/up
interleave at granularity 8 and the //2 bug).
"""
import numpy as np
import torch

import oracle as O
from conftest import golden_path
from nvfp4_block_scaled_05_gb300.workloads import bf16_bits


def _bits(vals):
    return bf16_bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))


def test_hand_worked_blocks_golden():
    n = 0
    for line in open(golden_path("quant_blocks.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        gs_s, vals_s, sf_s, codes_s = [p.strip() for p in line.split(";")]
        vals = [float(v) for v in vals_s.split()]
        x = _bits([vals])
        back = x.view(np.uint16).astype(np.uint32) << 16
        assert np.array_equal(back.view(np.float32)[0], np.float32(vals)), "not exact in BF16"
        codes, sf = O.quantize_bf16(x, np.float32(gs_s))
        assert sf[0, 0] == int(sf_s, 16), (line, hex(sf[0, 0]))
        assert [int(c, 16) for c in codes_s.split()] == list(codes[0]), (line, codes[0])
        n += 1
    assert n == 8


def test_zero_block_exact_zero_scale():
    x = np.zeros((3, 64), np.uint16)
    codes, sf = O.quantize_bf16(x, np.float32(7.0))
    assert not codes.any() and not sf.any()


def test_underflow_threshold_in_scaled_domain():
    thr = 6 * 2.0 ** -9
    gs = np.float32(3.0)
    # block maximum just below / at the threshold after scaling by gs
    for amax, expect_zero in [(thr / 3 * 0.999, True), (thr / 3 * 1.01, False)]:
        v = np.zeros((1, 16), np.float32)
        v[0, 0] = amax
        codes, sf = O.quantize_f32(v, gs)
        assert (sf[0, 0] == 0 and not codes.any()) == expect_zero, amax
    # exactly at the threshold the block is not an underflow block (the rule is
    # amax < 6*2^-9, strict): scale 2^-9 (E4M3 code 1) and the element maps to 6
    v = np.zeros((1, 16), np.float32)
    v[0, 3] = np.float32(thr / 4)
    codes, sf = O.quantize_f32(v, np.float32(4.0))
    assert sf[0, 0] == 1 and codes[0, 1] == 0x70 and codes.sum() == 0x70
    # a raw block maximum below 6*2^-9 is still a normal block when gs is large
    v = np.full((1, 16), 0.005, np.float32)
    codes, sf = O.quantize_f32(v, np.float32(100.0))
    assert sf[0, 0] != 0 and codes.any()


def test_error_bound_per_element():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, (64, 256)).astype(np.float32)
    gs = O.global_scale(O.amax_f32(x))
    codes, sf = O.quantize_f32(x, gs)
    deq = O.dequantize_f64(codes, sf, gs)
    s = np.array([[O.e4m3_decode(b) for b in row] for row in sf])
    s_el = np.repeat(s, 16, axis=1) / float(gs)
    xn = np.abs(x) / s_el
    # half of the E2M1 grid spacing at the element's magnitude; saturation is
    # bounded by the scale's own rounding (x_norm <= 6 * (1 + 2^-4))
    half = np.where(xn < 2, 0.25, np.where(xn < 4, 0.5, 1.0))
    assert np.all(np.abs(deq - x) <= half * s_el * (1 + 1e-6) + 6 * 2 ** -4 * s_el)
    # and the block maximum is represented by +-6 (scale = amax*gs/6 rounded)
    cmax = np.array([[max(O.e2m1_decode(c & 15), O.e2m1_decode(c >> 4), key=abs) for c in r]
                     for r in codes])
    blk_max_code = np.abs(cmax).reshape(64, 16, 8).max(axis=2)
    assert np.all(blk_max_code == 6.0)


def test_tensor_max_block_gets_scale_448():
    rng = np.random.default_rng(4)
    x = rng.normal(0, 1, (8, 128)).astype(np.float32)
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    gs = O.global_scale(O.amax_f32(x))
    codes, sf = O.quantize_f32(x, gs)
    assert O.e4m3_decode(sf[r, c // 16]) == 448.0
    byte = codes[r, c // 2]
    code = (byte >> 4) if c % 2 else (byte & 15)
    assert abs(O.e2m1_decode(code)) == 6.0


def test_round_trip_byte_identical():
    """Bug 2: requantize(dequantize(q)) == q, dequantizing in f32.

    Exception made by the threshold rule itself: a block whose scale is the
    smallest subnormal (0x01) can dequantize to a maximum one ulp under the
    underflow threshold and is then zeroed; such blocks are excluded.
    """
    rng = np.random.default_rng(5)
    for gs_mult in [1.0, 0.37, 13.0]:
        x = rng.normal(0, 1, (32, 512)).astype(np.float32)
        x[3, :64] = 0.0                          # zero blocks
        x[5, 16:32] *= 1e-7                      # underflow blocks
        x[7, 32:48] *= 1e-3
        gs = np.float32(O.global_scale(O.amax_f32(x)) * gs_mult)
        codes, sf = O.quantize_f32(x, gs)
        deq = O.dequantize_f32(codes, sf, gs)
        codes2, sf2 = O.quantize_f32(deq, gs)
        keep = sf != 1
        assert np.array_equal(sf2[keep], sf[keep])
        kc = np.repeat(keep, 8, axis=1)
        assert np.array_equal(codes2[kc], codes[kc])
        assert (sf == 0).any()


def test_round_trip_bf16_weights():
    w = bf16_bits((torch.randn(64, 512, generator=torch.Generator().manual_seed(6)) * 0.02).to(torch.bfloat16))
    c, s, gs = O.quantize_expert(w)
    d = O.dequantize_f32(c, s, gs)
    c2, s2 = O.quantize_f32(d, gs)
    assert np.array_equal(c, c2) and np.array_equal(s, s2)


def test_interleave_identity_and_granularity():
    I, K = 64, 32
    a = np.arange(2 * I * K, dtype=np.int32).reshape(2 * I, K)
    il = O.interleave_rows(a, 8)
    assert np.array_equal(O.deinterleave_rows(il, 8), a)
    # granularity exactly 8 (not 4, the //2 bug): rows 0-7 gate 0-7, 8-15 up 0-7
    assert np.array_equal(il[0:8], a[0:8])
    assert np.array_equal(il[8:16], a[I:I + 8])
    assert np.array_equal(il[16:24], a[8:16])
    assert np.array_equal(il[24:32], a[I + 8:I + 16])
    assert not np.array_equal(il, O.interleave_rows(a, 4))
    assert np.array_equal(O.interleave_rows(a), il) and np.array_equal(O.deinterleave_rows(il), a)


def test_interleave_commutes_with_quantize():
    w = bf16_bits(torch.randn(256, 128, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16))
    gs = O.global_scale(O.amax_bf16(w))
    c1, s1 = O.quantize_bf16(O.interleave_rows(w, 8), gs)
    c0, s0 = O.quantize_bf16(w, gs)
    assert np.array_equal(c1, O.interleave_rows(c0, 8))
    assert np.array_equal(s1, O.interleave_rows(s0, 8))
