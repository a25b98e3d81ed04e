"""GPU parity of the tcgen05 block-scaled grouped GEMMs against the fp64 oracle.

Inputs are built in the oracle's formats and laid out on the device with the
documented layouts (grouped-padded rows, tiled scales), so both sides see the
same bytes. Structured inputs (constant codes and scales) come first, so that a
failure says which part of the operand layout is wrong; on failure the raw GPU
output is saved to the folder named by NVFP4MOE_DUMP_DIR, when that is set.
"""
import os

import numpy as np
import pytest
import torch

import oracle as O
from helpers import (assert_close_tol, cosine, padded_rows_of_compact, padded_starts,
                     sf_rows_index, sf_tiled_index)
from nvfp4_block_scaled_05_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dump(name, **arrays):
    d = os.environ.get("NVFP4MOE_DUMP_DIR")
    if d and os.path.isdir(d):
        np.savez(os.path.join(d, "fail_%s.npz" % name), **arrays)


def _tile_sf(sf_rm, rows_cap, cols):
    """Row-major (rows, cols/16) scales -> tiled bytes of a (rows_cap, cols) matrix
    (the weight operand's layout)."""
    out = np.zeros(B.nvfp4_sf_bytes(rows_cap, cols), np.uint8)
    rows = sf_rm.shape[0]
    out[sf_tiled_index(rows, cols)] = sf_rm
    return out


def _rows_sf(sf_rm, rows_cap, cols):
    """Row-major (rows, cols/16) scales -> NVFP4_SF_TILED_ROWS bytes of a
    (rows_cap, cols) matrix (the activation operand's layout)."""
    out = np.zeros(B.nvfp4_sf_bytes(rows_cap, cols, B.NVFP4_SF_TILED_ROWS), np.uint8)
    rows = sf_rm.shape[0]
    out[sf_rows_index(rows, cols)] = sf_rm
    return out


def _rand_q(rng, rows, cols, std, mode="random"):
    if mode == "ones":
        codes = np.full((rows, cols // 2), 0x22, np.uint8)      # every element 1.0
        sf = np.full((rows, cols // 16), 0x38, np.uint8)        # every scale 1.0
        return codes, sf, np.float32(1.0)
    if mode == "codes":
        codes = rng.integers(0, 256, (rows, cols // 2)).astype(np.uint8)
        sf = np.full((rows, cols // 16), 0x38, np.uint8)
        return codes, sf, np.float32(1.0)
    if mode == "scales":
        codes = np.full((rows, cols // 2), 0x22, np.uint8)
        sf = rng.integers(0x20, 0x50, (rows, cols // 16)).astype(np.uint8)
        return codes, sf, np.float32(1.0)
    x = rng.normal(0, std, (rows, cols)).astype(np.float32)
    gs = O.global_scale(O.amax_f32(x))
    c, s = O.quantize_f32(x, gs)
    return c, s, gs


def _run_grouped(rng, counts, N, K, mode_a="random", mode_b="random", name="g", wide=False):
    E = len(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(offsets[-1])
    ac, asf, gsa = _rand_q(rng, M, K, 1.0, mode_a)
    bl = [_rand_q(rng, N, K, 0.02, mode_b) for _ in range(E)]
    bc = np.stack([b[0] for b in bl])
    bsf = np.stack([b[1] for b in bl])
    gsb = np.array([b[2] for b in bl], np.float32)
    ref = O.grouped_gemm(ac, asf, gsa, bc, bsf, gsb, offsets)
    # device layouts
    a_rows = B.nvfp4moe_padded_rows(M, E)
    prow = padded_rows_of_compact(offsets)
    a_pad = np.zeros((a_rows, K // 2), np.uint8)
    a_pad[prow] = ac
    asf_rm = np.zeros((a_rows, K // 16), np.uint8)
    asf_rm[prow] = asf
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    a_sf_t = _rows_sf(asf_rm, a_rows, K)
    b_sf_t = np.concatenate([_tile_sf(bsf[e], N, K) for e in range(E)])
    out = None
    if wide:
        # a 16-byte-offset view with ldc % 16 != 0: the 16-byte store path
        out = torch.zeros((max(M, 1), N + 24), dtype=torch.bfloat16, device=DEV)[:M, 8:8 + N]
    c = B.nvfp4_grouped_gemm(d(a_pad), d(a_sf_t), d(np.array([gsa], np.float32)), d(bc), d(b_sf_t),
                             d(gsb), d(offsets), out=out)
    st = B.nvfp4moe_last_device_status()
    got = c.float().cpu().numpy()
    ok = st == 0 and np.all(np.abs(got - ref) <= 2e-2 * np.maximum(1.0, np.abs(ref)))
    if not ok:
        _dump(name, got=got, ref=ref, offsets=offsets, ac=ac, asf=asf, bc=bc, bsf=bsf, gsa=gsa, gsb=gsb)
    assert st == 0, "device status %d" % st
    return got, ref


@pytest.mark.parametrize("mode", ["ones", "codes", "scales", "random"])
def test_single_tile_structured(mode):
    rng = np.random.default_rng(1)
    got, ref = _run_grouped(rng, [128], 128, 256, mode, mode, name="single_" + mode)
    assert_close_tol(got, ref, mode)
    assert cosine(got, ref) > 0.9999


def test_grouped_uneven_groups_and_empty_experts():
    rng = np.random.default_rng(2)
    got, ref = _run_grouped(rng, [5, 0, 130, 1, 0, 300, 17, 128], 256, 512, name="uneven")
    assert_close_tol(got, ref, "uneven")
    assert cosine(got, ref) > 0.9999
    rel = np.abs(got - ref) / (np.abs(ref).max())
    assert rel.max() < 1e-2


@pytest.mark.parametrize("K", [64, 128, 192, 320, 7168])
def test_k_tails(K):
    rng = np.random.default_rng(K)
    got, ref = _run_grouped(rng, [40, 200], 128, K, name="k%d" % K)
    assert_close_tol(got, ref, "K=%d" % K)
    assert cosine(got, ref) > 0.9999


def test_strided_output_matches_sector_path():
    """The same GEMM into a 16-byte-offset, odd-stride output view (16-byte
    stores) gives the same bits as into a packed output (32-byte stores)."""
    got_w, ref = _run_grouped(np.random.default_rng(11), [70, 0, 200], 256, 512, name="wide", wide=True)
    got_p, _ = _run_grouped(np.random.default_rng(11), [70, 0, 200], 256, 512, name="packed")
    assert np.array_equal(got_w, got_p)
    assert_close_tol(got_w, ref, "wide")


def test_linear_workload_sampled_rows():
    """The shared-expert linear (M=4096, K=7168, N=4096, one expert), every
    output column of 64 sampled rows against the fp64 oracle."""
    from nvfp4_block_scaled_05_gb300 import workloads as W
    cfg = W.CONFIGS["linear"]
    inp = W.linear_inputs(cfg, seed=0, device=DEV)
    xq, xsf, gsx = B.nvfp4_quantize(inp["x"], sf_layout=B.NVFP4_SF_TILED_ROWS)
    wq, wsf, gsw = B.nvfp4_quantize(inp["w"][0])
    offsets = torch.tensor([0, cfg.M], dtype=torch.int32, device=DEV)
    c = B.nvfp4_grouped_gemm(xq, xsf, gsx, wq.view(1, cfg.N, cfg.K // 2), wsf, gsw, offsets)
    assert B.nvfp4moe_last_device_status() == 0
    rows = np.sort(np.random.default_rng(0).choice(cfg.M, 64, replace=False))
    xb = W.bf16_bits(inp["x"])
    wb = W.bf16_bits(inp["w"][0])
    g1 = O.global_scale(O.amax_bf16(xb))
    g2 = O.global_scale(O.amax_bf16(wb))
    assert gsx.item() == g1 and gsw.item() == g2
    xc, xs = O.quantize_bf16(xb[rows], g1)
    wc, ws = O.quantize_bf16(wb, g2)
    ref = O.matmul_nt(O.dequantize_f64(xc, xs, g1), O.dequantize_f64(wc, ws, g2))
    got = c[torch.from_numpy(rows).to(DEV)].float().cpu().numpy()
    if not np.all(np.abs(got - ref) <= 2e-2 * np.maximum(1.0, np.abs(ref))):
        _dump("linear", got=got, ref=ref, rows=rows)
    assert_close_tol(got, ref, "linear")
    assert cosine(got, ref) > 0.9999


# ---------------------------------------------------------------- SwiGLU + requant epilogue
#
# The format restated here, independently of the oracle's encoders, to bound
# which codes and scales a kernel whose f32 h is within a known relative error
# of the exact h may legitimately write.

_E2M1_TH = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
_E4M3_VALS = np.array([(c & 7) * 2.0 ** -9 if c < 8 else (1 + (c & 7) / 8) * 2.0 ** ((c >> 3) - 7)
                       for c in range(127)])


def _e2m1_mag(a):
    """E2M1 magnitude index (0..7) of a >= 0: nearest of {0,.5,1,1.5,2,3,4,6},
    ties to the even index, saturating at 6."""
    idx = np.searchsorted(_E2M1_TH, a, side="left")
    tie = (idx < 7) & (_E2M1_TH[np.minimum(idx, 6)] == a)
    return np.where(tie & (idx % 2 == 1), idx + 1, idx)


def _e4m3_code(x):
    """E4M3 code (0..126) of x >= 0: nearest value, ties to the even code,
    saturating at 448."""
    i = np.clip(np.searchsorted(_E4M3_VALS, x, side="left"), 1, 126)
    lo, hi = _E4M3_VALS[i - 1], _E4M3_VALS[i]
    c = np.where(x - lo < hi - x, i - 1, np.where(hi - x < x - lo, i, np.where((i - 1) % 2 == 0, i - 1, i)))
    return np.where(x >= 448.0, 126, np.where(x <= 0, 0, c))


def _silu_rel_err(g):
    """Relative error bound of the kernel's f32 silu(g) * u for exact g, u: its
    exponential (__expf: at most 2 + floor(1.173 |x|) ulp), the rounding of
    1 + e, its divide (__fdividef: at most 2 ulp for divisors in [2^-126,
    2^126]) and the product with u, each at most 2^-23 relative per ulp,
    doubled as margin. Where 1 + exp(-g) exceeds 2^126 the fast divide returns
    0: relative error 1 (the exact value there is below 1e-36)."""
    rho = 2.0 * (5.0 + np.floor(1.173 * np.abs(g))) * 2.0 ** -23
    return np.where(-g > 87.0, 1.0, rho)


def _unjustified_requant(h64, rho, gs_h, gc, gsf):
    """Counts of h scale bytes and h codes the kernel wrote that NO f32 value
    within relative error rho of the exact h (h64, fp64) can produce under the
    block rule (p = amax * gs_h; scale 0 and codes 0 below 6 * 2^-9; sf =
    E4M3(p / 6); code = E2M1(h * gs_h / value(sf)), sign kept), allowing
    4 * 2^-24 more for the f32 roundings of the products and the quotient.
    Codes are judged against the scale the kernel wrote."""
    eps = 4 * 2.0 ** -24
    rows, I = h64.shape
    a = np.abs(h64)
    ab, rb = a.reshape(rows, I // 16, 16), rho.reshape(rows, I // 16, 16)
    p_lo = (ab * (1 - rb)).max(axis=2) * gs_h * (1 - eps)
    p_hi = (ab * (1 + rb)).max(axis=2) * gs_h * (1 + eps)
    thr = 6 * 2.0 ** -9
    c_lo = np.where(p_lo < thr, 0, _e4m3_code(p_lo / 6 * (1 - eps)))
    c_hi = np.where(p_hi < thr, 0, _e4m3_code(p_hi / 6 * (1 + eps)))
    gsf = gsf.astype(np.int64)
    bad_sf = (gsf < c_lo) | (gsf > c_hi) | (gsf > 126)
    code = np.empty((rows, I), np.int64)
    code[:, 0::2] = gc & 15
    code[:, 1::2] = gc >> 4
    mag, neg = code & 7, code >> 3
    zero_blk = np.repeat(gsf == 0, 16, axis=1)
    s = np.repeat(_E4M3_VALS[np.minimum(gsf, 126)], 16, axis=1)
    xn = np.where(zero_blk, 0.0, a * gs_h / np.where(s > 0, s, 1.0))
    m_lo = _e2m1_mag(xn * (1 - rho) * (1 - eps))
    m_hi = _e2m1_mag(xn * (1 + rho) * (1 + eps))
    ok = np.where(zero_blk, code == 0,
                  (mag >= m_lo) & (mag <= m_hi) & ((mag == 0) | (h64 == 0) | (neg == (h64 < 0))))
    return int(bad_sf.sum()), int((~ok).sum())


def _swiglu_case(ac, asf, gsa, w1, offsets, gs_h):
    """Runs the fused L1 kernel on compact activations (ac, asf) and per-expert
    W1 (codes, scales, gs) in [gate | up] row order; returns the oracle's v
    (fp64, (M, 2I)), the GPU's h codes and row-major h scales."""
    E = len(w1)
    M = int(offsets[-1])
    K = ac.shape[1] * 2
    I = w1[0][0].shape[0] // 2
    v = np.zeros((M, 2 * I), np.float64)
    A = O.dequantize_f64(ac, asf, gsa)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            v[r0:r1] = O.matmul_nt(A[r0:r1], O.dequantize_f64(w1[e][0], w1[e][1], w1[e][2]))
    a_rows = B.nvfp4moe_padded_rows(M, E)
    prow = padded_rows_of_compact(offsets)
    a_pad = np.zeros((a_rows, K // 2), np.uint8)
    a_pad[prow] = ac
    asf_rm = np.zeros((a_rows, K // 16), np.uint8)
    asf_rm[prow] = asf
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    w1c = np.stack([O.interleave_rows(w[0], 8) for w in w1])
    w1s = np.concatenate([_tile_sf(O.interleave_rows(w[1], 8), 2 * I, K) for w in w1])
    gsw = np.array([w[2] for w in w1], np.float32)
    h_codes, h_sf = B.nvfp4_grouped_gemm_swiglu(d(a_pad), d(_rows_sf(asf_rm, a_rows, K)),
                                                d(np.array([gsa], np.float32)), d(w1c), d(w1s), d(gsw),
                                                d(offsets), d(np.array([gs_h], np.float32)))
    assert B.nvfp4moe_last_device_status() == 0
    gc = h_codes.cpu().numpy()[prow]
    gsf = h_sf.cpu().numpy()[sf_rows_index(a_rows, I)][prow]
    return v, gc, gsf


def _pow2_q(rng, rows, cols, exps):
    """Random E2M1 codes (all 16) with scales drawn from the powers of two
    2^e, e in exps (exact E4M3 values), global scale 1."""
    codes = rng.integers(0, 256, (rows, cols // 2)).astype(np.uint8)
    sf = np.array([_e4m3_code(2.0 ** e) for e in exps], np.uint8)[rng.integers(0, len(exps), (rows, cols // 16))]
    return codes, sf, np.float32(1.0)


def test_swiglu_epilogue_exact_accumulation_every_mismatch_justified():
    """K=7168, I=2048, 300 routed rows in three experts (one empty). Inputs are
    chosen so that the tensor core's f32 accumulation is exact: every operand
    value is a code times a power-of-two scale in [2^-3, 2^-2] (a multiple of
    2^-4 of magnitude <= 1.5), so every product is a multiple of 2^-8 and every
    partial sum is below 7168 * 2.25 < 2^14: at most 2^22 steps of 2^-8, exact
    in f32 whatever the order of the additions; global scales are 1. The kernel's v is then the exact v, which the plain
    BF16 GEMM on the same operands shows bit for bit. What remains between
    kernel and oracle is the f32 evaluation of silu(g) * u, whose documented
    error bound (_silu_rel_err) decides for each h scale and code which values
    are possible: none may fall outside that set."""
    rng = np.random.default_rng(21)
    counts = [130, 0, 170]
    E, I, K = len(counts), 2048, 7168
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(offsets[-1])
    ac, asf, gsa = _pow2_q(rng, M, K, [-3, -2])
    w1 = [_pow2_q(rng, 2 * I, K, [-3, -2]) for _ in range(E)]
    # gs_h from the exact h of these rows (a pre-computed scale, the same f32 on both sides)
    v_probe = O.matmul_nt(O.dequantize_f64(ac[:64], asf[:64], gsa), O.dequantize_f64(*w1[0]))
    h_probe = O.swiglu(v_probe)
    gs_h = np.float32(2688.0 / (1.5 * np.abs(h_probe).max()))
    v, gc, gsf = _swiglu_case(ac, asf, gsa, w1, offsets, gs_h)
    # the accumulation is exact: the BF16 GEMM output equals RN_bf16(v) bit for bit
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    a_rows = B.nvfp4moe_padded_rows(M, E)
    prow = padded_rows_of_compact(offsets)
    a_pad = np.zeros((a_rows, K // 2), np.uint8)
    a_pad[prow] = ac
    asf_rm = np.zeros((a_rows, K // 16), np.uint8)
    asf_rm[prow] = asf
    bsf = np.concatenate([_tile_sf(w[1], 2 * I, K) for w in w1])
    c = B.nvfp4_grouped_gemm(d(a_pad), d(_rows_sf(asf_rm, a_rows, K)), d(np.array([1.0], np.float32)),
                             d(np.stack([w[0] for w in w1])), d(bsf), d(np.ones(E, np.float32)), d(offsets))
    assert B.nvfp4moe_last_device_status() == 0
    want = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(v.astype(np.float32).astype(np.float64), v)   # v exact in f32
    assert torch.equal(c.cpu(), want), "BF16 GEMM differs from RN(exact v)"
    # h: exact in fp64 from the exact v, the kernel's f32 within _silu_rel_err
    g, u = v[:, :I], v[:, I:]
    h64 = g / (1.0 + np.exp(-g)) * u
    rho = _silu_rel_err(g)
    bad_sf, bad_codes = _unjustified_requant(h64, rho, gs_h, gc, gsf)
    hc_ref, hs_ref = O.quantize_f32(O.swiglu(v), gs_h)
    print("exact-accumulation SwiGLU: %d of %d h scales and %d of %d h codes differ from the oracle's "
          "requantization, all within the silu error bound" % (int((gsf != hs_ref).sum()), gsf.size,
                                                               int((gc != hc_ref).sum()), gc.size))
    if bad_sf or bad_codes:
        _dump("swiglu_exact", gc=gc, gsf=gsf, v=v, gs_h=gs_h)
    assert bad_sf == 0 and bad_codes == 0, (bad_sf, bad_codes)
    # a wrong pairing, a wrong scale column or a missing term would show here
    assert np.mean(gsf != hs_ref) < 1e-3 and np.mean(gc != hc_ref) < 1e-3


def test_swiglu_epilogue_against_oracle_requant():
    """L1 GEMM + SwiGLU + NVFP4 requant at the layer's size (K=7168, I=2048,
    400 routed rows in five experts, one empty) on random N(0,1) activations
    and N(0,0.05) weights: h scales and codes equal the oracle's
    requantization of its fp64 SwiGLU output except where the kernel's f32
    accumulation (and its f32 silu) lands on the other side of a rounding
    boundary. Such an element sits within the accumulation error of a
    boundary, so it differs by one step of the format: a code by one E2M1
    magnitude step (or only in the sign of a zero), a scale by one E4M3 code.
    The measured rates at this size are a few per 10^4 (printed); the bound
    is 2e-3 for both, and every mismatch must be a one-step one."""
    rng = np.random.default_rng(4)
    counts = [3, 0, 140, 192, 65]
    E, I, K = len(counts), 2048, 7168
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(offsets[-1])
    ac, asf, gsa = _rand_q(rng, M, K, 1.0)
    w1 = []
    for _ in range(E):
        x = rng.normal(0, 0.05, (2 * I, K)).astype(np.float32)
        g = O.global_scale(O.amax_f32(x))
        c, s = O.quantize_f32(x, g)
        w1.append((c, s, g))
    gs_h = np.float32(2688.0 / 16.0)
    v, gc, gsf = _swiglu_case(ac, asf, gsa, w1, offsets, gs_h)
    hc_ref, hs_ref = O.quantize_f32(O.swiglu(v), gs_h)
    sf_mis = gsf != hs_ref
    code_mis = gc != hc_ref
    print("random SwiGLU (K=%d, I=%d, %d rows): h scale mismatch rate %.2e, h code byte mismatch rate %.2e"
          % (K, I, M, sf_mis.mean(), code_mis.mean()))
    # one E4M3 step for every differing scale
    assert np.all(np.abs(gsf.astype(int) - hs_ref.astype(int))[sf_mis] == 1)
    # one E2M1 magnitude step (or a signed zero) for every differing code, in
    # blocks whose scale agrees
    same_sf = np.repeat(~sf_mis, 8, axis=1)
    for sh in (0, 4):
        a = (gc >> sh) & 15
        b = (hc_ref >> sh) & 15
        d = (a != b) & same_sf
        step = np.abs((a & 7).astype(int) - (b & 7).astype(int))
        sign_ok = ((a >> 3) == (b >> 3)) | ((a & 7) == 0) | ((b & 7) == 0)
        assert np.all((step <= 1)[d] & sign_ok[d]), "a code differs by more than one step"
    if sf_mis.mean() > 2e-3 or code_mis.mean() > 2e-3:
        _dump("swiglu", gc=gc, gs=gsf, hc_ref=hc_ref, hs_ref=hs_ref)
    assert sf_mis.mean() <= 2e-3, sf_mis.mean()
    assert code_mis.mean() <= 2e-3, code_mis.mean()
    hd_gpu = O.dequantize_f64(gc, gsf, gs_h)
    hd_ref = O.dequantize_f64(hc_ref, hs_ref, gs_h)
    assert cosine(hd_gpu, hd_ref) > 0.9999


@pytest.mark.parametrize("swiglu", [False, True])
def test_pair_kernel_equals_single_cta_kernel(swiglu):
    """The 2-SM pair kernel (a cluster of two CTAs sharing one tcgen05 MMA of
    256 rows, each loading half of the weight tile) and the one-CTA-per-tile
    kernel give the same bits, on groups with odd and even numbers of
    activation tiles (the odd CTA of a pair then has no rows), an empty group
    and one-row groups."""
    rng = np.random.default_rng(31)
    counts = [1, 0, 129, 256, 300, 77, 512, 1]
    E, K = len(counts), 1024
    N = 512 if not swiglu else 1024
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(offsets[-1])
    ac, asf, gsa = _rand_q(rng, M, K, 1.0)
    bl = [_rand_q(rng, N, K, 0.05) for _ in range(E)]
    a_rows = B.nvfp4moe_padded_rows(M, E)
    prow = padded_rows_of_compact(offsets)
    a_pad = np.zeros((a_rows, K // 2), np.uint8)
    a_pad[prow] = ac
    asf_rm = np.zeros((a_rows, K // 16), np.uint8)
    asf_rm[prow] = asf
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    args = (d(a_pad), d(_rows_sf(asf_rm, a_rows, K)), d(np.array([gsa], np.float32)),
            d(np.stack([b[0] for b in bl])), d(np.concatenate([_tile_sf(b[1], N, K) for b in bl])),
            d(np.array([b[2] for b in bl], np.float32)), d(offsets))
    outs = []
    for mode in (1, 0):
        B.nvfp4moe_set_gemm_mode(mode)
        try:
            if swiglu:
                hc, hs = B.nvfp4_grouped_gemm_swiglu(*args, d(np.array([2688.0 / 4.0], np.float32)))
                outs.append((hc.cpu()[torch.from_numpy(prow)], hs.cpu()[torch.from_numpy(sf_rows_index(a_rows, N // 2)[prow].reshape(-1))]))
            else:
                outs.append((B.nvfp4_grouped_gemm(*args).cpu(),))
        finally:
            B.nvfp4moe_set_gemm_mode(0)
        assert B.nvfp4moe_last_device_status() == 0
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    if not swiglu:
        ref = O.grouped_gemm(ac, asf, gsa, np.stack([b[0] for b in bl]), np.stack([b[1] for b in bl]),
                             np.array([b[2] for b in bl], np.float32), offsets)
        got = outs[0][0].float().numpy()
        assert_close_tol(got, ref, "pair")
        assert cosine(got, ref) > 0.9999
