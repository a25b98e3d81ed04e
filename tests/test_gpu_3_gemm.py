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


def test_swiglu_epilogue_against_oracle_requant():
    """L1 GEMM + SwiGLU + NVFP4 requant: h scales/codes equal the oracle's
    requantization of its own fp64 SwiGLU output except where f32 accumulation
    lands on the other side of a rounding boundary (rare, one code step)."""
    rng = np.random.default_rng(4)
    counts = [3, 0, 140, 64, 1]
    E, I, K = len(counts), 128, 512
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(offsets[-1])
    ac, asf, gsa = _rand_q(rng, M, K, 1.0)
    w1 = []
    for _ in range(E):
        x = rng.normal(0, 0.05, (2 * I, K)).astype(np.float32)
        g = O.global_scale(O.amax_f32(x))
        c, s = O.quantize_f32(x, g)
        w1.append((c, s, g))
    gs_h = np.float32(2688.0 / 8.0)
    # oracle: natural [gate | up] weights
    h_ref = np.zeros((M, I), np.float32)
    A = O.dequantize_f64(ac, asf, gsa)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            v = O.matmul_nt(A[r0:r1], O.dequantize_f64(w1[e][0], w1[e][1], w1[e][2]))
            h_ref[r0:r1] = O.swiglu(v)
    hc_ref, hs_ref = O.quantize_f32(h_ref, gs_h)
    # device: interleaved weights, padded activations
    a_rows = B.nvfp4moe_padded_rows(M, E)
    prow = padded_rows_of_compact(offsets)
    a_pad = np.zeros((a_rows, K // 2), np.uint8)
    a_pad[prow] = ac
    asf_rm = np.zeros((a_rows, K // 16), np.uint8)
    asf_rm[prow] = asf
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    w1c = np.stack([O.interleave_rows(w[0], 8) for w in w1])
    w1s = np.concatenate([_tile_sf(O.interleave_rows(w[1], 8), 2 * I, K) for w in w1])
    gsw = np.array([w[2] for w in w1], np.float32)
    h_codes, h_sf = B.nvfp4_grouped_gemm_swiglu(d(a_pad), d(_rows_sf(asf_rm, a_rows, K)),
                                                d(np.array([gsa], np.float32)), d(w1c), d(w1s), d(gsw),
                                                d(offsets), d(np.array([gs_h], np.float32)))
    assert B.nvfp4moe_last_device_status() == 0
    gc = h_codes.cpu().numpy()[prow]
    gs_rm = h_sf.cpu().numpy()[sf_rows_index(a_rows, I)][prow]
    sf_mismatch = np.mean(gs_rm != hs_ref)
    code_mismatch = np.mean(gc != hc_ref)
    hd_gpu = O.dequantize_f64(gc, gs_rm, gs_h)
    hd_ref = O.dequantize_f64(hc_ref, hs_ref, gs_h)
    if sf_mismatch > 0.01 or code_mismatch > 0.01:
        _dump("swiglu", gc=gc, gs=gs_rm, hc_ref=hc_ref, hs_ref=hs_ref, h_ref=h_ref)
    assert sf_mismatch <= 0.01, sf_mismatch
    assert code_mismatch <= 0.01, code_mismatch
    assert cosine(hd_gpu, hd_ref) > 0.999
