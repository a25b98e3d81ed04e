"""Pins of the oracle's routing, permutation, GEMM, SwiGLU and combine.

Sources: "NVFP4 MegaMoE Kernel" README -- "MoE Runner" (the six steps),
"Correctness Bugs Fixed" bug 5 (per-expert counts by bincount),
"ScaledGroupedGemmKernel" (A(M,K) x B(E,K,N) -> C(M,N), rows grouped by
expert), "Key Lessons" 10 (SwiGLU pairs silu(gate) with up).
Each check uses a library routine (numpy sort, bincount, matmul; torch softmax),
a closed form, brute force, or an invariance, not the oracle's own formula.
"""
import math

import numpy as np
import torch

import oracle as O
from nvfp4_block_scaled_05_gb300 import workloads as W


def test_route_topk_vs_stable_sort_and_softmax():
    rng = np.random.default_rng(0)
    logits = rng.normal(0, 1, (200, 32)).astype(np.float32)
    logits[0, :] = 0.5                      # all tied: lower index first
    logits[1, [3, 9, 20]] = 5.0             # three-way tie at the top
    ids, w = O.route_topk(logits, 6)
    ref = np.argsort(-logits, axis=1, kind="stable")[:, :6]
    assert np.array_equal(ids, ref)
    assert list(ids[1, :3]) == [3, 9, 20]
    sel = np.take_along_axis(logits, ref, axis=1)
    ref_w = torch.softmax(torch.from_numpy(sel).double(), dim=1).numpy()
    assert np.allclose(w, ref_w, rtol=0, atol=1e-14)
    assert np.allclose(w.sum(1), 1.0, atol=1e-14)


def test_route_ignores_minus_inf_experts():
    logits = np.zeros((4, 8), np.float32)
    logits[:, [1, 2]] = -np.inf
    ids, w = O.route_topk(logits, 6)
    assert not np.isin(ids, [1, 2]).any()
    assert np.allclose(w, 1 / 6)


def test_route_nan_logits_rank_as_minus_inf():
    """Reading R16: a NaN logit ranks as -inf (ties with -inf to the lower
    index); checked against numpy's stable argsort of the logits with NaN
    replaced by -inf, and torch's softmax over the selected values."""
    rng = np.random.default_rng(7)
    T, E, k = 300, 64, 8
    logits = rng.normal(0, 1, (T, E)).astype(np.float32)
    logits[rng.random((T, E)) < 0.1] = np.nan      # scattered NaNs
    logits[:20, 0] = np.nan                        # a NaN in front of every other logit
    logits[20, :] = np.nan                         # a NaN-only row except three finite logits
    logits[20, [5, 40, 63]] = [1.0, -2.0, 3.0]
    logits[21, :] = -np.inf                        # NaN and -inf tie: lower index first
    logits[21, [2, 9]] = np.nan
    logits[21, 30] = 0.0
    ids, w = O.route_topk(logits, k)
    mapped = np.where(np.isnan(logits), -np.inf, logits)
    ref = np.argsort(-mapped, axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, ref)
    assert list(ids[20, :3]) == [63, 5, 40] and list(ids[21, :3]) == [30, 0, 1]
    sel = np.take_along_axis(mapped, ref, axis=1)
    ref_w = torch.softmax(torch.from_numpy(sel).double(), dim=1).numpy()
    assert np.allclose(w, ref_w, rtol=0, atol=1e-14)
    assert np.all(w[20, 3:] == 0.0) and np.all(np.isfinite(w))


def test_permute_vs_stable_argsort_and_bincount():
    rng = np.random.default_rng(1)
    for T, k, E in [(1, 1, 1), (50, 2, 8), (300, 8, 64), (64, 4, 300)]:
        ids = rng.integers(0, E, (T, k)).astype(np.int32)
        offsets, p2f, f2p = O.permute(ids, E)
        assert np.array_equal(np.diff(offsets), np.bincount(ids.ravel(), minlength=E))
        assert np.array_equal(p2f, np.argsort(ids.ravel(), kind="stable"))
        assert np.array_equal(f2p[p2f], np.arange(T * k))
        assert offsets[0] == 0 and offsets[-1] == T * k


def test_permute_all_tokens_one_expert_and_empty_experts():
    ids = np.full((10, 1), 3, np.int32)
    offsets, p2f, f2p = O.permute(ids, 5)
    assert list(offsets) == [0, 0, 0, 0, 10, 10]
    assert list(p2f) == list(range(10))


def _rand_nvfp4(rng, rows, cols, scale=1.0):
    x = (rng.normal(0, scale, (rows, cols))).astype(np.float32)
    gs = O.global_scale(O.amax_f32(x))
    c, s = O.quantize_f32(x, gs)
    return c, s, gs


def test_grouped_gemm_vs_numpy_matmul():
    rng = np.random.default_rng(2)
    E, N, K = 3, 48, 64
    counts = [5, 0, 11]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ac, asf, gsa = _rand_nvfp4(rng, offsets[-1], K)
    bc, bsf, gsb = [], [], []
    for e in range(E):
        c, s, g = _rand_nvfp4(rng, N, K, 0.02)
        bc.append(c), bsf.append(s), gsb.append(g)
    C = O.grouped_gemm(ac, asf, gsa, np.stack(bc), np.stack(bsf), np.array(gsb, np.float32), offsets)
    A = O.dequantize_f64(ac, asf, gsa)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        ref = A[r0:r1] @ O.dequantize_f64(bc[e], bsf[e], gsb[e]).T
        assert np.allclose(C[r0:r1], ref, rtol=1e-12, atol=1e-12)


def test_matmul_brute_force_tiny():
    A = np.array([[1.0, 2.0, 3.0], [-1.0, 0.5, 0.0]])
    B = np.array([[1.0, 0.0, 0.0], [0.0, 1.0, 0.0], [1.0, 1.0, 1.0], [2.0, -1.0, 0.5]])
    C = O.matmul_nt(A, B)
    expect = [[1, 2, 6, 1.5], [-1, 0.5, -0.5, -2.5]]
    assert np.array_equal(C, np.array(expect))


def test_swiglu_closed_forms_and_pairing():
    I = 4
    v = np.zeros((3, 2 * I))
    v[0, :I] = [0.0, 1.0, -1.0, 30.0]      # gate
    v[0, I:] = [5.0, 2.0, 2.0, 0.5]        # up
    v[1, :I] = -40.0
    v[1, I:] = 1.0
    v[2, :] = np.arange(1, 2 * I + 1)
    h = O.swiglu(v)
    silu1 = 1.0 / (1.0 + math.exp(-1.0))
    assert h[0, 0] == 0.0
    assert np.isclose(h[0, 1], 2 * silu1, rtol=1e-7)
    assert np.isclose(h[0, 2], 2 * (-1.0 + silu1), rtol=1e-6)   # silu(-1) = silu(1) - 1
    assert np.isclose(h[0, 3], 15.0, rtol=1e-7)
    assert np.all(np.abs(h[1]) < 1e-15)
    # h[:, i] depends on columns i and I+i only
    base = O.swiglu(v[2:3])
    for col in range(2 * I):
        vv = v[2:3].copy()
        vv[0, col] += 1.0
        changed = np.nonzero(O.swiglu(vv)[0] != base[0])[0]
        assert list(changed) == [col % I]


def test_combine_brute_force():
    rng = np.random.default_rng(3)
    T, k, K = 7, 3, 5
    M = T * k
    out = rng.normal(size=(M, K))
    perm = rng.permutation(M).astype(np.int32)
    w = rng.random((T, k))
    y = O.combine(out, w, perm)
    for t in range(T):
        ref = sum(w[t, j] * out[perm[t * k + j]] for j in range(k))
        assert np.allclose(y[t], ref, rtol=0, atol=1e-15)


def _tiny(seed=0):
    cfg = W.CONFIGS["tiny"]
    inp = W.moe_inputs(cfg, seed)
    return cfg, W.bf16_bits(inp["x"]), inp["logits"].numpy(), W.bf16_bits(inp["w1"]), W.bf16_bits(inp["w2"])


def test_moe_forward_token_permutation_invariance():
    cfg, x, logits, w1, w2 = _tiny()
    r = O.moe_forward(x, logits, lambda e: w1[e], lambda e: w2[e], cfg.k, cfg.gs_h)
    perm = np.random.default_rng(4).permutation(cfg.T)
    rp = O.moe_forward(x[perm], logits[perm], lambda e: w1[e], lambda e: w2[e], cfg.k, cfg.gs_h)
    assert np.array_equal(rp["y"], r["y"][perm])


def test_moe_forward_expert_relabel_invariance():
    cfg, x, logits, w1, w2 = _tiny()
    r = O.moe_forward(x, logits, lambda e: w1[e], lambda e: w2[e], cfg.k, cfg.gs_h)
    p = np.random.default_rng(5).permutation(cfg.E)      # new label of expert e is p[e]
    inv = np.argsort(p)
    logits2 = np.empty_like(logits)
    logits2[:, p] = logits
    r2 = O.moe_forward(x, logits2, lambda e: w1[inv[e]], lambda e: w2[inv[e]], cfg.k, cfg.gs_h)
    assert np.array_equal(r2["y"], r["y"])


def test_moe_forward_single_expert_is_a_two_layer_mlp():
    """E=1, k=1: routing weight 1, so y = W2 . swiglu(W1 . x) on dequantized operands."""
    rng = np.random.default_rng(6)
    T, K, I = 5, 64, 32
    x = bf16_bits_np(rng.normal(0, 1, (T, K)))
    w1 = bf16_bits_np(rng.normal(0, 0.1, (2 * I, K)))
    w2 = bf16_bits_np(rng.normal(0, 0.1, (K, I)))
    logits = np.zeros((T, 1), np.float32)
    gs_h = np.float32(500.0)
    r = O.moe_forward(x, logits, lambda e: w1, lambda e: w2, 1, gs_h)
    gx = O.global_scale(O.amax_bf16(x))
    xd = O.dequantize_f64(*O.quantize_bf16(x, gx), gx)
    c1, s1, g1 = O.quantize_expert(w1)
    c2, s2, g2 = O.quantize_expert(w2)
    v = xd @ O.dequantize_f64(c1, s1, g1).T
    g, u = v[:, :I], v[:, I:]
    h = (g / (1 + np.exp(-g)) * u).astype(np.float32)
    hd = O.dequantize_f64(*O.quantize_f32(h, gs_h), gs_h)
    y = hd @ O.dequantize_f64(c2, s2, g2).T
    assert np.allclose(r["y"], y, rtol=1e-12, atol=1e-14)


def test_moe_forward_is_the_routing_weighted_sum_of_expert_mlps():
    """E=3, k=2: y[t] = sum_j w[t, j] * MLP_{ids[t, j]}(x[t]), with the top-2 and
    its softmax from torch and each expert's two-layer MLP composed in numpy on
    dequantized operands."""
    rng = np.random.default_rng(8)
    T, K, I, E, k = 6, 64, 32, 3, 2
    x = bf16_bits_np(rng.normal(0, 1, (T, K)))
    w1 = [bf16_bits_np(rng.normal(0, 0.1, (2 * I, K))) for _ in range(E)]
    w2 = [bf16_bits_np(rng.normal(0, 0.1, (K, I))) for _ in range(E)]
    logits = rng.normal(0, 1, (T, E)).astype(np.float32)
    gs_h = np.float32(400.0)
    r = O.moe_forward(x, logits, lambda e: w1[e], lambda e: w2[e], k, gs_h)
    top = torch.topk(torch.from_numpy(logits).double(), k, dim=1)
    ids = top.indices.numpy()
    wts = torch.softmax(top.values, dim=1).numpy()
    gx = O.global_scale(O.amax_bf16(x))
    xd = O.dequantize_f64(*O.quantize_bf16(x, gx), gx)

    def mlp(e, xrow):
        c1, s1, g1 = O.quantize_expert(w1[e])
        c2, s2, g2 = O.quantize_expert(w2[e])
        v = xrow[None, :] @ O.dequantize_f64(c1, s1, g1).T
        g, u = v[:, :I], v[:, I:]
        h = (g / (1 + np.exp(-g)) * u).astype(np.float32)
        hd = O.dequantize_f64(*O.quantize_f32(h, gs_h), gs_h)
        return (hd @ O.dequantize_f64(c2, s2, g2).T)[0]

    assert len({tuple(sorted(r)) for r in ids}) > 1       # more than one expert pair in use
    for t in range(T):
        y = sum(wts[t, j] * mlp(int(ids[t, j]), xd[t]) for j in range(k))
        assert np.allclose(r["y"][t], y, rtol=1e-12, atol=1e-14), t


def bf16_bits_np(a):
    return W.bf16_bits(torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16))


def test_moe_forward_given_gs_x():
    """A pre-computed gs_x equal to the computed one changes nothing; another
    one changes the quantized activations exactly as quantizing x with it."""
    cfg, x, logits, w1, w2 = _tiny()
    r = O.moe_forward(x, logits, lambda e: w1[e], lambda e: w2[e], cfg.k, cfg.gs_h)
    r2 = O.moe_forward(x, logits, lambda e: w1[e], lambda e: w2[e], cfg.k, cfg.gs_h, gs_x=r["gs_x"])
    assert np.array_equal(r2["y"], r["y"])
    g = np.float32(r["gs_x"] * 0.5)
    r3 = O.moe_forward(x, logits, lambda e: w1[e], lambda e: w2[e], cfg.k, cfg.gs_h, gs_x=g)
    c, s = O.quantize_bf16(x, g)
    assert r3["gs_x"] == g and np.array_equal(r3["x_codes"], c) and np.array_equal(r3["x_sf"], s)
    assert not np.array_equal(r3["x_sf"], r["x_sf"])
