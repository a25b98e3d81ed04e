"""NVFP4 MoE oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow CPU statement of the NVFP4 Mixture-of-Experts expert forward
described by the "NVFP4 MegaMoE Kernel" README (sections "What We Have",
"MoE Runner", "Correctness Bugs Fixed", "Fused SwiGLU - How It Works") and
CURRENT_BUG.md ("What Works": activation global scale recomputed per call).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA path:
arithmetic lives in ``nvfp4_oracle.cpp`` (plain C++, fp64 GEMMs) and this file
only marshals numpy arrays and strings the steps together in the pages' order.

BF16 tensors are passed as ``numpy.uint16`` bit patterns. Scale bytes are in
plain row-major order: ``sf[r, c // 16]`` is the E4M3 scale of elements
``16*(c//16) .. 16*(c//16)+15`` of row ``r``; codes are ``codes[r, c // 2]``
with element ``c`` in the low nibble when ``c`` is even.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        sig = {
            "orc_e2m1_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e2m1_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "orc_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "orc_global_scale": (ctypes.c_float, [ctypes.c_float]),
            "orc_amax_bf16": (ctypes.c_float, [_u16p, _i64, _i64, _i64]),
            "orc_amax_f32": (ctypes.c_float, [_f32p, _i64]),
            "orc_quantize_bf16": (None, [_u16p, _i64, _i64, _i64, ctypes.c_float, _u8p, _u8p]),
            "orc_quantize_f32": (None, [_f32p, _i64, _i64, ctypes.c_float, _u8p, _u8p]),
            "orc_dequantize_f32": (None, [_u8p, _u8p, _i64, _i64, ctypes.c_float, _f32p]),
            "orc_dequantize_f64": (None, [_u8p, _u8p, _i64, _i64, ctypes.c_float, _f64p]),
            "orc_interleave_rows": (None, [_u8p, _u8p, _i64, _i64, _i64]),
            "orc_deinterleave_rows": (None, [_u8p, _u8p, _i64, _i64, _i64]),
            "orc_route_topk": (None, [_f32p, _i64, ctypes.c_int, ctypes.c_int, _i32p, _f64p]),
            "orc_permute": (None, [_i32p, _i64, ctypes.c_int, ctypes.c_int, _i32p, _i32p, _i32p]),
            "orc_set_threads": (None, [ctypes.c_int]),
            "orc_get_threads": (ctypes.c_int, []),
            "orc_matmul_nt": (None, [_f64p, _f64p, _i64, _i64, _i64, _f64p]),
            "orc_grouped_gemm": (None, [_u8p, _u8p, ctypes.c_float, _u8p, _u8p, _f32p, _i32p,
                                        _i64, _i64, ctypes.c_int, _f64p]),
            "orc_swiglu": (None, [_f64p, _i64, _i64, _f32p]),
            "orc_combine": (None, [_f64p, _i64, _f64p, _i32p, _i64, ctypes.c_int, _f64p]),
            "orc_rmsnorm_rope": (None, [_u16p, _i64, _i64, _i64, _f64p, ctypes.c_double, _i64, _i32p,
                                        _f64p, _f64p, _f64p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ------------------------------------------------------------------ formats

def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(int(code))


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(float(v))


def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code))


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(float(v))


def global_scale(amax: float) -> np.float32:
    return np.float32(lib().orc_global_scale(float(np.float32(amax))))


def amax_bf16(x: np.ndarray) -> np.float32:
    x = _c(x, np.uint16)
    x2 = x.reshape(-1, x.shape[-1]) if x.ndim != 2 else x
    return np.float32(lib().orc_amax_bf16(x2, x2.shape[0], x2.shape[1], x2.shape[1]))


def amax_f32(x: np.ndarray) -> np.float32:
    x = _c(x, np.float32).reshape(-1)
    return np.float32(lib().orc_amax_f32(x, x.size))


def quantize_bf16(x: np.ndarray, gs):
    """Block-quantize (rows, cols) BF16 bits with global scale gs -> (codes, sf)."""
    x = _c(x, np.uint16)
    rows, cols = x.shape
    assert cols % 16 == 0
    codes = np.zeros((rows, cols // 2), np.uint8)
    sf = np.zeros((rows, cols // 16), np.uint8)
    lib().orc_quantize_bf16(x, rows, cols, cols, float(np.float32(gs)), codes, sf)
    return codes, sf


def quantize_f32(x: np.ndarray, gs):
    x = _c(x, np.float32)
    rows, cols = x.shape
    assert cols % 16 == 0
    codes = np.zeros((rows, cols // 2), np.uint8)
    sf = np.zeros((rows, cols // 16), np.uint8)
    lib().orc_quantize_f32(x, rows, cols, float(np.float32(gs)), codes, sf)
    return codes, sf


def dequantize_f32(codes, sf, gs) -> np.ndarray:
    codes = _c(codes, np.uint8)
    sf = _c(sf, np.uint8)
    rows, half = codes.shape
    out = np.zeros((rows, half * 2), np.float32)
    lib().orc_dequantize_f32(codes, sf, rows, half * 2, float(np.float32(gs)), out)
    return out


def dequantize_f64(codes, sf, gs) -> np.ndarray:
    codes = _c(codes, np.uint8)
    sf = _c(sf, np.uint8)
    rows, half = codes.shape
    out = np.zeros((rows, half * 2), np.float64)
    lib().orc_dequantize_f64(codes, sf, rows, half * 2, float(np.float32(gs)), out)
    return out


# ------------------------------------------------------------------ layout

def interleave_rows(a: np.ndarray, g: int = 8) -> np.ndarray:
    """(2I, ...) rows [gate | up] -> gate/up interleaved at granularity g."""
    a = np.ascontiguousarray(a)
    two_i = a.shape[0]
    flat = a.reshape(two_i, -1).view(np.uint8)
    out = np.empty_like(flat)
    lib().orc_interleave_rows(np.ascontiguousarray(flat), out, two_i, flat.shape[1], g)
    return out.view(a.dtype).reshape(a.shape)


def deinterleave_rows(a: np.ndarray, g: int = 8) -> np.ndarray:
    a = np.ascontiguousarray(a)
    two_i = a.shape[0]
    flat = a.reshape(two_i, -1).view(np.uint8)
    out = np.empty_like(flat)
    lib().orc_deinterleave_rows(np.ascontiguousarray(flat), out, two_i, flat.shape[1], g)
    return out.view(a.dtype).reshape(a.shape)


# ------------------------------------------------------------------ routing

def route_topk(logits: np.ndarray, k: int):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    lib().orc_route_topk(logits, T, E, k, ids, w)
    return ids, w


def permute(ids: np.ndarray, E: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    offsets = np.zeros(E + 1, np.int32)
    p2f = np.zeros(T * k, np.int32)
    f2p = np.zeros(T * k, np.int32)
    lib().orc_permute(ids, T, k, E, offsets, p2f, f2p)
    return offsets, p2f, f2p


# ------------------------------------------------------------------ GEMM

def set_threads(n: int):
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return lib().orc_get_threads()


def matmul_nt(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    A = _c(A, np.float64)
    B = _c(B, np.float64)
    M, K = A.shape
    N = B.shape[0]
    C = np.zeros((M, N), np.float64)
    lib().orc_matmul_nt(A, B, M, N, K, C)
    return C


def grouped_gemm(a_codes, a_sf, gs_a, b_codes, b_sf, gs_b, offsets) -> np.ndarray:
    """C (M, N) fp64 of the grouped GEMM; A compact rows, B (E, N, K) NVFP4."""
    a_codes = _c(a_codes, np.uint8)
    a_sf = _c(a_sf, np.uint8)
    b_codes = _c(b_codes, np.uint8)
    b_sf = _c(b_sf, np.uint8)
    gs_b = _c(gs_b, np.float32).reshape(-1)
    offsets = _c(offsets, np.int32)
    E, N, khalf = b_codes.shape
    K = khalf * 2
    M = int(offsets[-1])
    C = np.zeros((M, N), np.float64)
    lib().orc_grouped_gemm(a_codes, a_sf, float(np.float32(gs_a)), b_codes.reshape(-1),
                           b_sf.reshape(-1), gs_b, offsets, N, K, E, C)
    return C


def swiglu(v: np.ndarray) -> np.ndarray:
    """h = silu(v[:, :I]) * v[:, I:], rounded once to f32."""
    v = _c(v, np.float64)
    M, two_i = v.shape
    h = np.zeros((M, two_i // 2), np.float32)
    lib().orc_swiglu(v, M, two_i // 2, h)
    return h


def combine(out: np.ndarray, w: np.ndarray, flat_to_perm: np.ndarray) -> np.ndarray:
    out = _c(out, np.float64)
    w = _c(w, np.float64)
    T, k = w.shape
    K = out.shape[1]
    y = np.zeros((T, K), np.float64)
    lib().orc_combine(out, K, w, _c(flat_to_perm, np.int32), T, k, y)
    return y


def rmsnorm_rope(x, gamma, eps, rope_dims, positions, cos_t, sin_t) -> np.ndarray:
    """README "THE PLAN", item 3 ("Q norm -> RoPE -> NVFP4 quant", one pass),
    the norm and rotation steps, in fp64: y = x / sqrt(mean(x^2) + eps) * gamma
    per row, then adjacent pairs of the last ``rope_dims`` elements rotated by
    the angle whose cosine / sine are ``cos_t[pos, j]`` / ``sin_t[pos, j]``.
    x: (rows, D) BF16 bits; gamma (D,); positions (rows,) int; tables
    (max_pos, rope_dims/2). Returns (rows, D) fp64."""
    x = _c(x, np.uint16)
    rows, D = x.shape
    y = np.zeros((rows, D), np.float64)
    half = rope_dims // 2
    ct = _c(np.asarray(cos_t, np.float64).reshape(-1, max(half, 1)), np.float64)
    st = _c(np.asarray(sin_t, np.float64).reshape(-1, max(half, 1)), np.float64)
    lib().orc_rmsnorm_rope(x, rows, D, D, _c(gamma, np.float64), float(eps), rope_dims,
                           _c(positions, np.int32), ct, st, y)
    return y


# ------------------------------------------------------------------ composites

def quantize_expert(w_bf16: np.ndarray):
    """One expert matrix (N, K) BF16 -> (codes, sf, gs); gs from the matrix amax
    (README "What We Have": global scales per expert)."""
    gs = global_scale(amax_bf16(w_bf16))
    codes, sf = quantize_bf16(w_bf16, gs)
    return codes, sf, gs


def moe_forward(x, logits, get_w1, get_w2, k, gs_h, tokens=None, keep=False, experts=None,
                qweights=None, gs_x=None):
    """README "MoE Runner", steps 1-6, for the tokens listed in ``tokens``.

    x: (T, K) BF16 bits; logits: (T, E) f32; get_w1(e) -> (2I, K) BF16 bits with
    rows [gate | up] (not interleaved); get_w2(e) -> (K, I) BF16 bits; gs_h: the
    pre-computed global scale of the intermediate activation (README "Bridge
    Layer": quantize_activation_nvfp4 with pre-computed gs).

    Routing, permutation and gs_x always cover all T tokens; the expert work is
    done for the listed tokens only, one expert at a time (so only one expert's
    dequantized weights are held in memory). ``experts`` (optional) restricts
    the expert work to the routed rows of those experts, so y then holds only
    their share of the weighted sum. ``qweights`` (optional) maps an expert to
    its already-quantized (c1, s1, g1, c2, s2, g2), skipping the offline weight
    quantization. ``gs_x`` (optional) is a pre-computed activation global scale
    (README "Bridge Layer": quantize_activation_nvfp4 with pre-computed gs,
    the CUDA-graph-safe path); by default gs_x = 2688 / amax|x| over all T
    tokens. Returns a dict with the routing, the permutation, gs_x,
    y (len(tokens), K) fp64, and per-(token, j) intermediates when ``keep``.
    """
    T, K = x.shape
    E = logits.shape[1]
    ids, w = route_topk(logits, k)
    offsets, p2f, f2p = permute(ids, E)
    amax_x = amax_bf16(x)
    gs_x = global_scale(amax_x) if gs_x is None else np.float32(gs_x)
    tokens = list(range(T)) if tokens is None else [int(t) for t in tokens]
    xc, xs = quantize_bf16(np.ascontiguousarray(x[tokens]), gs_x)
    xd = dequantize_f64(xc, xs, gs_x)
    by_expert = {}
    for ti, t in enumerate(tokens):
        for j in range(k):
            if experts is None or int(ids[t, j]) in experts:
                by_expert.setdefault(int(ids[t, j]), []).append((ti, j))
    outs = np.zeros((len(tokens), k, K), np.float64)
    inter = {}
    gs_w = {}
    for e in sorted(by_expert):
        if qweights is not None:
            c1, s1, g1, c2, s2, g2 = qweights(e)
        else:
            c1, s1, g1 = quantize_expert(get_w1(e))
            c2, s2, g2 = quantize_expert(get_w2(e))
        gs_w[e] = (g1, g2)
        pairs = by_expert[e]
        a = xd[[ti for ti, _ in pairs]]
        v = matmul_nt(a, dequantize_f64(c1, s1, g1))          # (n, 2I): [gate | up]
        h = swiglu(v)                                          # (n, I) f32
        hc, hs = quantize_f32(h, gs_h)
        o = matmul_nt(dequantize_f64(hc, hs, gs_h), dequantize_f64(c2, s2, g2))
        for r, (ti, j) in enumerate(pairs):
            outs[ti, j] = o[r]
            if keep:
                inter[(tokens[ti], j)] = dict(v=v[r], h=h[r], hc=hc[r], hs=hs[r], o=o[r])
    # step 6: weighted sum over j, in j order, fp64 (slot (ti, j) is row ti*k + j of outs)
    n = len(tokens)
    y = combine(outs.reshape(n * k, K), w[tokens], np.arange(n * k, dtype=np.int32))
    return dict(ids=ids, w=w, offsets=offsets, perm_to_flat=p2f, flat_to_perm=f2p,
                amax_x=amax_x, gs_x=gs_x, tokens=tokens, x_codes=xc, x_sf=xs, y=y,
                inter=inter, gs_w=gs_w)
