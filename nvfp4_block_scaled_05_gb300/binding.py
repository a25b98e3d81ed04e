"""Thin Python binding of libnvfp4moe.so (the C ABI in include/nvfp4moe.h).

Every function here has the name of the C entry point it calls and only
marshals arguments: it allocates outputs with torch (device memory is the one
thing torch is used for), passes raw pointers and torch's current stream, and
raises on a non-zero status. All arithmetic runs in the library's kernels; if
the library cannot be loaded, every call fails loudly.
"""
import ctypes
import os

import torch

from . import build as _build

NVFP4_SF_ROWMAJOR = 0
NVFP4_SF_TILED = 1          # weight (B) operand scales of the GEMMs
NVFP4_SF_TILED_ROWS = 2     # activation (A) operand scales of the GEMMs
# include/nvfp4moe.h NVFP4MOE_FRONT_FUSED_QUANTIZE_MAX_ROWS: routed rows up to
# which the fused dispatch quantizes inside its cooperative kernel
FRONT_FUSED_QUANTIZE_MAX_ROWS = 32768

_c_void_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_size = ctypes.c_size_t

_SIGS = {
    "nvfp4moe_status_string": (ctypes.c_char_p, [_int]),
    "nvfp4_sf_bytes": (_size, [_i64, _i64, _int]),
    "nvfp4moe_padded_rows": (_i64, [_i64, _int]),
    "nvfp4moe_interleave_row_map": (_int, [_i64, _c_void_p]),
    "nvfp4_sf_to_tiled": (_int, [_c_void_p, _i64, _i64, _i64, _int, _c_void_p, _c_void_p]),
    "nvfp4_sf_from_tiled": (_int, [_c_void_p, _i64, _i64, _i64, _int, _c_void_p, _c_void_p]),
    "nvfp4_interleave_gate_up": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _int, _int, _c_void_p,
                                        _c_void_p, _c_void_p]),
    "nvfp4_quantize_workspace_size": (_size, []),
    "nvfp4_quantize": (_int, [_c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p, _c_void_p,
                              _c_void_p, _c_void_p, _int, _c_void_p, _size, _c_void_p]),
    "moe_route_topk": (_int, [_c_void_p, _i64, _int, _int, _c_void_p, _c_void_p, _c_void_p]),
    "moe_permute_workspace_size": (_size, [_i64, _int, _int]),
    "moe_permute": (_int, [_c_void_p, _i64, _int, _int, _c_void_p, _c_void_p, _c_void_p,
                           _c_void_p, _size, _c_void_p]),
    "moe_permute_static_ws": (_int, [_c_void_p, _i64, _int, _int, _c_void_p, _c_void_p, _c_void_p,
                                     _c_void_p]),
    "moe_quantize_dispatch_workspace_size": (_size, [_int]),
    "moe_quantize_dispatch": (_int, [_c_void_p, _i64, _i64, _i64, _int, _int, _c_void_p,
                                     _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                     _c_void_p, _i64, _c_void_p, _size, _c_void_p]),
    "nvfp4_grouped_gemm": (_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p, _c_void_p,
                                  _c_void_p, _c_void_p, _int, _i64, _i64, _c_void_p, _i64,
                                  _c_void_p]),
    "nvfp4_grouped_gemm_swiglu": (_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p,
                                         _c_void_p, _c_void_p, _c_void_p, _int, _i64, _i64,
                                         _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "moe_combine": (_int, [_c_void_p, _i64, _c_void_p, _c_void_p, _i64, _int, _i64, _c_void_p,
                           _i64, _c_void_p]),
    "moe_forward_workspace_size": (_size, [_i64, _i64, _i64, _int, _int]),
    "moe_forward_workspace_layout": (_int, [_i64, _i64, _i64, _int, _int, _c_void_p]),
    "moe_forward": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _int, _int, _c_void_p,
                           _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                           _c_void_p, _c_void_p, _size, _c_void_p]),
    "moe_forward_static": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _int, _int, _c_void_p,
                                  _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                  _c_void_p, _c_void_p, _c_void_p, _size, _c_void_p]),
    "moe_dispatch_static_workspace_size": (_size, [_i64, _int]),
    "moe_dispatch_static": (_int, [_c_void_p, _i64, _c_void_p, _i64, _i64, _int, _int, _c_void_p, _c_void_p,
                                   _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i64,
                                   _c_void_p, _size, _c_void_p]),
    "moe_dispatch_supported": (_int, [_i64, _int, _int]),
    "moe_forward_uses_fused_dispatch": (_int, [_i64, _int, _int]),
    "moe_dispatch": (_int, [_c_void_p, _i64, _c_void_p, _i64, _i64, _int, _int, _c_void_p, _c_void_p,
                            _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i64,
                            _c_void_p, _size, _c_void_p]),
    "nvfp4_rmsnorm_rope_quantize": (_int, [_c_void_p, _i64, _i64, _i64, _c_void_p, ctypes.c_float, _i64,
                                           _c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p, _c_void_p,
                                           _c_void_p, _int, _c_void_p, _c_void_p]),
    "nvfp4_linear_workspace_size": (_size, []),
    "nvfp4_linear": (_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _i64, _c_void_p, _c_void_p, _c_void_p,
                            _i64, _i64, _c_void_p, _i64, _c_void_p, _size, _c_void_p]),
    "nvfp4moe_last_device_status": (_int, [_c_void_p]),
    "nvfp4moe_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "nvfp4moe_set_test_stall": (None, [_int]),
    "nvfp4moe_num_sms": (_int, []),
    "nvfp4moe_set_gemm_mode": (_int, [_int]),
}

_lib = None


class NVFP4Error(RuntimeError):
    pass


def lib():
    """Load (building first if stale) the in-tree libnvfp4moe.so."""
    global _lib
    if _lib is None:
        path = _build.LIB if os.path.exists(_build.LIB) and not _build.stale() else _build.build()
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(status, what):
    if status != 0:
        msg = lib().nvfp4moe_status_string(status).decode()
        raise NVFP4Error("%s failed: %s (%d)" % (what, msg, status))


def _dev(t, name):
    if not (isinstance(t, torch.Tensor) and t.is_cuda):
        raise NVFP4Error("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise NVFP4Error("%s must be contiguous" % name)
    return t


# ------------------------------------------------------------------ sizes

def nvfp4_sf_bytes(rows, cols, sf_layout=NVFP4_SF_TILED):
    return int(lib().nvfp4_sf_bytes(rows, cols, sf_layout))


def nvfp4moe_padded_rows(M, E):
    return int(lib().nvfp4moe_padded_rows(M, E))


def nvfp4moe_interleave_row_map(two_i):
    m = (ctypes.c_int32 * two_i)()
    _check(lib().nvfp4moe_interleave_row_map(two_i, ctypes.cast(m, ctypes.c_void_p)), "interleave_row_map")
    return torch.tensor(list(m), dtype=torch.int32)


def nvfp4_sf_to_tiled(sf, rows, cols, sf_layout=NVFP4_SF_TILED, out=None):
    """Row-major scales (batch, rows, cols//16) or (rows, cols//16) -> the tiled
    layout, batch * nvfp4_sf_bytes(rows, cols, sf_layout) bytes (README "Bridge
    Layer": assemble_scales_2d_side / _3d_side)."""
    _dev(sf, "sf")
    batch = sf.numel() // max(1, rows * (cols // 16))
    per = nvfp4_sf_bytes(rows, cols, sf_layout)
    if out is None:
        out = torch.empty(batch * per, dtype=torch.uint8, device=sf.device)
    _check(lib().nvfp4_sf_to_tiled(_ptr(sf), batch, rows, cols, sf_layout, _ptr(out), _stream()),
           "nvfp4_sf_to_tiled")
    return out


def nvfp4_sf_from_tiled(sf_tiled, batch, rows, cols, sf_layout=NVFP4_SF_TILED, out=None):
    """Tiled scales of `batch` (rows x cols) matrices -> (batch, rows, cols//16) row-major."""
    _dev(sf_tiled, "sf_tiled")
    if out is None:
        out = torch.empty((batch, rows, cols // 16), dtype=torch.uint8, device=sf_tiled.device)
    _check(lib().nvfp4_sf_from_tiled(_ptr(sf_tiled), batch, rows, cols, sf_layout, _ptr(out), _stream()),
           "nvfp4_sf_from_tiled")
    return out


def nvfp4_interleave_gate_up(codes, sf, two_i, K, sf_layout=NVFP4_SF_ROWMAJOR, inverse=False):
    """W1 rows [gate | up] <-> interleaved at granularity 8 (README "Bridge
    Layer": interleave_l1_weights / deinterleave_l1_weights). codes: (batch,
    two_i, K//2) bytes or None; sf: batch scale matrices in sf_layout or None.
    Returns (codes_out, sf_out)."""
    if codes is not None:
        _dev(codes, "codes")
    if sf is not None:
        _dev(sf, "sf")
    batch = (codes.numel() // (two_i * (K // 2))) if codes is not None else \
        (sf.numel() // nvfp4_sf_bytes(two_i, K, sf_layout))
    co = torch.empty_like(codes) if codes is not None else None
    so = torch.empty_like(sf) if sf is not None else None
    _check(lib().nvfp4_interleave_gate_up(_ptr(codes), _ptr(sf), batch, two_i, K, sf_layout, int(bool(inverse)),
                                          _ptr(co), _ptr(so), _stream()), "nvfp4_interleave_gate_up")
    return co, so


def nvfp4moe_set_gemm_mode(mode):
    """0: one CTA per tile (default); 1: the 2-SM pair kernel where N % 256 == 0."""
    _check(lib().nvfp4moe_set_gemm_mode(int(mode)), "nvfp4moe_set_gemm_mode")


def nvfp4moe_num_sms():
    return int(lib().nvfp4moe_num_sms())


def nvfp4moe_last_device_status():
    return int(lib().nvfp4moe_last_device_status(_stream()))


def nvfp4moe_set_wait_limit_ns(ns):
    lib().nvfp4moe_set_wait_limit_ns(int(ns))


def nvfp4moe_set_test_stall(on):
    lib().nvfp4moe_set_test_stall(1 if on else 0)


def moe_forward_workspace_size(T, K, I, E, k):
    return int(lib().moe_forward_workspace_size(T, K, I, E, k))


def moe_forward_workspace_layout(T, K, I, E, k):
    offs = (ctypes.c_int64 * 12)()
    _check(lib().moe_forward_workspace_layout(T, K, I, E, k, ctypes.cast(offs, ctypes.c_void_p)),
           "moe_forward_workspace_layout")
    names = ["topk_ids", "topk_w", "offsets", "perm_to_flat", "flat_to_perm", "gs_x", "a_codes",
             "a_sf", "h_codes", "h_sf", "out", "a_rows"]
    return dict(zip(names, list(offs)))


# ------------------------------------------------------------------ ops

def nvfp4_quantize(x, gs=None, row_src=None, sf_layout=NVFP4_SF_TILED, rows=None,
                   codes=None, sf=None, gs_out=None):
    """BF16 (rows, cols) -> (codes, sf, gs). gs: device f32 tensor or None (computed)."""
    _dev(x, "x")
    assert x.dtype == torch.bfloat16 and x.dim() == 2
    cols = x.shape[1]
    if rows is None:
        rows = row_src.numel() if row_src is not None else x.shape[0]
    dev = x.device
    if codes is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
    if sf is None:
        sf = torch.empty(nvfp4_sf_bytes(rows, cols, sf_layout), dtype=torch.uint8, device=dev)
    if gs_out is None:
        gs_out = torch.empty(1, dtype=torch.float32, device=dev)
    ws = None
    ws_bytes = 0
    if gs is None:
        ws_bytes = int(lib().nvfp4_quantize_workspace_size())
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _check(lib().nvfp4_quantize(_ptr(x), rows, cols, x.stride(0), _ptr(gs), _ptr(gs_out),
                                _ptr(row_src), _ptr(codes), _ptr(sf), sf_layout, _ptr(ws), ws_bytes,
                                _stream()), "nvfp4_quantize")
    return codes, sf, gs_out


def moe_route_topk(logits, k):
    _dev(logits, "logits")
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check(lib().moe_route_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _stream()), "moe_route_topk")
    return ids, w


def moe_permute(topk_ids, E):
    _dev(topk_ids, "topk_ids")
    T, k = topk_ids.shape
    dev = topk_ids.device
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    p2f = torch.empty(T * k, dtype=torch.int32, device=dev)
    f2p = torch.empty(T * k, dtype=torch.int32, device=dev)
    nb = int(lib().moe_permute_workspace_size(T, k, E))
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)
    _check(lib().moe_permute(_ptr(topk_ids), T, k, E, _ptr(offsets), _ptr(p2f), _ptr(f2p), _ptr(ws),
                             nb, _stream()), "moe_permute")
    return offsets, p2f, f2p


def moe_permute_static_ws(topk_ids, E):
    """moe_permute using the library's fixed scratch array: no workspace is
    allocated or passed (for callers that cannot allocate at the call)."""
    _dev(topk_ids, "topk_ids")
    T, k = topk_ids.shape
    dev = topk_ids.device
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    p2f = torch.empty(T * k, dtype=torch.int32, device=dev)
    f2p = torch.empty(T * k, dtype=torch.int32, device=dev)
    _check(lib().moe_permute_static_ws(_ptr(topk_ids), T, k, E, _ptr(offsets), _ptr(p2f), _ptr(f2p),
                                       _stream()), "moe_permute_static_ws")
    return offsets, p2f, f2p


def moe_quantize_dispatch(x, topk_ids, offsets, flat_to_perm, E, gs=None, a_rows=None):
    _dev(x, "x")
    T, K = x.shape
    k = topk_ids.shape[1]
    dev = x.device
    if a_rows is None:
        a_rows = nvfp4moe_padded_rows(T * k, E)
    a_codes = torch.zeros((a_rows, K // 2), dtype=torch.uint8, device=dev)
    a_sf = torch.zeros(nvfp4_sf_bytes(a_rows, K, NVFP4_SF_TILED_ROWS), dtype=torch.uint8, device=dev)
    gs_out = torch.empty(1, dtype=torch.float32, device=dev)
    nb = int(lib().moe_quantize_dispatch_workspace_size(E))
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    _check(lib().moe_quantize_dispatch(_ptr(x), T, K, x.stride(0), k, E, _ptr(topk_ids), _ptr(offsets),
                                       _ptr(flat_to_perm), _ptr(gs), _ptr(gs_out), _ptr(a_codes),
                                       _ptr(a_sf), a_rows, _ptr(ws), nb, _stream()),
           "moe_quantize_dispatch")
    return a_codes, a_sf, gs_out


def nvfp4_grouped_gemm(a_codes, a_sf, gs_a, b_codes, b_sf, gs_b, offsets, out=None):
    """A grouped-padded (a_rows, K/2); B (E, N, K/2) -> C (M, N) BF16, compact rows."""
    E, N, khalf = b_codes.shape
    K = khalf * 2
    M = None
    if out is None:
        M = int(offsets[-1].item())
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a_codes.device)
    _check(lib().nvfp4_grouped_gemm(_ptr(a_codes), _ptr(a_sf), _ptr(gs_a), a_codes.shape[0],
                                    _ptr(b_codes), _ptr(b_sf), _ptr(gs_b), _ptr(offsets), E, N, K,
                                    _ptr(out), out.stride(0), _stream()), "nvfp4_grouped_gemm")
    return out


def nvfp4_rmsnorm_rope_quantize(x, gamma, eps, rope_dims, positions, cos_tab, sin_tab, gs,
                                sf_layout=NVFP4_SF_TILED, y_out=None, codes=None, sf=None):
    """(rows, D) BF16 -> RMS norm -> RoPE on the last rope_dims -> NVFP4 (codes, sf)."""
    _dev(x, "x")
    assert x.dtype == torch.bfloat16 and x.dim() == 2
    rows, D = x.shape
    dev = x.device
    if codes is None:
        codes = torch.empty((rows, D // 2), dtype=torch.uint8, device=dev)
    if sf is None:
        sf = torch.empty(nvfp4_sf_bytes(rows, D, sf_layout), dtype=torch.uint8, device=dev)
    max_pos = cos_tab.shape[0] if cos_tab is not None else 0
    _check(lib().nvfp4_rmsnorm_rope_quantize(_ptr(x), rows, D, x.stride(0), _ptr(gamma), float(eps), rope_dims,
                                             _ptr(positions), _ptr(cos_tab), _ptr(sin_tab), max_pos, _ptr(gs),
                                             _ptr(codes), _ptr(sf), sf_layout, _ptr(y_out), _stream()),
           "nvfp4_rmsnorm_rope_quantize")
    return codes, sf


def nvfp4_linear(a_codes, a_sf, gs_a, M, w_codes, w_sf, gs_w, out=None, ws=None):
    """A (a_rows >= 128*ceil(M/128), K/2) x W (N, K/2) -> C (M, N) BF16."""
    N, khalf = w_codes.shape
    K = khalf * 2
    dev = a_codes.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = torch.empty(int(lib().nvfp4_linear_workspace_size()), dtype=torch.uint8, device=dev)
    _check(lib().nvfp4_linear(_ptr(a_codes), _ptr(a_sf), _ptr(gs_a), M, a_codes.shape[0], _ptr(w_codes),
                              _ptr(w_sf), _ptr(gs_w), N, K, _ptr(out), out.stride(0), _ptr(ws), ws.numel(),
                              _stream()), "nvfp4_linear")
    return out


def nvfp4_grouped_gemm_swiglu(a_codes, a_sf, gs_a, w1_codes, w1_sf, gs_w1, offsets, gs_h,
                              h_codes=None, h_sf=None):
    E, two_i, khalf = w1_codes.shape
    K, I = khalf * 2, two_i // 2
    a_rows = a_codes.shape[0]
    dev = a_codes.device
    if h_codes is None:
        h_codes = torch.zeros((a_rows, I // 2), dtype=torch.uint8, device=dev)
    if h_sf is None:
        h_sf = torch.zeros(nvfp4_sf_bytes(a_rows, I, NVFP4_SF_TILED_ROWS), dtype=torch.uint8, device=dev)
    _check(lib().nvfp4_grouped_gemm_swiglu(_ptr(a_codes), _ptr(a_sf), _ptr(gs_a), a_rows,
                                           _ptr(w1_codes), _ptr(w1_sf), _ptr(gs_w1), _ptr(offsets), E,
                                           I, K, _ptr(gs_h), _ptr(h_codes), _ptr(h_sf), _stream()),
           "nvfp4_grouped_gemm_swiglu")
    return h_codes, h_sf


def moe_combine(out, topk_w, flat_to_perm, y=None):
    T, k = topk_w.shape
    K = out.shape[1]
    if y is None:
        y = torch.empty((T, K), dtype=torch.bfloat16, device=out.device)
    _check(lib().moe_combine(_ptr(out), out.stride(0), _ptr(topk_w), _ptr(flat_to_perm), T, k, K,
                             _ptr(y), y.stride(0), _stream()), "moe_combine")
    return y


def moe_forward(x, logits, weights, k, gs_h, ws=None, y=None):
    """The whole expert forward; weights from prepare_moe_weights()."""
    T, K = x.shape
    E = logits.shape[1]
    I = weights["I"]
    nb = moe_forward_workspace_size(T, K, I, E, k)
    if ws is None:
        ws = torch.empty(nb, dtype=torch.uint8, device=x.device)
    if y is None:
        y = torch.empty((T, K), dtype=torch.bfloat16, device=x.device)
    _check(lib().moe_forward(_ptr(x), _ptr(logits), T, K, I, E, k, _ptr(weights["w1_codes"]),
                             _ptr(weights["w1_sf"]), _ptr(weights["gs_w1"]), _ptr(weights["w2_codes"]),
                             _ptr(weights["w2_sf"]), _ptr(weights["gs_w2"]), _ptr(gs_h), _ptr(y),
                             _ptr(ws), ws.numel(), _stream()), "moe_forward")
    return y


def moe_forward_static(x, logits, weights, k, gs_h, gs_x, ws=None, y=None):
    """moe_forward with a pre-computed activation global scale gs_x (device
    f32); the front (route, permute, quantize, scatter) is one kernel."""
    T, K = x.shape
    E = logits.shape[1]
    I = weights["I"]
    if ws is None:
        ws = torch.empty(moe_forward_workspace_size(T, K, I, E, k), dtype=torch.uint8, device=x.device)
    if y is None:
        y = torch.empty((T, K), dtype=torch.bfloat16, device=x.device)
    _check(lib().moe_forward_static(_ptr(x), _ptr(logits), T, K, I, E, k, _ptr(gs_x),
                                    _ptr(weights["w1_codes"]), _ptr(weights["w1_sf"]), _ptr(weights["gs_w1"]),
                                    _ptr(weights["w2_codes"]), _ptr(weights["w2_sf"]), _ptr(weights["gs_w2"]),
                                    _ptr(gs_h), _ptr(y), _ptr(ws), ws.numel(), _stream()), "moe_forward_static")
    return y


def prepare_moe_weights(w1, w2, free_source=False):
    """Offline weight preparation through nvfp4_quantize (README "Bridge Layer":
    quantize_weight_to_nvfp4, interleave_l1_weights, make_b_k_major).

    w1: (E, 2I, K) BF16 rows [gate | up]; w2: (E, K, I) BF16. Each expert gets
    its own global scale; W1 rows are gathered into the granularity-8
    interleaved order by the quantizer's row map.
    """
    E, two_i, K = w1.shape
    I = two_i // 2
    dev = w1.device
    rmap = nvfp4moe_interleave_row_map(two_i).to(dev)
    out = {"E": E, "I": I, "K": K}
    out["w1_codes"] = torch.empty((E, two_i, K // 2), dtype=torch.uint8, device=dev)
    sf1 = nvfp4_sf_bytes(two_i, K)
    out["w1_sf"] = torch.empty(E * sf1, dtype=torch.uint8, device=dev)
    out["gs_w1"] = torch.empty(E, dtype=torch.float32, device=dev)
    out["w2_codes"] = torch.empty((E, K, I // 2), dtype=torch.uint8, device=dev)
    sf2 = nvfp4_sf_bytes(K, I)
    out["w2_sf"] = torch.empty(E * sf2, dtype=torch.uint8, device=dev)
    out["gs_w2"] = torch.empty(E, dtype=torch.float32, device=dev)
    for e in range(E):
        nvfp4_quantize(w1[e], row_src=rmap, codes=out["w1_codes"][e],
                       sf=out["w1_sf"][e * sf1:(e + 1) * sf1], gs_out=out["gs_w1"][e:e + 1])
        nvfp4_quantize(w2[e], codes=out["w2_codes"][e], sf=out["w2_sf"][e * sf2:(e + 1) * sf2],
                       gs_out=out["gs_w2"][e:e + 1])
    return out


SPLIT_STAGES = ("route", "permute", "quantize", "l1_swiglu", "l2", "combine")
FUSED_STAGES = ("dispatch", "l1_swiglu", "l2", "combine")
STATIC_STAGES = ("dispatch_static", "l1_swiglu", "l2", "combine")


def moe_dispatch_supported(T, E, k):
    return bool(lib().moe_dispatch_supported(T, E, k))


def moe_forward_uses_fused_dispatch(T, E, k):
    return bool(lib().moe_forward_uses_fused_dispatch(T, E, k))


def forward_stages(T, E, k):
    """The stages moe_forward runs for this shape: the fused dispatch (one
    call), or the separate route, permute and quantize."""
    return FUSED_STAGES if moe_forward_uses_fused_dispatch(T, E, k) else SPLIT_STAGES


def moe_forward_stages(x, logits, weights, k, gs_h, ws, y, events=None):
    """The C calls moe_forward makes (forward_stages(T, E, k)), issued one by
    one on the current stream with the same workspace carving, so that CUDA
    events can be recorded between them: events, if given, is a list of
    len(forward_stages(T, E, k)) + 1 torch.cuda.Event; events[i] is recorded
    before stage i."""
    T, K = x.shape
    E = logits.shape[1]
    I = weights["I"]
    L = lib()
    lay = moe_forward_workspace_layout(T, K, I, E, k)
    base = ws.data_ptr()
    p = {n: ctypes.c_void_p(base + o) for n, o in lay.items() if n != "a_rows"}
    a_rows = lay["a_rows"]
    M = T * k
    up = lambda v: -(-v // 256) * 256
    perm_ws = base + lay["out"] + up(M * K * 2)
    perm_bytes = int(L.moe_permute_workspace_size(T, k, E))
    disp_ws = perm_ws + up(perm_bytes)
    disp_bytes = int(L.moe_quantize_dispatch_workspace_size(E))
    s = _stream()
    st = torch.cuda.current_stream()

    def mark(i):
        if events is not None:
            events[i].record(st)

    if moe_forward_uses_fused_dispatch(T, E, k):
        mark(0)
        _check(L.moe_dispatch(_ptr(x), K, _ptr(logits), T, K, E, k, p["gs_x"], p["topk_ids"], p["topk_w"],
                              p["offsets"], p["perm_to_flat"], p["flat_to_perm"], p["a_codes"], p["a_sf"],
                              a_rows, ctypes.c_void_p(perm_ws), ws.numel() - (perm_ws - base), s), "dispatch")
        first = 1
    else:
        mark(0)
        _check(L.moe_route_topk(_ptr(logits), T, E, k, p["topk_ids"], p["topk_w"], s), "route")
        mark(1)
        _check(L.moe_permute(p["topk_ids"], T, k, E, p["offsets"], p["perm_to_flat"], p["flat_to_perm"],
                             ctypes.c_void_p(perm_ws), perm_bytes, s), "permute")
        mark(2)
        _check(L.moe_quantize_dispatch(_ptr(x), T, K, K, k, E, p["topk_ids"], p["offsets"], p["flat_to_perm"],
                                       None, p["gs_x"], p["a_codes"], p["a_sf"], a_rows,
                                       ctypes.c_void_p(disp_ws), disp_bytes, s), "quantize")
        first = 3
    mark(first)
    _check(L.nvfp4_grouped_gemm_swiglu(p["a_codes"], p["a_sf"], p["gs_x"], a_rows,
                                       _ptr(weights["w1_codes"]), _ptr(weights["w1_sf"]),
                                       _ptr(weights["gs_w1"]), p["offsets"], E, I, K, _ptr(gs_h),
                                       p["h_codes"], p["h_sf"], s), "l1_swiglu")
    mark(first + 1)
    _check(L.nvfp4_grouped_gemm(p["h_codes"], p["h_sf"], _ptr(gs_h), a_rows, _ptr(weights["w2_codes"]),
                                _ptr(weights["w2_sf"]), _ptr(weights["gs_w2"]), p["offsets"], E, K, I,
                                p["out"], K, s), "l2")
    mark(first + 2)
    _check(L.moe_combine(p["out"], K, p["topk_w"], p["flat_to_perm"], T, k, K, _ptr(y), y.stride(0), s),
           "combine")
    mark(first + 3)
    return y


def moe_forward_static_stages(x, logits, weights, k, gs_h, gs_x, ws, y, events=None):
    """The four C calls moe_forward_static makes (moe_dispatch_static, L1, L2,
    combine) issued one by one with the same workspace carving; events[i] is
    recorded before stage i (len(STATIC_STAGES) + 1 events)."""
    T, K = x.shape
    E = logits.shape[1]
    I = weights["I"]
    L = lib()
    lay = moe_forward_workspace_layout(T, K, I, E, k)
    base = ws.data_ptr()
    p = {n: ctypes.c_void_p(base + o) for n, o in lay.items() if n != "a_rows"}
    a_rows = lay["a_rows"]
    M = T * k
    up = lambda v: -(-v // 256) * 256
    front_off = lay["out"] + up(M * K * 2)
    front_ws = base + front_off
    front_bytes = ws.numel() - front_off
    s = _stream()
    st = torch.cuda.current_stream()

    def mark(i):
        if events is not None:
            events[i].record(st)

    mark(0)
    _check(L.moe_dispatch_static(_ptr(x), K, _ptr(logits), T, K, E, k, _ptr(gs_x), p["topk_ids"], p["topk_w"],
                                 p["offsets"], p["perm_to_flat"], p["flat_to_perm"], p["a_codes"], p["a_sf"],
                                 a_rows, ctypes.c_void_p(front_ws), front_bytes, s), "dispatch_static")
    mark(1)
    _check(L.nvfp4_grouped_gemm_swiglu(p["a_codes"], p["a_sf"], _ptr(gs_x), a_rows,
                                       _ptr(weights["w1_codes"]), _ptr(weights["w1_sf"]),
                                       _ptr(weights["gs_w1"]), p["offsets"], E, I, K, _ptr(gs_h),
                                       p["h_codes"], p["h_sf"], s), "l1_swiglu")
    mark(2)
    _check(L.nvfp4_grouped_gemm(p["h_codes"], p["h_sf"], _ptr(gs_h), a_rows, _ptr(weights["w2_codes"]),
                                _ptr(weights["w2_sf"]), _ptr(weights["gs_w2"]), p["offsets"], E, K, I,
                                p["out"], K, s), "l2")
    mark(3)
    _check(L.moe_combine(p["out"], K, p["topk_w"], p["flat_to_perm"], T, k, K, _ptr(y), K, s), "combine")
    mark(4)
    return y
