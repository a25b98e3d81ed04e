"""The C-ABI library builds, loads, and exports every function include/nvfp4moe.h
declares; host-only entry points behave as documented (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT


def _declared():
    text = open(os.path.join(ROOT, "include", "nvfp4moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[a-z_0-9 ]+?\**\s*\b([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return")))


@pytest.fixture(scope="module")
def lib():
    from nvfp4_block_scaled_05_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_entry_points():
    names = _declared()
    for must in ["nvfp4_quantize", "moe_permute", "nvfp4_grouped_gemm", "nvfp4_grouped_gemm_swiglu",
                 "moe_forward", "moe_route_topk", "moe_combine", "moe_quantize_dispatch"]:
        assert must in names


def test_binding_constants_match_the_header():
    """The binding's copies of the header's #define constants (bench.py counts
    the front's launches from the threshold)."""
    from nvfp4_block_scaled_05_gb300 import binding as B
    with open(os.path.join(ROOT, "include", "nvfp4moe.h")) as f:
        text = f.read()
    defs = dict(re.findall(r"#define (NVFP4\w+) (\d+)", text))
    assert int(defs["NVFP4MOE_FRONT_FUSED_QUANTIZE_MAX_ROWS"]) == B.FRONT_FUSED_QUANTIZE_MAX_ROWS
    for name in ("NVFP4_SF_ROWMAJOR", "NVFP4_SF_TILED", "NVFP4_SF_TILED_ROWS"):
        assert int(defs[name]) == getattr(B, name)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_host_only_entry_points(lib):
    from nvfp4_block_scaled_05_gb300 import binding as B
    assert B.nvfp4_sf_bytes(128, 64, B.NVFP4_SF_TILED) == 512
    assert B.nvfp4_sf_bytes(129, 65, B.NVFP4_SF_TILED) == 2 * 2 * 512
    assert B.nvfp4_sf_bytes(3, 32, B.NVFP4_SF_ROWMAJOR) == 6
    assert B.nvfp4_sf_bytes(128, 256, B.NVFP4_SF_TILED_ROWS) == 2048
    assert B.nvfp4_sf_bytes(129, 257 // 16 * 16, B.NVFP4_SF_TILED_ROWS) == 2 * 1 * 2048
    assert B.nvfp4_sf_bytes(128, 7168, B.NVFP4_SF_TILED_ROWS) == B.nvfp4_sf_bytes(128, 7168, B.NVFP4_SF_TILED)
    assert B.nvfp4_sf_bytes(256, 320, B.NVFP4_SF_TILED_ROWS) == 2 * 2 * 2048
    assert B.nvfp4moe_padded_rows(1024, 256) == -(-(1024 + 256 * 127) // 128) * 128
    assert B.nvfp4moe_padded_rows(1000, 3) == -(-(1000 + 3 * 127) // 128) * 128
    assert B.nvfp4moe_padded_rows(1, 8) == 128
    m = B.nvfp4moe_interleave_row_map(32).numpy()
    assert list(m[:16]) == list(range(8)) + list(range(16, 24))
    assert sorted(m) == list(range(32))
    import oracle as O
    a = np.arange(64).reshape(32, 2)
    assert np.array_equal(a[m], O.interleave_rows(a, 8))


def test_invalid_arguments_are_rejected_on_the_host(lib):
    vp = ctypes.c_void_p
    lib.nvfp4_quantize.restype = ctypes.c_int
    # cols not a multiple of 16
    st = lib.nvfp4_quantize(vp(16), ctypes.c_int64(4), ctypes.c_int64(20), ctypes.c_int64(32), None,
                            None, None, vp(16), vp(16), 1, None, ctypes.c_size_t(0), None)
    assert st == -1
    # no workspace while the global scale has to be computed
    st = lib.nvfp4_quantize(vp(256), ctypes.c_int64(4), ctypes.c_int64(32), ctypes.c_int64(32), None,
                            None, None, vp(256), vp(256), 1, None, ctypes.c_size_t(0), None)
    assert st == -3
    lib.moe_route_topk.restype = ctypes.c_int
    st = lib.moe_route_topk(vp(256), ctypes.c_int64(4), 8, 17, vp(256), vp(256), None)
    assert st == -2
    lib.nvfp4_grouped_gemm.restype = ctypes.c_int
    st = lib.nvfp4_grouped_gemm(vp(256), vp(256), vp(256), ctypes.c_int64(128), vp(256), vp(256),
                                vp(256), vp(256), 1, ctypes.c_int64(100), ctypes.c_int64(64), vp(256),
                                ctypes.c_int64(128), None)
    assert st == -2
    lib.moe_forward_workspace_size.restype = ctypes.c_size_t
    assert lib.moe_forward_workspace_size(ctypes.c_int64(8), ctypes.c_int64(100), ctypes.c_int64(64), 8, 2) == 0


def test_host_fault_injection_rejected_before_any_launch(lib):
    """Too-small workspaces, null and misaligned pointers and unsupported shapes
    come back as status codes from the host checks, before anything is
    launched (no GPU needed)."""
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    for name in ["moe_forward", "moe_forward_static", "nvfp4_linear", "nvfp4_rmsnorm_rope_quantize",
                 "moe_dispatch_static", "moe_permute", "moe_combine"]:
        getattr(lib, name).restype = ctypes.c_int
    lib.moe_forward_workspace_size.restype = ctypes.c_size_t
    T, K, I, E, k = 16, 256, 128, 8, 2
    need = lib.moe_forward_workspace_size(i64(T), i64(K), i64(I), E, k)
    assert need > 0
    p = vp(1 << 20)
    # workspace one byte short / misaligned / absent
    args = [p, p, i64(T), i64(K), i64(I), E, k, p, p, p, p, p, p, p, p]
    assert lib.moe_forward(*args, p, sz(need - 1), None) == -3
    assert lib.moe_forward(*args, vp((1 << 20) + 16), sz(need), None) == -3
    assert lib.moe_forward(*args, None, sz(need), None) == -3
    # a null weight pointer
    bad = list(args)
    bad[7] = None
    assert lib.moe_forward(*bad, p, sz(need), None) == -1
    # unsupported shapes: K not a multiple of 128, k > E
    assert lib.moe_forward(p, p, i64(T), i64(200), i64(I), E, k, p, p, p, p, p, p, p, p, p, sz(need), None) == -2
    assert lib.moe_forward(p, p, i64(T), i64(K), i64(I), 4, 5, p, p, p, p, p, p, p, p, p, sz(need), None) == -2
    # the static forward needs its pre-computed gs_x
    assert lib.moe_forward_static(p, p, i64(T), i64(K), i64(I), E, k, None, p, p, p, p, p, p, p, p, p, sz(need),
                                  None) == -1
    # static dispatch: padded operand too small
    lib.moe_dispatch_static_workspace_size.restype = ctypes.c_size_t
    wsd = lib.moe_dispatch_static_workspace_size(i64(T), E)
    assert wsd > 0
    assert lib.moe_dispatch_static(p, i64(K), p, i64(T), i64(K), E, k, p, p, p, p, p, p, p, p, i64(128), p, sz(wsd),
                                   None) == -1
    # linear: row capacity below 128 * ceil(M / 128); workspace too small
    lib.nvfp4_linear_workspace_size.restype = ctypes.c_size_t
    lws = lib.nvfp4_linear_workspace_size()
    assert lib.nvfp4_linear(p, p, p, i64(130), i64(128), p, p, p, i64(256), i64(256), p, i64(256), p, sz(lws),
                            None) == -1
    assert lib.nvfp4_linear(p, p, p, i64(100), i64(128), p, p, p, i64(256), i64(256), p, i64(256), p,
                            sz(lws - 1), None) == -3
    # norm + rope + quant: rope_dims not a multiple of 16, missing tables, misaligned gamma
    f = ctypes.c_float
    assert lib.nvfp4_rmsnorm_rope_quantize(p, i64(4), i64(192), i64(192), p, f(1e-6), i64(40), p, p, p, i64(10),
                                           p, p, p, 1, None, None) == -2
    assert lib.nvfp4_rmsnorm_rope_quantize(p, i64(4), i64(192), i64(192), p, f(1e-6), i64(64), None, p, p,
                                           i64(10), p, p, p, 1, None, None) == -1
    assert lib.nvfp4_rmsnorm_rope_quantize(p, i64(4), i64(192), i64(192), vp((1 << 20) + 4), f(1e-6), i64(64), p,
                                           p, p, i64(10), p, p, p, 1, None, None) == -1
    # permute: workspace too small
    lib.moe_permute_workspace_size.restype = ctypes.c_size_t
    pws = lib.moe_permute_workspace_size(i64(T), k, E)
    assert lib.moe_permute(p, i64(T), k, E, p, p, p, p, sz(pws - 1), None) == -3


def test_layout_helpers_reject_bad_arguments(lib):
    """The offline layout helpers check their arguments on the host."""
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    for name in ["nvfp4_sf_to_tiled", "nvfp4_sf_from_tiled", "nvfp4_interleave_gate_up"]:
        getattr(lib, name).restype = ctypes.c_int
    p, q = vp(1 << 20), vp(1 << 21)
    assert lib.nvfp4_sf_to_tiled(p, i64(1), i64(128), i64(40), 1, q, None) == -1     # cols % 16
    assert lib.nvfp4_sf_to_tiled(p, i64(1), i64(128), i64(64), 0, q, None) == -1     # row-major is not tiled
    assert lib.nvfp4_sf_from_tiled(None, i64(1), i64(128), i64(64), 2, q, None) == -1
    assert lib.nvfp4_sf_to_tiled(None, i64(0), i64(128), i64(64), 1, None, None) == 0  # nothing to do
    assert lib.nvfp4_interleave_gate_up(p, None, i64(1), i64(24), i64(64), 0, 0, q, None, None) == -1  # 2I % 16
    assert lib.nvfp4_interleave_gate_up(p, None, i64(1), i64(32), i64(64), 0, 2, q, None, None) == -1  # inverse
    assert lib.nvfp4_interleave_gate_up(p, None, i64(1), i64(32), i64(64), 0, 0, None, None, None) == -1
    assert lib.nvfp4_interleave_gate_up(p, None, i64(1), i64(32), i64(64), 0, 0, p, None, None) == -1  # in place
    assert lib.nvfp4_interleave_gate_up(p, p, i64(1), i64(32), i64(64), 3, 0, q, q, None) == -1      # layout
