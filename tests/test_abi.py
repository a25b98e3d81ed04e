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


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_host_only_entry_points(lib):
    from nvfp4_block_scaled_05_gb300 import binding as B
    assert B.nvfp4_sf_bytes(128, 64, B.NVFP4_SF_TILED) == 512
    assert B.nvfp4_sf_bytes(129, 65, B.NVFP4_SF_TILED) == 2 * 2 * 512
    assert B.nvfp4_sf_bytes(3, 32, B.NVFP4_SF_ROWMAJOR) == 6
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
