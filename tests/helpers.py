"""Test-side helpers: layout conversions written from the layouts documented in
include/nvfp4moe.h (independent of both the CUDA code and the oracle)."""
import numpy as np
import torch


def sf_tiled_index(rows, cols):
    """Byte index in the tiled layout of every (r, b) scale, as (rows, cols//16)."""
    r = np.arange(rows, dtype=np.int64)[:, None]
    b = np.arange(cols // 16, dtype=np.int64)[None, :]
    c4 = (cols + 63) // 64
    return ((r // 128) * c4 + b // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + b % 4


def sf_tiled_to_rowmajor(sf_tiled, rows, cols):
    sf = np.asarray(sf_tiled).reshape(-1)
    return sf[sf_tiled_index(rows, cols)]


def sf_rows_index(rows, cols):
    """Byte index in the NVFP4_SF_TILED_ROWS layout (the GEMMs' activation
    scales) of every (r, b) scale, as (rows, cols//16)."""
    r = np.arange(rows, dtype=np.int64)[:, None]
    b = np.arange(cols // 16, dtype=np.int64)[None, :]
    s = (cols + 255) // 256
    return ((r // 128) * s + b // 16) * 2048 + (r % 128) * 16 + b % 16


def sf_rows_to_rowmajor(sf_rows, rows, cols):
    sf = np.asarray(sf_rows).reshape(-1)
    return sf[sf_rows_index(rows, cols)]


def padded_starts(offsets):
    """P_e = 128 * sum_{e'<e} ceil(n_e'/128)."""
    offsets = np.asarray(offsets, np.int64)
    counts = np.diff(offsets)
    tiles = (counts + 127) // 128
    return np.concatenate([[0], np.cumsum(tiles) * 128])


def padded_rows_of_compact(offsets):
    """Padded row of every compact row r (grouped order)."""
    offsets = np.asarray(offsets, np.int64)
    P = padded_starts(offsets)
    M = int(offsets[-1])
    rows = np.empty(M, np.int64)
    for e in range(len(offsets) - 1):
        rows[offsets[e]:offsets[e + 1]] = P[e] + np.arange(offsets[e + 1] - offsets[e])
    return rows


def cosine(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float((a * b).sum() / np.sqrt((a * a).sum() * (b * b).sum()))


def to_np(t):
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def assert_close_tol(got, ref, what=""):
    """|gpu - oracle| <= 2e-2 * max(1, |oracle|) per element."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    lim = 2e-2 * np.maximum(1.0, np.abs(ref))
    bad = np.nonzero(err > lim)
    assert bad[0].size == 0, "%s: %d elements out of tolerance, max err %.4g" % (
        what, bad[0].size, err.max())
