"""Pins of the oracle's fused-front-end steps (README "THE PLAN", item 3:
"Q norm -> RoPE -> NVFP4 quant" in one pass): the RMS norm against torch's
rms_norm, the rotation against complex multiplication, and closed forms."""
import numpy as np
import torch

import oracle as O
from nvfp4_block_scaled_05_gb300.workloads import bf16_bits


def _bits(a):
    return bf16_bits(torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16))


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_norm_matches_torch_rms_norm():
    rng = np.random.default_rng(0)
    x = _bits(rng.normal(0, 3, (40, 192)))
    gamma = rng.normal(1, 0.2, 192)
    eps = 1e-6
    y = O.rmsnorm_rope(x, gamma, eps, 0, np.zeros(40, np.int32), np.zeros((1, 1)), np.zeros((1, 1)))
    ref = torch.nn.functional.rms_norm(torch.from_numpy(_f64(x)), (192,), torch.from_numpy(gamma), eps).numpy()
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-15)


def test_rotation_matches_complex_multiplication():
    rng = np.random.default_rng(1)
    rows, D, R, P = 25, 192, 64, 300
    x = _bits(rng.normal(0, 1, (rows, D)))
    gamma = rng.normal(1, 0.1, D)
    ang = rng.uniform(-np.pi, np.pi, (P, R // 2))
    pos = rng.integers(0, P, rows).astype(np.int32)
    y = O.rmsnorm_rope(x, gamma, 1e-5, R, pos, np.cos(ang), np.sin(ang))
    n = O.rmsnorm_rope(x, gamma, 1e-5, 0, pos, np.zeros((1, 1)), np.zeros((1, 1)))   # norm only
    assert np.array_equal(y[:, :D - R], n[:, :D - R])                              # nope part untouched
    z = (n[:, D - R::2] + 1j * n[:, D - R + 1::2]) * np.exp(1j * ang[pos])
    assert np.allclose(y[:, D - R::2], z.real, rtol=1e-13, atol=1e-14)
    assert np.allclose(y[:, D - R + 1::2], z.imag, rtol=1e-13, atol=1e-14)


def test_closed_forms():
    D, R = 64, 32
    # a constant row normalises to gamma * sign (up to eps)
    x = _bits(np.full((2, D), [[2.5], [-0.75]]))
    gamma = np.linspace(0.5, 1.5, D)
    y = O.rmsnorm_rope(x, gamma, 0.0, 0, np.zeros(2, np.int32), np.zeros((1, 1)), np.zeros((1, 1)))
    assert np.allclose(y[0], gamma, rtol=1e-15) and np.allclose(y[1], -gamma, rtol=1e-15)
    # cos 1 / sin 0: identity; cos 0 / sin 1: (a, b) -> (-b, a), exactly
    rng = np.random.default_rng(2)
    x = _bits(rng.normal(0, 1, (3, D)))
    g1 = np.ones(D)
    base = O.rmsnorm_rope(x, g1, 1e-6, 0, np.zeros(3, np.int32), np.zeros((1, 1)), np.zeros((1, 1)))
    tab_c = np.stack([np.ones(R // 2), np.zeros(R // 2)])
    tab_s = np.stack([np.zeros(R // 2), np.ones(R // 2)])
    same = O.rmsnorm_rope(x, g1, 1e-6, R, np.zeros(3, np.int32), tab_c, tab_s)
    quarter = O.rmsnorm_rope(x, g1, 1e-6, R, np.ones(3, np.int32), tab_c, tab_s)
    assert np.array_equal(same, base)
    assert np.array_equal(quarter[:, D - R::2], -base[:, D - R + 1::2])
    assert np.array_equal(quarter[:, D - R + 1::2], base[:, D - R::2])
    # every rotation keeps each pair's length
    ang = rng.uniform(0, 2 * np.pi, (5, R // 2))
    rot = O.rmsnorm_rope(x, g1, 1e-6, R, np.array([4, 1, 3], np.int32), np.cos(ang), np.sin(ang))
    l0 = base[:, D - R::2] ** 2 + base[:, D - R + 1::2] ** 2
    l1 = rot[:, D - R::2] ** 2 + rot[:, D - R + 1::2] ** 2
    assert np.allclose(l0, l1, rtol=1e-13)
