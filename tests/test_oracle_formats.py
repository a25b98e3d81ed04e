"""Pins of the oracle's number formats against things other than itself.

* E2M1 decode: the bit-level definition (sign, 2-bit exponent with bias 1,
  1-bit mantissa) and the printed value set (golden table).
* E2M1 encode: the golden tie table and, for random values, minifloat rounding
  done a different way (scale to the local grid spacing, np.rint).
* E4M3 decode/encode: torch's float8_e4m3fn cast (a library routine).
"""
import numpy as np
import pytest
import torch

import oracle as O
from conftest import golden_path


def _read_table(name):
    rows = []
    for line in open(golden_path(name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a, b = line.split()
        rows.append((a, b))
    return rows


def test_e2m1_value_set_golden():
    for code_hex, val in _read_table("e2m1_codes.txt"):
        code = int(code_hex, 16)
        got = O.e2m1_decode(code)
        assert got == float(val), (code, got, val)
        assert np.signbit(got) == bool(code & 8)


def test_e2m1_decode_bit_definition():
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        assert O.e2m1_decode(code) == (-mag if s else mag)


def test_e2m1_rounding_golden():
    for v, code_hex in _read_table("e2m1_rounding.txt"):
        assert O.e2m1_encode(float(v)) == int(code_hex, 16), v


def _e2m1_minifloat(v):
    """Round |v| onto the E2M1 grid by spacing: 0.5 below 2, 1 in [2,4), 2 in [4,6]."""
    a = abs(float(np.float32(v)))
    if a < 2.0:
        q = np.rint(a * 2.0) / 2.0          # np.rint: ties to even multiple
    elif a < 4.0:
        q = np.rint(a)
    else:
        q = min(2.0 * np.rint(a / 2.0), 6.0)
    q = min(q, 6.0)
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    return (8 if np.signbit(np.float32(v)) else 0) | mags.index(q)


def test_e2m1_encode_random_vs_minifloat_rounding():
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.uniform(-7, 7, 20000), rng.normal(0, 2, 20000),
                           np.arange(-6.5, 6.5, 0.125)]).astype(np.float32)
    for v in vals:
        assert O.e2m1_encode(v) == _e2m1_minifloat(v), v


def test_e4m3_decode_all_codes_vs_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = O.e4m3_decode(c)
        if np.isnan(ref[c]):
            assert np.isnan(got)
        else:
            assert got == ref[c], (c, got, ref[c])
    assert O.e4m3_decode(0x7E) == 448.0
    assert O.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_vs_torch_cast():
    rng = np.random.default_rng(2)
    reps = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    mids = (reps[:-1] + reps[1:]) / 2
    vals = np.concatenate([reps, mids, np.nextafter(mids, 0), np.nextafter(mids, 1000),
                           rng.uniform(0, 448, 50000), 2.0 ** rng.uniform(-12, 8.8, 50000)])
    vals = vals[vals <= 448].astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([O.e4m3_encode(v) for v in vals], np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (vals[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_e4m3_encode_saturates():
    # the reading taken: saturating (satfinite) conversion, never NaN
    for v in [448.0, 449.0, 463.9, 464.0, 1e6, float("inf")]:
        assert O.e4m3_encode(v) == 0x7E
    assert O.e4m3_encode(0.0) == 0
    assert O.e4m3_encode(2.0 ** -10) == 0          # tie between 0 and 2^-9 -> even (0)
    assert O.e4m3_encode(1.5 * 2.0 ** -10) == 1


def test_global_scale():
    assert O.global_scale(0.0) == 1.0
    assert O.global_scale(448.0) == np.float32(6.0)
    assert O.global_scale(6.0) == np.float32(448.0)
    a = np.float32(5.123)
    assert O.global_scale(a) == np.float32(2688.0) / a


def test_amax_is_the_largest_magnitude():
    """amax = max |x| (the activation global scale is 2688 / amax): the extreme
    element may be negative."""
    rng = np.random.default_rng(11)
    x = rng.normal(0, 1, (6, 48)).astype(np.float32)
    x[4, 17] = -9.5
    xb = torch.from_numpy(x).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    ref = float(xb.float().abs().max())
    assert ref == 9.5
    assert O.amax_bf16(bits) == np.float32(ref)
    assert O.amax_f32(x) == np.float32(np.abs(x).max())
    assert O.global_scale(O.amax_bf16(bits)) == np.float32(2688.0) / np.float32(9.5)
