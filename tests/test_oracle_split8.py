"""Pins of the oracle's binary16 / E4M3 rounding and of the fp16 + e4m3 dX operands.

The split encodes scale[c] * T as h_c * T (binary16) plus 2^-7 * l_c * T (e4m3),
with scale[c] = a_c * 2^e_c, a_c in +-[1, 2).  The oracle states it from the two
formats' definitions (IEEE 754 binary16; the OCP 8-bit E4M3 format).  These pins
tie it to independent implementations of the same formats (numpy's float16 and
torch's float8_e4m3fn conversions), to values the format definitions fix, and to
the reconstruction identity the encoding exists for.
"""
import numpy as np
import pytest
import torch

import oracle


def _f16_bits(x):
    return int(np.array(x, dtype=np.float64).astype(np.float16).view(np.uint16))


# --------------------------------------------------------------- binary16

def test_f16_value_matches_numpy_on_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    for b in range(0, 1 << 16, 7):   # a spread of patterns, NaNs excluded
        if np.isnan(ref[b]):
            continue
        assert oracle.f16_value(b) == ref[b], hex(b)


def test_f16_round_matches_numpy():
    rng = np.random.default_rng(3)
    vals = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.integers(-9, 5, 3000),   # normal and subnormal range
        rng.uniform(-65504, 65504, 500),
        np.ldexp(rng.integers(1, 2048, 500).astype(np.float64) + 0.5, rng.integers(-35, 5, 500)),   # ties
        [0.0, -0.0, 65504.0, 65519.99, -65519.99, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14],
    ])
    for x in vals:
        assert oracle.f16_round(float(x)) == _f16_bits(x), x


def test_f16_golden_values():
    # IEEE 754 binary16 patterns fixed by the format's definition
    assert oracle.f16_round(1.0) == 0x3C00
    assert oracle.f16_round(-2.0) == 0xC000
    assert oracle.f16_round(65504.0) == 0x7BFF
    assert oracle.f16_round(65520.0) == 0x7C00          # rounds past the largest finite value
    assert oracle.f16_round(2.0 ** -24) == 0x0001       # smallest subnormal
    assert oracle.f16_round(2.0 ** -14) == 0x0400       # smallest normal
    assert oracle.f16_round(1.0 + 2.0 ** -11) == 0x3C00   # tie: to even
    assert oracle.f16_round(1.0 + 3 * 2.0 ** -11) == 0x3C02


# --------------------------------------------------------------- E4M3

def test_e4m3_value_matches_torch_on_every_pattern():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        if np.isnan(ref[b]):
            assert b & 0x7F == 0x7F
            continue
        assert oracle.e4m3_value(b) == ref[b], hex(b)


def test_e4m3_round_matches_torch_in_range():
    rng = np.random.default_rng(4)
    vals = np.concatenate([
        rng.uniform(-464, 464, 2000),
        rng.standard_normal(2000) * 10.0 ** rng.integers(-4, 2, 2000),
        np.ldexp(rng.integers(1, 16, 600).astype(np.float64) + 0.5, rng.integers(-12, 6, 600)),   # ties
        [0.0, -0.0, 448.0, 460.0, -460.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -6],
    ]).astype(np.float32)
    vals = vals[np.abs(vals) <= 464.0]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, r in zip(vals, ref):
        assert oracle.e4m3_round(float(x)) == int(r), float(x)


def test_e4m3_golden_values():
    # E4M3 patterns fixed by the format's definition (bias 7, three fraction bits)
    assert oracle.e4m3_round(1.0) == 0x38
    assert oracle.e4m3_round(448.0) == 0x7E              # largest finite
    assert oracle.e4m3_round(2.0 ** -6) == 0x08          # smallest normal
    assert oracle.e4m3_round(2.0 ** -9) == 0x01          # smallest subnormal
    assert oracle.e4m3_round(2.0 ** -10) == 0x00         # tie between 0 and 2^-9: to even
    assert oracle.e4m3_round(1.0625) == 0x38             # tie: to even
    assert oracle.e4m3_round(1.1875) == 0x3A
    assert oracle.e4m3_round(-0.0) == 0x80


@pytest.mark.parametrize("x", [464.0, 470.0, 500.0, 1e4, 3.4e38])
def test_e4m3_saturates(x):
    assert oracle.e4m3_round(x) == 0x7E
    assert oracle.e4m3_round(-x) == 0xFE


# --------------------------------------------------------------- the split planes

def _split_case(K=24, N=64, seed=5):
    rng = np.random.default_rng(seed)
    q = rng.integers(-7, 8, (K, N)).astype(np.int8)
    scale = np.concatenate([
        rng.uniform(0.005, 0.1, N - 8),
        [0.0, -0.05, 1e-30, 2.0 ** -140, 3.0e4, -7.0, 0.1, 0.005],   # zero, negative, fp32 subnormal, large
    ]).astype(np.float32)
    return q, scale


def test_split_reconstructs_the_scale():
    q, scale = _split_case()
    wh, wl = oracle.split8_planes(q, scale)
    T = np.where(q >= 2, 1, np.where(q <= -2, -1, 0))
    s = scale.astype(np.float64)
    m, e = np.frexp(np.abs(s))   # |s| = m * 2^e, m in [0.5, 1)
    a = np.where(s != 0, np.ldexp(s, -(e - 1)), 0.0)
    assert np.all((np.abs(a) >= 1) & (np.abs(a) < 2) | (s == 0))
    h = wh.view(np.float16).astype(np.float64)
    l = torch.from_numpy(wl).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    recon = h + l / 128.0
    assert np.all(np.abs(recon - a * T) <= 2.0 ** -15 * np.abs(a * T))
    # times 2^e_c it is scale[c] * T within the same relative bound
    full = np.ldexp(recon, np.where(s != 0, e - 1, 0))
    assert np.all(np.abs(full - s * T) <= 2.0 ** -15 * np.abs(s * T))


def test_split_planes_match_library_conversions():
    q, scale = _split_case(seed=6)
    wh, wl = oracle.split8_planes(q, scale)
    T = np.where(q >= 2, 1, np.where(q <= -2, -1, 0))
    s = scale.astype(np.float64)
    m, e = np.frexp(np.abs(s))
    a = np.where(s != 0, np.ldexp(s, -(e - 1)), 0.0)
    h = a.astype(np.float16)                              # numpy: binary16, ties to even
    d = (np.ldexp(a - h.astype(np.float64), 7)).astype(np.float32)   # exact
    l = torch.from_numpy(d).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    hb = h.view(np.uint16)
    for r in range(q.shape[0]):
        for c in range(q.shape[1]):
            t = T[r, c]
            want_h = 0 if t == 0 else (hb[c] ^ 0x8000 if t < 0 else hb[c])
            want_l = 0 if t == 0 else (l[c] ^ 0x80 if t < 0 else l[c])
            assert wh[r, c] == want_h and wl[r, c] == want_l, (r, c)


def test_split_of_exact_scales_has_no_low_part():
    # a scale with at most 11 significant bits is exact in binary16: l_c = 0
    K, N = 4, 16
    q = np.full((K, N), 5, np.int8)
    scale = np.ldexp(np.arange(1, N + 1) * 3.0 + 1024.0, -12).astype(np.float32)
    wh, wl = oracle.split8_planes(q, scale)
    assert np.all(wl == 0)
    m, e = np.frexp(scale.astype(np.float64))
    assert np.all(wh.view(np.float16).astype(np.float64) == np.ldexp(scale.astype(np.float64), -(e - 1)))
