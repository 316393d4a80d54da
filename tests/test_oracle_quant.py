"""Pins of the oracle's int4 quantiser against facts other than itself:
a hand-built grid group (closed form), exact rational arithmetic with an
IEEE round-to-nearest-even written from its definition, the error bound of
rounding to the nearest code, constant groups, short last groups and
re-quantisation of the dequantised values."""
from fractions import Fraction
import math

import numpy as np
import pytest
import torch

from oracle import quant
from oracle.bf16 import round_bf16, bits_bf16, from_bits
import synthetic


def rne(x: Fraction, p: int) -> Fraction:
    """Round a rational to the nearest binary number with p significant bits,
    ties to even (IEEE 754 roundTiesToEven, no exponent limits)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - p + 1)
    m = a / ulp
    n = math.floor(m)
    r = m - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def exact_group(vals):
    """s, z, codes of one group by exact rationals + explicit rounding."""
    fr = [Fraction(float(v)) for v in vals]
    lo, hi = min(fr), max(fr)
    s = rne(rne(rne(hi - lo, 24) / 15, 24), 8)
    if s == 0:
        s = Fraction(1)
    z = rne(rne(-lo / s, 24), 8)
    codes = []
    for w in fr:
        t = rne(rne(w / s, 24) + z, 24)
        n = math.floor(t)
        r = t - n
        if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
            n += 1
        codes.append(min(15, max(0, n)))
    return s, z, codes


def test_round_bf16_matches_rational_rne():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(2000) * 10.0 ** rng.integers(-6, 6, 2000)).astype(np.float32)
    got = round_bf16(x)
    for xi, gi in zip(x, got):
        assert Fraction(float(gi)) == rne(Fraction(float(xi)), 8)


def test_grid_group_closed_form():
    # codes c_j = 7j mod 16 cover 0..15; w = (c - 8) * 2^-6 lies on the grid with
    # lo = -0.125, hi = 7 * 2^-6, so s = 2^-6 and z = 8 exactly and q = c.
    c = (np.arange(64) * 7) % 16
    w = ((c - 8) * 2.0 ** -6).astype(np.float32)[None, :]
    q, s, z = quant.w4_pack(w)
    assert s[0, 0] == 2.0 ** -6 and z[0, 0] == 8.0
    assert np.array_equal(quant.unpack_codes(q, 64)[0], c)
    # byte j holds element 2j low, 2j+1 high
    assert q[0, 0] == (c[0] | (c[1] << 4)) and q[0, 5] == (c[10] | (c[11] << 4))
    assert np.array_equal(quant.w4_dequant(q, s, z, 64), w)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_pack_matches_exact_rationals(seed):
    w = synthetic.randn_bf16((6, 64 * 3), seed, std=0.02).float().numpy()
    q, s, z = quant.w4_pack(w)
    codes = quant.unpack_codes(q, w.shape[1])
    for r in range(w.shape[0]):
        for g in range(3):
            es, ez, ec = exact_group(w[r, g * 64:(g + 1) * 64])
            assert Fraction(float(s[r, g])) == es
            assert Fraction(float(z[r, g])) == ez
            assert list(codes[r, g * 64:(g + 1) * 64]) == ec


def test_dequant_error_bound_and_short_group():
    k = 688                                   # 10 full groups + one of 48
    w = synthetic.randn_bf16((32, k), 5, std=0.02).float().numpy()
    q, s, z = quant.w4_pack(w)
    assert q.shape == (32, 11 * 32) and s.shape == (32, 11)
    # padding nibbles past K are zero
    assert np.all(quant.unpack_codes(q, 11 * 64)[:, k:] == 0)
    deq = quant.w4_dequant(q, s, z, k)
    sg = s[:, np.arange(k) // 64]
    # nearest code: |q - (w/s + z)| <= 1/2 (+ clamp slack from the bf16 z and
    # s roundings), then one bf16 rounding of the product
    assert np.all(np.abs(deq - w) <= 0.57 * sg + 2.0 ** -9 * np.abs(deq))
    # the last, short group uses only its own 48 elements
    es, ez, ec = exact_group(w[3, 640:688])
    assert Fraction(float(s[3, 10])) == es and Fraction(float(z[3, 10])) == ez


def test_constant_group_exact():
    w = np.full((2, 64), 0.03125, np.float32)
    w[1] = -0.0078125
    q, s, z = quant.w4_pack(w)
    assert np.all(s == 1.0)
    assert np.array_equal(quant.w4_dequant(q, s, z, 64), w)


def test_requantise_dequantised_is_idempotent():
    w = synthetic.randn_bf16((16, 256), 9, std=0.02).float().numpy()
    q, s, z = quant.w4_pack(w)
    deq = quant.w4_dequant(q, s, z, 256)
    codes = quant.unpack_codes(q, 256)
    sg = s[:, np.arange(256) // 64]
    zg = z[:, np.arange(256) // 64]
    again = np.clip(np.rint(deq / sg + zg), 0, 15)
    assert np.array_equal(again, codes)


def test_w4_gemm_identity_equals_dequant():
    k = 128
    w = synthetic.randn_bf16((8, k), 11, std=0.02).float().numpy()
    q, s, z = quant.w4_pack(w)
    y = quant.w4_gemm(np.eye(k, dtype=np.float32), q, s, z, k)
    assert np.array_equal(y.T, quant.w4_dequant(q, s, z, k))


def test_bits_roundtrip():
    x = round_bf16(np.linspace(-3, 3, 101, dtype=np.float32))
    assert np.array_equal(from_bits(bits_bf16(x)), x)
    t = torch.tensor(x).to(torch.bfloat16)
    assert np.array_equal(t.view(torch.int16).numpy().view(np.uint16), bits_bf16(x))
