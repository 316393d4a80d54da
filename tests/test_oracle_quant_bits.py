"""Pins of the oracle's 2- and 3-bit quantiser and code layouts (lower and
mixed precision for the substitute layers, "Low-Bit Shadow" report 5.1
point 2, 10.1 (2)): exact rational arithmetic with an IEEE
round-to-nearest-even written from its definition, hand-built grid groups
(closed form), the bit positions of every code read back bit by bit,
the rounding error bound, constant and short groups, and agreement of the
4-bit case with the separately written int4 quantiser."""
from fractions import Fraction
import math

import numpy as np
import pytest

from oracle import quant
from test_oracle_quant import rne
import synthetic


def exact_group(vals, levels):
    fr = [Fraction(float(v)) for v in vals]
    lo, hi = min(fr), max(fr)
    s = rne(rne(rne(hi - lo, 24) / levels, 24), 8)
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
        codes.append(min(levels, max(0, n)))
    return s, z, codes


def code_at(q_row, bits, e):
    """Code of element e read bit by bit from the stated layout."""
    g, j = divmod(e, 64)
    base = g * 8 * bits
    if bits == 4:
        byte = int(q_row[base + j // 2])
        return (byte >> (4 * (j % 2))) & 15
    byte = int(q_row[base + j // 4])
    c = (byte >> (2 * (j % 4))) & 3
    if bits == 3:
        hb = (int(q_row[base + 16 + j // 8]) >> (j % 8)) & 1
        c |= hb << 2
    return c


@pytest.mark.parametrize("bits", [2, 3])
@pytest.mark.parametrize("seed", [0, 1])
def test_pack_matches_exact_rationals(bits, seed):
    w = synthetic.randn_bf16((4, 64 * 3), seed + 10 * bits, std=0.02).float().numpy()
    q, s, z = quant.wq_pack(w, bits)
    assert q.shape == (4, 3 * 8 * bits)
    for r in range(w.shape[0]):
        for g in range(3):
            es, ez, ec = exact_group(w[r, g * 64:(g + 1) * 64], 2 ** bits - 1)
            assert Fraction(float(s[r, g])) == es
            assert Fraction(float(z[r, g])) == ez
            got = [code_at(q[r], bits, g * 64 + j) for j in range(64)]
            assert got == ec


@pytest.mark.parametrize("bits", [2, 3])
def test_grid_group_closed_form(bits):
    # codes c_j = 5j mod 2^b cover every level; w = (c - m) * 2^-6 lies on the
    # grid with lo = -m 2^-6 and hi = (L - m) 2^-6, so s = 2^-6, z = m, q = c
    L = 2 ** bits - 1
    m = (L + 1) // 2
    c = (np.arange(64) * 5) % (L + 1)
    w = ((c - m) * 2.0 ** -6).astype(np.float32)[None, :]
    q, s, z = quant.wq_pack(w, bits)
    assert s[0, 0] == 2.0 ** -6 and z[0, 0] == float(m)
    assert [code_at(q[0], bits, e) for e in range(64)] == list(c)
    assert np.array_equal(quant.wq_unpack_codes(q, 64, bits)[0], c)
    assert np.array_equal(quant.wq_dequant(q, s, z, 64, bits), w)


def test_four_bits_equals_the_int4_quantiser():
    w = synthetic.randn_bf16((8, 688), 3, std=0.02).float().numpy()
    a = quant.wq_pack(w, 4)
    b = quant.w4_pack(w)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert np.array_equal(quant.wq_dequant(*a, 688, 4), quant.w4_dequant(*b, 688))


@pytest.mark.parametrize("bits", [2, 3])
def test_error_bound_short_group_and_padding(bits):
    k = 688                                   # 10 full groups + one of 48
    w = synthetic.randn_bf16((16, k), 5, std=0.02).float().numpy()
    q, s, z = quant.wq_pack(w, bits)
    assert q.shape == (16, 11 * 8 * bits) and s.shape == (16, 11)
    assert np.all(quant.wq_unpack_codes(q, 11 * 64, bits)[:, k:] == 0)
    deq = quant.wq_dequant(q, s, z, k, bits)
    sg = s[:, np.arange(k) // 64]
    assert np.all(np.abs(deq - w) <= 0.57 * sg + 2.0 ** -9 * np.abs(deq))
    es, ez, _ = exact_group(w[3, 640:688], 2 ** bits - 1)
    assert Fraction(float(s[3, 10])) == es and Fraction(float(z[3, 10])) == ez


@pytest.mark.parametrize("bits", [2, 3])
def test_constant_group_and_requantise(bits):
    w = np.full((2, 64), 0.03125, np.float32)
    w[1] = -0.0078125
    q, s, z = quant.wq_pack(w, bits)
    assert np.all(s == 1.0)
    assert np.array_equal(quant.wq_dequant(q, s, z, 64, bits), w)
    w = synthetic.randn_bf16((8, 256), 9, std=0.02).float().numpy()
    q, s, z = quant.wq_pack(w, bits)
    deq = quant.wq_dequant(q, s, z, 256, bits)
    sg = s[:, np.arange(256) // 64]
    zg = z[:, np.arange(256) // 64]
    again = np.clip(np.rint(deq / sg + zg), 0, 2 ** bits - 1)
    assert np.array_equal(again, quant.wq_unpack_codes(q, 256, bits))


def test_fewer_bits_larger_error():
    w = synthetic.randn_bf16((32, 512), 13, std=0.02).float().numpy()
    err = []
    for bits in (2, 3, 4):
        deq = quant.wq_dequant(*quant.wq_pack(w, bits), 512, bits)
        err.append(float(np.sqrt(np.mean((deq - w) ** 2))))
    assert err[0] > 1.8 * err[1] > 1.8 * 1.8 * err[2] * 0.9, err


@pytest.mark.parametrize("bits", [2, 3])
def test_gemm_identity_equals_dequant(bits):
    k = 128
    w = synthetic.randn_bf16((8, k), 11, std=0.02).float().numpy()
    q, s, z = quant.wq_pack(w, bits)
    y = quant.wq_gemm(np.eye(k, dtype=np.float32), q, s, z, k, bits)
    assert np.array_equal(y.T, quant.wq_dequant(q, s, z, k, bits))
