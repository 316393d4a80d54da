"""Pins of the oracle's HQQ zero optimisation (the pages' quantiser, "Low-Bit
Shadow" report Critique 3, 6.2; restated from the published half-quadratic
method): one iteration is the min-max quantiser exactly; groups on an exact
grid are fixed points; the shrinkage at p = 1 is textbook soft-thresholding;
the zero step minimises its quadratic; the kept zero never has a larger
sum |r| than the min-max zero; short groups ignore their padding; the fixed
summation order is a plain sum up to rounding; and the optimisation lowers
the dequantisation error on random groups."""
import numpy as np
import pytest

from oracle import quant
import synthetic


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_one_iteration_is_min_max(bits):
    w = synthetic.randn_bf16((64, 200), 3 + bits, std=0.02).float().numpy()
    a = quant.hqq_codes(w, bits, iters=1)
    b = quant.wq_codes(w, bits)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_grid_group_is_a_fixed_point(bits):
    L = 2 ** bits - 1
    m = (L + 1) // 2
    c = (np.arange(64) * 5) % (L + 1)
    w = ((c - m) * 2.0 ** -6).astype(np.float32)[None, :]
    codes, s, z = quant.hqq_codes(w, bits)
    assert s[0, 0] == 2.0 ** -6 and z[0, 0] == float(m)
    assert np.array_equal(codes[0], c)


def test_shrink_at_p1_is_soft_thresholding_and_p_half_closed_form():
    r = np.array([-0.5, -0.01, 0.0, 0.003, 0.2, 1.5], np.float32)
    beta = 20.0
    soft = np.sign(r) * np.maximum(np.abs(r) - 1 / beta, 0)
    assert np.allclose(quant.shrink_lp(r, beta, p=1.0), soft, rtol=0, atol=1e-7)
    ar = np.abs(r.astype(np.float64))
    half = np.sign(r) * np.maximum(ar - np.where(ar > 0, ar ** -0.5, 0) / beta, 0)
    assert np.allclose(quant.shrink_lp(r, beta, p=0.5), half, rtol=1e-6, atol=1e-9)


def test_zero_step_minimises_its_quadratic():
    rng = np.random.default_rng(1)
    w = synthetic.randn_bf16((1, 64), 7, std=0.02).float().numpy()[0].astype(np.float64)
    s = 0.004
    q = np.clip(np.rint(w / s + 4.0), 0, 15)
    e = rng.standard_normal(64) * 1e-4
    z = np.mean(q - (w - e) / s)                 # the update the oracle forms

    def obj(zz):
        return np.sum((w - e - s * (q - zz)) ** 2)
    for d in (1e-3, -1e-3, 1e-1, -1e-1):
        assert obj(z + d) > obj(z)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_kept_zero_not_worse_than_min_max(bits):
    """The kept zero is no worse in sum |r| than the min-max zero (iteration 0
    is a candidate); after both are rounded to bf16 that holds up to the
    rounding's effect, at most 64 * s * ulp(z) / 2 per group."""
    w = synthetic.randn_bf16((256, 64), 11 + bits, std=0.02).float().numpy()
    L = np.float32(2 ** bits - 1)
    codes, s, z_h = quant.hqq_codes(w, bits)
    _, s0, z_0 = quant.wq_codes(w, bits)
    assert np.array_equal(s, s0)
    s, z_h, z_0 = s[:, 0].astype(np.float64), z_h[:, 0].astype(np.float64), z_0[:, 0]

    def l1(z):
        q = np.clip(np.rint(w / s[:, None] + z[:, None]), 0, L)
        return np.abs(w - s[:, None] * (q - z[:, None])).sum(1)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(z_h), 1e-30))) - 7)
    assert np.all(l1(z_h) <= l1(z_0.astype(np.float64)) + 64 * s * ulp)
    assert np.mean(l1(z_h)) < np.mean(l1(z_0.astype(np.float64)))


def test_short_group_ignores_padding():
    w = synthetic.randn_bf16((8, 112), 5, std=0.02).float().numpy()   # groups of 64 and 48
    codes, s, z = quant.hqq_codes(w, 3)
    c2, s2, z2 = quant.hqq_codes(w[:, 64:].copy(), 3)                 # the 48 alone
    assert np.array_equal(codes[:, 64:], c2)
    assert np.array_equal(s[:, 1], s2[:, 0]) and np.array_equal(z[:, 1], z2[:, 0])


def test_pair_sum_is_a_sum():
    x = np.random.default_rng(3).standard_normal((16, 64)).astype(np.float32)
    assert np.allclose(quant.pair_sum64(x), x.astype(np.float64).sum(1), rtol=0, atol=1e-5)
    assert quant.pair_sum64(np.arange(64, dtype=np.float32)[None])[0] == 2016.0


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_lowers_the_error_on_random_groups(bits):
    w = synthetic.randn_bf16((2048, 64), 1, std=0.02).float().numpy()
    q, s, z = quant.wq_pack_hqq(w, bits)
    q0, s0, z0 = quant.wq_pack(w, bits)
    e_h = np.abs(quant.wq_dequant(q, s, z, 64, bits) - w).mean()
    e_0 = np.abs(quant.wq_dequant(q0, s0, z0, 64, bits) - w).mean()
    assert e_h < 0.98 * e_0, (e_h, e_0)
