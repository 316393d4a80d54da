"""Pins of the oracle's decoder pieces: closed forms of RMSNorm, RoPE, SiLU
and masked attention, the GQA head mapping, and the causal-cache property
(incremental decoding with a KV cache equals recomputing the whole sequence)."""
import numpy as np

from oracle import model as om
from oracle.model import forward_rows, prefill
import synthetic
from helpers import oracle_model


def test_rmsnorm_closed_forms():
    x = np.full((1, 8), 3.0, np.float32)
    y = om.rmsnorm(x, np.ones(8), 0.0)
    assert np.allclose(y, 1.0, rtol=0, atol=1e-7)
    eps = 1e-6
    y = om.rmsnorm(x, np.full(8, 2.0), eps)
    assert np.allclose(y, 2 * 3 / np.sqrt(9 + eps), atol=1e-7)
    r = np.random.default_rng(0).standard_normal((4, 256)).astype(np.float32)
    y = om.rmsnorm(r, np.ones(256), 0.0)
    assert np.allclose(np.sqrt((y.astype(np.float64) ** 2).mean(-1)), 1.0, atol=1e-6)


def test_rope_closed_forms():
    d = 8
    x = np.zeros((1, 1, d), np.float32)
    x[0, 0, 0] = 1.0
    p = 5
    y = om.rope(x, [p], 10000.0)
    # element 0 pairs with element d/2 and turns by p * theta^0 = p radians
    assert np.isclose(y[0, 0, 0], np.cos(p), atol=1e-7)
    assert np.isclose(y[0, 0, d // 2], np.sin(p), atol=1e-7)
    assert np.allclose(np.delete(y[0, 0], [0, d // 2]), 0)
    # element 1 pairs with d/2+1 and turns by p * theta^(-2/d)
    x = np.zeros((1, 1, d), np.float32)
    x[0, 0, 1] = 1.0
    y = om.rope(x, [p], 10000.0)
    ang = p * 10000.0 ** (-2.0 / d)
    assert np.isclose(y[0, 0, 1], np.cos(ang), atol=1e-7)
    assert np.isclose(y[0, 0, d // 2 + 1], np.sin(ang), atol=1e-7)


def test_rope_identity_norm_and_relative_position():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 2, 64)).astype(np.float32)
    k = rng.standard_normal((1, 2, 64)).astype(np.float32)
    assert np.allclose(om.rope(q, [0], 1e4), q)
    qq = om.rope(q, [37], 1e4)
    assert np.allclose(np.linalg.norm(qq, axis=-1), np.linalg.norm(q, axis=-1), rtol=1e-6)
    # <rope(q, m), rope(k, n)> depends only on m - n
    a = (om.rope(q, [50], 1e4) * om.rope(k, [20], 1e4)).sum(-1)
    b = (om.rope(q, [130], 1e4) * om.rope(k, [100], 1e4)).sum(-1)
    assert np.allclose(a, b, atol=1e-5)


def test_silu_mul_closed_forms():
    assert om.silu_mul(np.zeros(3), np.ones(3)).tolist() == [0, 0, 0]
    assert np.isclose(om.silu_mul(np.array([30.0]), np.array([2.0]))[0], 60.0)
    assert np.isclose(om.silu_mul(np.array([1.0]), np.array([1.0]))[0], 1 / (1 + np.exp(-1)))


def test_attention_closed_forms_and_gqa():
    rng = np.random.default_rng(2)
    hq, hkv, d, s = 4, 2, 16, 5
    q = rng.standard_normal((3, hq, d)).astype(np.float32)
    # each KV head's values are a constant that names the head
    k = rng.standard_normal((s, hkv, d)).astype(np.float32)
    v = np.zeros((s, hkv, d), np.float32)
    v[:, 0, :] = 1.0
    v[:, 1, :] = 2.0
    vis = np.ones((3, s), bool)
    o = om.attention(q, k, v, vis, hkv)
    assert np.allclose(o[:, 0:2], 1.0) and np.allclose(o[:, 2:4], 2.0)
    # a single visible key returns its value
    v2 = rng.standard_normal((s, hkv, d)).astype(np.float32)
    vis1 = np.zeros((3, s), bool)
    vis1[:, 3] = True
    o = om.attention(q, k, v2, vis1, hkv)
    assert np.allclose(o[:, 1], v2[3, 0]) and np.allclose(o[:, 3], v2[3, 1])
    # a zero query weighs visible keys uniformly
    o = om.attention(np.zeros_like(q), k, v2, vis, hkv)
    assert np.allclose(o[0, 0], v2[:, 0].mean(0), atol=1e-6)


def test_incremental_cache_equals_full_recompute():
    cfg = synthetic.CONFIGS["tiny"]
    m = synthetic.make_model(cfg, norm_gain_std=0.1)
    glob, layers = oracle_model(m)
    prompt = synthetic.make_prompt(cfg, n=12).numpy()
    full, ks, vs = prefill(cfg, glob, layers, prompt)
    head, hk, hv = prefill(cfg, glob, layers, prompt[:9])
    # rows 9..11 one at a time through the cache
    for i in range(9, 12):
        lg, nk, nv = forward_rows(cfg, glob, layers, [prompt[i]], [i], hk, hv,
                                  np.ones((1, i), bool), np.ones((1, 1), bool))
        assert np.allclose(lg[0], full[i], atol=1e-5, rtol=1e-5)
        hk = [np.concatenate([a, b]) for a, b in zip(hk, nk)]
        hv = [np.concatenate([a, b]) for a, b in zip(hv, nv)]
    for a, b in zip(hk, ks):
        assert np.array_equal(a, b)
