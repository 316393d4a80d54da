"""Decoder forward of the target (and of the draft) over a set of rows with an
explicit visibility mask (test infrastructure only).

Architecture (the pages evaluate Qwen2.5-7B/14B/32B and Llama-3.1-8B; they give
no layer equations, so this is the plainest reading of a dense Llama/Qwen
decoder): pre-norm blocks, no biases,
  h  = bf16(RMSNorm(x) * gain)                 RMSNorm: x / sqrt(mean(x^2) + eps)
  q, k, v = h Wq^T, h Wk^T, h Wv^T             (fp32)
  q, k = RoPE(q, pos), RoPE(k, pos)            rotate-half, inv_freq_i = theta^(-2i/d)
  q, k, v -> bf16 (k, v are what the KV cache stores)
  o  = bf16(softmax(q K^T / sqrt(d)) V)        GQA: query head h reads KV head h // (Hq/Hkv)
  x  = x + o Wo^T                              (fp32 residual stream)
  h2 = bf16(RMSNorm(x) * gain2)
  a  = bf16(silu(h2 Wg^T) * (h2 Wu^T))
  x  = x + a Wd^T
then final RMSNorm -> bf16 -> untied lm_head -> fp32 logits.

The draft differs only in its weights: layers [0, R) are the target's own
bf16 layers (layer sharing) and layers [R, L) are the dequantised int4
substitutes ("Low-Bit Shadow" report, 2.2 Step 4 and 4.1 point 2;
"Speculate Deep and Accurate" abstract).  KV sharing -- the draft attends
over the target's committed KV -- is expressed by the caller passing the
target's cache as `past`.
"""
import numpy as np

from .bf16 import round_bf16, mm


def rmsnorm(x, gain, eps: float) -> np.ndarray:
    x64 = np.asarray(x, np.float64)
    r = 1.0 / np.sqrt(np.mean(x64 * x64, axis=-1, keepdims=True) + eps)
    return (x64 * r * np.asarray(gain, np.float64)).astype(np.float32)


def rope(x, pos, theta: float) -> np.ndarray:
    """x: [M, H, d] fp32, pos: [M] ints.  Rotate-half: element i pairs with
    element i + d/2 and the pair turns by angle pos * theta^(-2i/d)."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    half = d // 2
    inv = theta ** (-(np.arange(half, dtype=np.float64) * 2.0) / d)
    ang = np.asarray(pos, np.float64)[:, None] * inv[None, :]          # [M, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1).astype(np.float32)


def attention(q, k, v, vis, n_heads_kv: int) -> np.ndarray:
    """q: [M, Hq, d], k, v: [S, Hkv, d], vis: [M, S] bool (row m may read key s).
    Returns [M, Hq, d] fp32: softmax over visible keys in float64."""
    m, hq, d = q.shape
    group = hq // n_heads_kv
    out = np.zeros((m, hq, d), dtype=np.float64)
    q64 = np.asarray(q, np.float64)
    k64 = np.asarray(k, np.float64)
    v64 = np.asarray(v, np.float64)
    scale = 1.0 / np.sqrt(d)
    for h in range(hq):
        kh = k64[:, h // group, :]
        vh = v64[:, h // group, :]
        sc = (q64[:, h, :] @ kh.T) * scale                 # [M, S]
        sc = np.where(vis, sc, -np.inf)
        sc = sc - sc.max(axis=1, keepdims=True)
        p = np.exp(sc)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ vh
    return out.astype(np.float32)


def silu_mul(g, u) -> np.ndarray:
    g64 = np.asarray(g, np.float64)
    return (g64 / (1.0 + np.exp(-g64)) * np.asarray(u, np.float64)).astype(np.float32)


def forward_rows(cfg, glob, layers, tokens, pos, past_k, past_v, past_vis, self_vis):
    """Run the decoder on M rows.

    tokens, pos : [M] ints
    layers      : list of per-layer weight dicts (float32 arrays of bf16 values)
    past_k/v    : per layer [P, Hkv, d] bf16-valued keys/values already cached
    past_vis    : [M, P] bool, row m may read cached key p
    self_vis    : [M, M] bool, row m may read the key of row m' (self included)
    Returns (logits fp32 [M, V], new_k, new_v per layer [M, Hkv, d]).
    """
    tokens = np.asarray(tokens, np.int64)
    m = tokens.shape[0]
    x = np.asarray(glob["embed"], np.float32)[tokens].copy()
    new_k, new_v = [], []
    vis = np.concatenate([np.asarray(past_vis, bool).reshape(m, -1),
                          np.asarray(self_vis, bool)], axis=1)
    for li, w in enumerate(layers):
        h = round_bf16(rmsnorm(x, w["attn_norm"], cfg.rms_eps))
        q = mm(h, w["wq"]).reshape(m, cfg.n_heads_q, cfg.head_dim)
        k = mm(h, w["wk"]).reshape(m, cfg.n_heads_kv, cfg.head_dim)
        v = mm(h, w["wv"]).reshape(m, cfg.n_heads_kv, cfg.head_dim)
        q = round_bf16(rope(q, pos, cfg.rope_theta))
        k = round_bf16(rope(k, pos, cfg.rope_theta))
        v = round_bf16(v)
        kk = np.concatenate([past_k[li].reshape(-1, cfg.n_heads_kv, cfg.head_dim), k], axis=0)
        vv = np.concatenate([past_v[li].reshape(-1, cfg.n_heads_kv, cfg.head_dim), v], axis=0)
        o = round_bf16(attention(q, kk, vv, vis, cfg.n_heads_kv)).reshape(m, -1)
        x = x + mm(o, w["wo"])
        h2 = round_bf16(rmsnorm(x, w["ffn_norm"], cfg.rms_eps))
        a = round_bf16(silu_mul(mm(h2, w["wg"]), mm(h2, w["wu"])))
        x = x + mm(a, w["wd"])
        new_k.append(k)
        new_v.append(v)
    hf = round_bf16(rmsnorm(x, glob["final_norm"], cfg.rms_eps))
    logits = mm(hf, glob["lm_head"])
    return logits, new_k, new_v


def empty_kv(cfg):
    z = np.zeros((0, cfg.n_heads_kv, cfg.head_dim), np.float32)
    return [z] * cfg.n_layers, [z] * cfg.n_layers


def prefill(cfg, glob, layers, prompt):
    """Causal forward of the prompt; returns (logits [P, V], K, V caches)."""
    p = len(prompt)
    pk, pv = empty_kv(cfg)
    causal = np.tril(np.ones((p, p), bool))
    return forward_rows(cfg, glob, layers, prompt, np.arange(p), pk, pv,
                        np.zeros((p, 0), bool), causal)
