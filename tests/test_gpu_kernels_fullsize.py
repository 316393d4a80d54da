"""Kernel parity at the full sizes of the kernel sweep (Qwen2.5-32B layer
shapes): tree attention with 385 tree nodes (depth 48, width 8) over 4k and
16k committed keys, verify-shaped (every node a query, the node outputs
sampled and computed one by one by the oracle) and draft-shaped (the 8
deepest nodes, every output checked, the 16-way key split and its cluster
merge in play); the int4 product on the 32B gate+up (55296 x 5120) and down
(5120 x 27648, 432 groups) matrices at draft, four-tile GEMV and verify widths, sampled
output rows against the oracle's dequantisation."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import quant
from oracle.model import attention

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sub():
    import substitute_speculative_decoding_gb300 as s
    return s


def np32(t):
    return t.detach().float().cpu().numpy()


def close(got, ref, atol, rtol):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    assert np.all(err <= bound), f"max excess {np.max(err - bound):.3e}, max err {err.max():.3e}"


def _fill(kv_t, layer, positions, k_rows, v_rows, page_size):
    k, v, pt = kv_t
    pos = torch.as_tensor(positions, dtype=torch.int64, device=k.device)
    pages = pt.to(k.device).long()[pos // page_size]
    offs = pos % page_size
    k[layer, pages, :, offs, :] = k_rows
    v[layer, pages, :, offs, :] = v_rows


@pytest.mark.parametrize("n_prefix", [4096, 16384])
def test_tree_attn_fullsize(sub, n_prefix):
    hq, hkv, d, depth, width = 40, 8, 128, 48, 8
    seed = n_prefix
    tok, par, dep = synthetic.random_tree(depth, width, seed, 1000)
    anc = synthetic.ancestors(par, dep, depth)
    n = len(par)
    tree_base = n_prefix
    cap = tree_base + n + 64
    kv, kv_t = sub.make_kv(1, hkv, d, cap, page_size=64, shuffle_seed=seed)
    kp = synthetic.randn_bf16((n_prefix, hkv, d), seed + 1)
    vp = synthetic.randn_bf16((n_prefix, hkv, d), seed + 2)
    kt = synthetic.randn_bf16((n, hkv, d), seed + 3)
    vt = synthetic.randn_bf16((n, hkv, d), seed + 4)
    _fill(kv_t, 0, list(range(n_prefix)), kp.to(DEV), vp.to(DEV), 64)
    _fill(kv_t, 0, [tree_base + s for s in range(n)], kt.to(DEV), vt.to(DEV), 64)
    q = synthetic.randn_bf16((n, hq, d), seed + 5)
    ancd, depd = anc.to(DEV), dep.to(DEV)
    o_verify = np32(sub.tree_attn(q.to(DEV), kv, 0, n_prefix, tree_base, n, anc=ancd,
                                  depth=depd))
    o_draft = np32(sub.tree_attn(q[-width:].contiguous().to(DEV), kv, 0, n_prefix, tree_base, n,
                                 anc=ancd[-width:].contiguous(), depth=depd[-width:].contiguous()))
    torch.cuda.synchronize()
    kp64, vp64, kt64, vt64, q64 = np32(kp), np32(vp), np32(kt), np32(vt), np32(q)

    def oracle_row(u):
        path = [int(s) for s in anc[u] if s >= 0]
        kk = np.concatenate([kp64, kt64[path]])
        vv = np.concatenate([vp64, vt64[path]])
        return attention(q64[u:u + 1], kk, vv, np.ones((1, len(kk)), bool), hkv)[0]

    rng = np.random.default_rng(seed)
    sample = sorted({0, n - 1, *rng.choice(n, 22, replace=False).tolist()})
    for u in sample:
        close(o_verify[u], oracle_row(u), atol=2e-2, rtol=2 ** -7)
    for i, u in enumerate(range(n - width, n)):
        close(o_draft[i], oracle_row(u), atol=2e-2, rtol=2 ** -7)


@pytest.mark.parametrize("n,k", [(55296, 5120), (5120, 27648)])
@pytest.mark.parametrize("m", [1, 8, 32, 48, 385])
def test_w4_gemm_fullsize(sub, n, k, m):
    q, s, z = synthetic.random_w4(n, k, 3)
    x = synthetic.randn_bf16((m, k), 7 + m)
    y = np32(sub.w4_gemm(x.to(DEV), q.to(DEV), s.to(DEV), z.to(DEV), n, k))
    rows = np.sort(np.random.default_rng(n + m).choice(n, 64, replace=False))
    deq = quant.w4_dequant(q.numpy()[rows], np32(s)[rows], np32(z)[rows], k)
    ref = np32(x).astype(np.float64) @ deq.astype(np.float64).T
    scale = np.abs(ref).max()
    close(y[:, rows], ref, atol=3e-3 * scale, rtol=2 ** -8)
