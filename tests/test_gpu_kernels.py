"""Kernel parity: each CUDA entry point against the oracle on the same seeded
inputs.  Bit-exact for the quantiser, dequantisation, tree topology, choices,
accepted paths and KV copies; floating-point products within a tolerance
derived from bf16 output rounding plus fp32 accumulation order."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import quant, tree as otree
from oracle.bf16 import round_bf16

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
    assert np.all(err <= bound), f"max excess {np.max(err - bound):.3e} (max err {err.max():.3e})"


# ---------------------------------------------------------------- int4 --
@pytest.mark.parametrize("n,k", [(48, 688), (64, 3584), (16, 64), (40, 200)])
def test_w4_pack_and_dequant_bit_exact(sub, n, k):
    w = synthetic.randn_bf16((n, k), n * 7 + k, std=0.02)
    w[3, :64] = 0.25                       # a constant group
    q, s, z = sub.w4_pack(w.to(DEV))
    rq, rs, rz = quant.w4_pack(np32(w))
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(np32(s), rs) and np.array_equal(np32(z), rz)
    deq = sub.w4_dequant(q, s, z, k)
    assert np.array_equal(np32(deq), quant.w4_dequant(rq, rs, rz, k))


@pytest.mark.parametrize("m", [1, 3, 8, 13, 16, 17, 48, 130, 385])
@pytest.mark.parametrize("n,k", [(256, 688), (4608, 3584), (96, 512)])
def test_w4_gemm(sub, m, n, k):
    w = synthetic.randn_bf16((n, k), 3 + n + k, std=0.02)
    q, s, z = sub.w4_pack(w.to(DEV))
    x = synthetic.randn_bf16((m, k), 11 + m + k)
    y = sub.w4_gemm(x.to(DEV), q, s, z, n, k)
    ref = quant.w4_gemm(np32(x), q.cpu().numpy(), np32(s), np32(z), k)
    # bf16 output rounding (2^-8 relative) + the GEMV's unrounded dequant
    # (|deq - (q-z)s| <= 2^-9 |deq| per weight, random signs: sqrt(K) growth)
    scale = np.abs(ref).max()
    close(np32(y), ref, atol=3e-3 * scale, rtol=2 ** -8)


def test_w4_gemm_identity_is_exact_dequant(sub):
    k = 256
    w = synthetic.randn_bf16((64, k), 5, std=0.02)
    q, s, z = sub.w4_pack(w.to(DEV))
    eye = torch.eye(k, dtype=torch.bfloat16, device=DEV)
    y = sub.w4_gemm(eye, q, s, z, 64, k)          # M = 256: tiled kernel
    assert torch.equal(y.t().contiguous(), sub.w4_dequant(q, s, z, k))
    y16 = sub.w4_gemm(eye[:16].contiguous(), q, s, z, 64, k)   # GEMV kernel
    assert torch.equal(y16.t().contiguous(), sub.w4_dequant(q, s, z, k)[:, :16])


def test_w4_wide_gemv_rows_match_narrow(sub):
    """Up to 32 rows an int4 product with a bf16 output stays on the TMA GEMV
    (four token tiles of 8 past 16 rows): a row's result is the same, bit for
    bit, whether it shares the pass with 7 or 31 other rows; identity rows give
    the dequantised values exactly, on the GEMV and past 32 rows on the
    tensor-core GEMM."""
    n, k = 640, 1024
    w = synthetic.randn_bf16((n, k), 31, std=0.02)
    q, s, z = sub.w4_pack(w.to(DEV))
    x = synthetic.randn_bf16((48, k), 33).to(DEV)
    y32 = sub.w4_gemm(x[:32].contiguous(), q, s, z, n, k)
    y24 = sub.w4_gemm(x[:24].contiguous(), q, s, z, n, k)
    y8 = sub.w4_gemm(x[:8].contiguous(), q, s, z, n, k)
    assert torch.equal(y32[:24], y24) and torch.equal(y32[:8], y8)
    deq = sub.w4_dequant(q, s, z, k)
    eye = torch.eye(k, dtype=torch.bfloat16, device=DEV)
    for r0, m in ((0, 48), (48, 40), (88, 24)):
        y = sub.w4_gemm(eye[r0:r0 + m].contiguous(), q, s, z, n, k)
        assert torch.equal(y.t().contiguous(), deq[:, r0:r0 + m])


@pytest.mark.parametrize("m", [1, 8, 16, 17, 385])
@pytest.mark.parametrize("n,k", [(1024, 256), (512, 3584), (144, 688)])
def test_bf16_gemm(sub, m, n, k):
    w = synthetic.randn_bf16((n, k), 21 + n, std=0.02)
    x = synthetic.randn_bf16((m, k), 23 + m)
    y = sub.bf16_gemm(x.to(DEV), w.to(DEV))
    ref = np32(x).astype(np.float64) @ np32(w).astype(np.float64).T
    close(np32(y), ref, atol=1e-4 * np.abs(ref).max(), rtol=2 ** -8)


def test_bf16_gemm_rows_independent_of_m(sub):
    """A row's result is the same whether it is computed alone in the tiled
    kernel's tile or with 384 other rows (no M-dependent split)."""
    k, n = 512, 256
    w = synthetic.randn_bf16((n, k), 1, std=0.02).to(DEV)
    x = synthetic.randn_bf16((385, k), 2).to(DEV)
    y_all = sub.bf16_gemm(x, w)
    y_17 = sub.bf16_gemm(x[100:117].contiguous(), w)
    assert torch.equal(y_all[100:117], y_17)


# ----------------------------------------------------------- attention --
def _fill_cache(sub, kv_t, layer, positions, k_rows, v_rows, page_size):
    k, v, pt = kv_t
    for i, p in enumerate(positions):
        page = int(pt[p // page_size])
        k[layer, page, :, p % page_size, :] = k_rows[i]
        v[layer, page, :, p % page_size, :] = v_rows[i]


@pytest.mark.parametrize("hq,hkv,d,n_prefix,depth,width", [
    (4, 2, 64, 37, 3, 2), (28, 4, 128, 130, 6, 3), (8, 8, 64, 0, 4, 2), (40, 8, 128, 515, 8, 8),
    (4, 1, 128, 64, 2, 1)])
def test_tree_attn_matches_per_path_attention(sub, hq, hkv, d, n_prefix, depth, width):
    seed = hq + d + n_prefix
    tok, par, dep = synthetic.random_tree(depth, width, seed, 100)
    anc = synthetic.ancestors(par, dep, depth)
    n = len(par)
    tree_base = n_prefix + 5
    cap = tree_base + n + 70
    kv, kv_t = sub.make_kv(2, hkv, d, cap, page_size=64, shuffle_seed=seed)
    kp = synthetic.randn_bf16((n_prefix, hkv, d), seed + 1)
    vp = synthetic.randn_bf16((n_prefix, hkv, d), seed + 2)
    kt = synthetic.randn_bf16((n, hkv, d), seed + 3)
    vt = synthetic.randn_bf16((n, hkv, d), seed + 4)
    _fill_cache(sub, kv_t, 1, list(range(n_prefix)), kp.to(DEV), vp.to(DEV), 64)
    _fill_cache(sub, kv_t, 1, [tree_base + s for s in range(n)], kt.to(DEV), vt.to(DEV), 64)
    q = synthetic.randn_bf16((n, hq, d), seed + 5)
    o = sub.tree_attn(q.to(DEV), kv, 1, n_prefix, tree_base, n, anc=anc.to(DEV),
                      depth=dep.to(DEV))
    ref = otree.tree_attention(np32(q), np32(kp), np32(vp), np32(kt), np32(vt), par.numpy(), hkv)
    # P is rounded to bf16 before P.V and O to bf16: ~2^-8 relative
    close(np32(o), ref, atol=2e-2, rtol=2 ** -7)


def test_tree_attn_chain_is_causal(sub):
    from oracle.model import attention
    hq, hkv, d, n = 4, 2, 64, 150
    kv, kv_t = sub.make_kv(1, hkv, d, 256)
    kk = synthetic.randn_bf16((n, hkv, d), 1)
    vv = synthetic.randn_bf16((n, hkv, d), 2)
    _fill_cache(sub, kv_t, 0, list(range(n)), kk.to(DEV), vv.to(DEV), 64)
    q = synthetic.randn_bf16((n, hq, d), 3)
    o = sub.tree_attn(q.to(DEV), kv, 0, 0, 0, n)
    ref = attention(np32(q), np32(kk), np32(vv), np.tril(np.ones((n, n), bool)), hkv)
    close(np32(o), ref, atol=2e-2, rtol=2 ** -7)


# --------------------------------------------------------------- tree --
@pytest.mark.parametrize("width,vocab,depth", [(2, 1024, 4), (8, 152064, 3), (3, 5000, 3),
                                               (16, 2048, 2)])
def test_draft_expand_teacher_forced(sub, width, vocab, depth):
    """Expansion on the same logits: topology bit-exact, scores close."""
    tr = sub.DeviceTree(depth, width, DEV)
    tr.token[0] = 5
    rng = np.random.default_rng(width + vocab)
    o_tok, o_par, o_score = [5], [-1], [0.0]
    for lvl in range(depth):
        kp = 1 if lvl == 0 else width
        lg = (rng.standard_normal((kp, vocab)) * 2.0).astype(np.float32)
        lg[0, 7] = lg[0, 9] = lg[0].max() + 0.5          # an exact tie inside a row
        sub.draft_expand(torch.tensor(lg, device=DEV), 0.2, tr, lvl)
        s0 = 0 if lvl == 0 else 1 + (lvl - 1) * width
        frontier = list(range(s0, s0 + kp))
        tok, par, sc = otree.expand_level(lg, [o_score[u] for u in frontier], frontier, width, 0.2)
        o_tok += tok.tolist()
        o_par += par.tolist()
        o_score += sc.tolist()
    torch.cuda.synchronize()
    n = 1 + depth * width
    assert tr.token.cpu().tolist() == o_tok[:n]
    assert tr.parent.cpu().tolist() == o_par[:n]
    assert np.allclose(tr.score.cpu().numpy(), np.array(o_score[:n]), atol=1e-3)
    dep = tr.depth.cpu().numpy()
    assert np.array_equal(dep, otree.depth_of(np.array(o_par[:n])))
    anc = synthetic.ancestors(torch.tensor(o_par[:n]), torch.tensor(dep), depth)
    assert torch.equal(tr.anc.cpu(), anc)


@pytest.mark.parametrize("mode,vocab", [(0, 1024), (1, 1024), (0, 152064), (1, 152064)])
def test_verify_accept_bit_exact(sub, mode, vocab):
    depth, width = 6, 3
    tok, par, dep = synthetic.random_tree(depth, width, 4, vocab)
    n = len(par)
    rng = np.random.default_rng(mode + vocab)
    lg = (rng.standard_normal((n, vocab)) * 3).astype(np.float32)
    # plant a matching chain along the root path of a deepest node, so that
    # at least three nodes are accepted
    path = [n - 1]
    while par[path[-1]] >= 0:
        path.append(int(par[path[-1]]))
    path = path[::-1]
    for u, c in zip(path[:3], path[1:4]):
        lg[u, tok[c]] = lg[u].max() + (5.0 if mode == 0 else 40.0)
    tr = sub.DeviceTree(depth, width, DEV)
    tr.token.copy_(tok)
    tr.parent.copy_(par)
    tr.depth.copy_(dep)
    root_pos = 77
    acc, na, bonus, choice = sub.verify_accept(torch.tensor(lg, device=DEV), tr, n, mode=mode,
                                               temperature=0.6, seed=7, root_pos=root_pos)
    sc = otree.choice_scores(lg, "greedy" if mode == 0 else "gumbel", 0.6, 7,
                             root_pos + dep.numpy() + 1)
    ref_choice = otree.argmax_first(sc)
    got = choice.cpu().numpy()
    # compare choices away from near-ties of the float64 oracle scores
    srt = np.sort(sc, axis=1)
    gap = srt[:, -1] - srt[:, -2]
    ok = gap >= 1e-4
    assert np.array_equal(got[ok], ref_choice[ok])
    ref_acc, ref_bonus = otree.accept_walk(tok.numpy(), par.numpy(), got)
    a = int(na.item())
    assert a == len(ref_acc) and a >= 3
    assert acc[:a].cpu().tolist() == ref_acc and int(bonus.item()) == ref_bonus


def test_kv_compact_in_place(sub):
    hkv, d, layers = 4, 128, 3
    cap = 600
    kv, (k, v, pt) = sub.make_kv(layers, hkv, d, cap, page_size=64, shuffle_seed=3)
    k.copy_(torch.randn_like(k, dtype=torch.float32).to(torch.bfloat16))
    v.copy_(torch.randn_like(v, dtype=torch.float32).to(torch.bfloat16))
    root = 130
    # a path whose destinations overwrite later sources: slot 2 at depth 1
    slots = [2, 9, 17, 26]
    acc = torch.tensor(slots + [0] * 4, dtype=torch.int32, device=DEV)
    na = torch.tensor([len(slots)], dtype=torch.int32, device=DEV)

    def rows(t, positions):
        return torch.stack([t[:, pt[p // 64], :, p % 64, :] for p in positions], 1).clone()

    want_k = rows(k, [root + s for s in slots])
    want_v = rows(v, [root + s for s in slots])
    keep = rows(k, [root - 1, root])
    sub.kv_compact(kv, root, acc, na, 8)
    torch.cuda.synchronize()
    assert torch.equal(rows(k, [root + 1 + j for j in range(len(slots))]), want_k)
    assert torch.equal(rows(v, [root + 1 + j for j in range(len(slots))]), want_v)
    assert torch.equal(rows(k, [root - 1, root]), keep)
