"""Pins of the oracle's tree logic: the two-stage expansion equals a brute-force
top-k over every (parent, token) candidate, the accept walk equals a brute-force
search over all root paths, tree attention equals per-path causal attention,
and log-softmax normalises."""
import itertools

import numpy as np
import pytest

from oracle import tree as ot
import synthetic


def test_log_softmax_normalises():
    z = np.random.default_rng(0).standard_normal((3, 50)) * 4
    lp = ot.log_softmax_t(z, 0.2)
    assert np.allclose(np.exp(lp).sum(-1), 1.0)
    # T scales the logits before normalising
    assert np.allclose(lp[0] - lp[0].max(), (z[0] - z[0].max()) / 0.2)


@pytest.mark.parametrize("k_prev,k,vocab,seed", [(1, 2, 7, 0), (2, 2, 9, 1), (3, 4, 11, 2),
                                                  (4, 3, 6, 3), (8, 8, 40, 4)])
def test_expand_equals_bruteforce(k_prev, k, vocab, seed):
    rng = np.random.default_rng(seed)
    # coarse logits so that ties occur, both within and across parents
    logits = rng.integers(-3, 3, (k_prev, vocab)).astype(np.float64)
    score = rng.integers(-2, 1, k_prev).astype(np.float64) * 0.5
    slots = np.arange(5, 5 + k_prev)
    tok, par, sc = ot.expand_level(logits, score, slots, k, 0.2)
    lp = ot.log_softmax_t(logits, 0.2)
    allc = [(score[j] + lp[j, v], slots[j], v) for j in range(k_prev) for v in range(vocab)]
    # brute force: the best k of all k_prev*V candidates under the same order
    allc.sort(key=lambda c: (-c[0], c[1], c[2]))
    best = allc[:k]
    assert [c[2] for c in best] == tok.tolist()
    assert [c[1] for c in best] == par.tolist()
    assert np.allclose([c[0] for c in best], sc)
    # siblings are distinct tokens
    for p in set(par.tolist()):
        t = tok[par == p]
        assert len(set(t.tolist())) == len(t)


def test_expand_descending_and_temperature():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((3, 30))
    tok, par, sc = ot.expand_level(logits, [0.0, -0.1, -0.3], [1, 2, 3], 5, 0.2)
    assert np.all(np.diff(sc) <= 0)
    # one parent: the children are that parent's own top-k at any temperature
    for t in (0.05, 0.2, 1.0, 3.0):
        tok1, _, _ = ot.expand_level(logits[:1], [0.0], [0], 5, t)
        assert tok1.tolist() == np.argsort(-logits[0], kind="stable")[:5].tolist()


def _all_paths(parent):
    n = len(parent)
    kids = {u: [c for c in range(n) if parent[c] == u] for u in range(n)}
    stack = [[0]]
    while stack:
        p = stack.pop()
        yield p
        for c in kids[p[-1]]:
            stack.append(p + [c])


@pytest.mark.parametrize("seed", range(6))
def test_accept_walk_equals_bruteforce(seed):
    depth, width, vocab = 4, 3, 5
    tok, par, dep = synthetic.random_tree(depth, width, seed, vocab)
    tok, par = tok.numpy(), par.numpy()
    rng = np.random.default_rng(seed)
    choice = rng.integers(0, vocab, len(tok))
    # make some matches likely: copy a child's token into the parent's choice
    for u in range(len(tok)):
        kids = np.nonzero(par == u)[0]
        if len(kids) and rng.random() < 0.7:
            choice[u] = tok[rng.choice(kids)]
    acc, bonus = ot.accept_walk(tok, par, choice)
    best = [0]
    for p in _all_paths(par):
        if all(tok[p[i + 1]] == choice[p[i]] for i in range(len(p) - 1)) and len(p) > len(best):
            best = p
    assert [0] + acc == best
    assert bonus == choice[best[-1]]
    assert 0 <= len(acc) <= depth


def test_tree_attention_equals_per_path_causal_attention():
    """Each node of a verify pass reads prefix + its own root path, which is
    what causal attention over the sequence prefix || path computes for the
    path's last token ("Low-Bit Shadow" report 6.3, tree verification)."""
    from oracle.model import attention
    rng = np.random.default_rng(3)
    hq, hkv, d, p = 4, 2, 8, 6
    tok, par, dep = synthetic.random_tree(3, 2, 1, 50)
    par = par.numpy()
    n = len(par)
    q = rng.standard_normal((n, hq, d)).astype(np.float32)
    kp, vp = rng.standard_normal((2, p, hkv, d)).astype(np.float32)
    kt, vt = rng.standard_normal((2, n, hkv, d)).astype(np.float32)
    got = ot.tree_attention(q, kp, vp, kt, vt, par, hkv)
    # masked-matrix form over [prefix | all tree slots]
    vis = np.concatenate([np.ones((n, p), bool), ot.ancestor_mask(par)], axis=1)
    alt = attention(q, np.concatenate([kp, kt]), np.concatenate([vp, vt]), vis, hkv)
    assert np.allclose(got, alt, atol=1e-6)
    # sequence form: build prefix || path as a causal sequence for one leaf
    leaf = n - 1
    path = []
    u = leaf
    while u >= 0:
        path.append(u)
        u = par[u]
    path = path[::-1]
    kk = np.concatenate([kp, kt[path]])
    vv = np.concatenate([vp, vt[path]])
    qs = np.zeros((len(path), hq, d), np.float32)
    qs[-1] = q[leaf]
    causal = np.tril(np.ones((len(path), p + len(path)), bool), k=p)
    seq = attention(qs, kk, vv, causal, hkv)
    assert np.allclose(seq[-1], got[leaf], atol=1e-6)


def test_ancestor_mask_and_depth():
    tok, par, dep = synthetic.random_tree(5, 3, 2, 100)
    par = par.numpy()
    m = ot.ancestor_mask(par)
    assert np.array_equal(m.sum(1), dep.numpy() + 1)
    assert np.array_equal(ot.depth_of(par), dep.numpy())
