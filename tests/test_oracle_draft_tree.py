"""Pin of the oracle's draft-tree construction at widths k > 1.

With the draft equal to the target (every substitute replaced by its
original: the "self" draft of the "Low-Bit Shadow" report, 3.x), the draft's
forward at a tree node u sees the committed prefix plus the draft KV of u's
root path, which is then the target's own KV of that path.  So the draft
logits at u must equal the target's logits at u from the one-pass tree
verification ("Low-Bit Shadow" report 6.3, SpecInfer: tree verification is
per-path causal attention), up to float64 summation order.  A draft that let a
node read the draft KV of slots that are not its ancestors (cousins drafted on
earlier levels) breaks this equality; the planted-mistake test below shows
that the pin catches exactly that mistake.

Also pinned: the tree's shape -- every level keeps k slots whose parents are on
the level above, depth = parent depth + 1, and siblings carry distinct tokens.
"""
import numpy as np
import pytest

import synthetic
from oracle import decode, tree
from oracle.model import prefill
from helpers import oracle_model

CFG = synthetic.CONFIGS["tiny"]


@pytest.fixture(scope="module")
def tiny():
    m = synthetic.make_model(CFG, norm_gain_std=0.1)
    glob, layers = oracle_model(m)
    prompt = synthetic.make_prompt(CFG).numpy()
    _, ks, vs = prefill(CFG, glob, layers, prompt)
    return glob, layers, prompt, ks, vs


def _slot_of(level, i, width):
    """Slot of the i-th frontier row drafted at `level` (0 = the root)."""
    return 0 if level == 0 else 1 + (level - 1) * width + i


def _draft_and_verify(tiny, depth, width, root_token=5):
    glob, layers, prompt, ks, vs = tiny
    n = len(prompt)
    tok, par, dep, dl = decode.draft_tree(CFG, glob, layers, root_token, n, ks, vs, depth, width,
                                          0.2)
    lg, _, _ = decode.verify_tree(CFG, glob, layers, tok, par, dep, n, ks, vs)
    return tok, par, dep, dl, lg


@pytest.mark.parametrize("depth,width", [(3, 2), (5, 2), (3, 3), (5, 3)])
def test_self_draft_logits_equal_tree_verify_logits(tiny, depth, width):
    tok, par, dep, dl, lg = _draft_and_verify(tiny, depth, width)
    assert len(dl) == depth
    for level, rows in enumerate(dl):
        assert rows.shape == ((1 if level == 0 else width), CFG.vocab)
        for i in range(rows.shape[0]):
            u = _slot_of(level, i, width)
            assert dep[u] == level
            np.testing.assert_allclose(rows[i], lg[u], rtol=1e-5, atol=1e-5,
                                       err_msg=f"slot {u} (level {level})")


@pytest.mark.parametrize("depth,width", [(4, 2), (3, 3)])
def test_tree_shape(tiny, depth, width):
    tok, par, dep, _, _ = _draft_and_verify(tiny, depth, width)
    assert len(tok) == 1 + depth * width
    assert par[0] == -1 and dep[0] == 0
    for level in range(1, depth + 1):
        lo, hi = 1 + (level - 1) * width, 1 + level * width
        prev = (0, 1) if level == 1 else (1 + (level - 2) * width, 1 + (level - 1) * width)
        for u in range(lo, hi):
            assert prev[0] <= par[u] < prev[1]
            assert dep[u] == dep[par[u]] + 1 == level
        for p in set(par[lo:hi].tolist()):
            kids = [int(tok[u]) for u in range(lo, hi) if par[u] == p]
            assert len(kids) == len(set(kids)), "siblings must carry distinct tokens"
    # the ancestor lists the tree implies reach the root from every slot
    assert np.array_equal(tree.depth_of(par), dep)


def test_a_cousin_visible_draft_breaks_the_pin(tiny, monkeypatch):
    """Planted mistake: the draft's visibility mask lets each node read every
    slot drafted so far (its cousins included).  The draft logits of the
    deeper levels then no longer equal the tree-verify logits."""
    glob, layers, prompt, ks, vs = tiny
    n = len(prompt)
    depth, width = 4, 3

    def everything_before(parent):
        m = len(parent)
        return np.tril(np.ones((m, m), bool))

    monkeypatch.setattr(decode, "ancestor_mask", everything_before)
    tok, par, dep, dl = decode.draft_tree(CFG, glob, layers, 5, n, ks, vs, depth, width, 0.2)
    monkeypatch.undo()
    lg, _, _ = decode.verify_tree(CFG, glob, layers, tok, par, dep, n, ks, vs)
    worst = 0.0
    for level, rows in enumerate(dl):
        for i in range(rows.shape[0]):
            worst = max(worst, float(np.max(np.abs(rows[i] - lg[_slot_of(level, i, width)]))))
    assert worst > 1e-3, "the pin does not see a draft that reads its cousins' KV"
