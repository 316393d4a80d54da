"""Pins of the oracle's decoding: the pages' central claim that SubSpec is
lossless (its stream equals plain target decoding token for token, greedy and
seeded sampling), the all-accept closed form of a self-draft chain
(tau = D + 1), verify rows equal to a causal forward of prefix || path, and the
teacher-forced stream check catching a planted wrong token."""
import numpy as np
import pytest

from oracle import decode
from oracle.model import prefill
from oracle.decode import verify_tree
import synthetic
from helpers import oracle_model, oracle_draft_layers

CFG = synthetic.CONFIGS["tiny"]


@pytest.fixture(scope="module")
def tiny():
    m = synthetic.make_model(CFG, norm_gain_std=0.1)
    glob, layers = oracle_model(m)
    draft = oracle_draft_layers(CFG, layers)
    prompt = synthetic.make_prompt(CFG).numpy()
    return glob, layers, draft, prompt


@pytest.mark.parametrize("mode,temp", [("greedy", 1.0), ("gumbel", 0.6)])
def test_plain_streams(tiny, mode, temp):
    glob, layers, draft, prompt = tiny
    ref = decode.generate_plain(CFG, glob, layers, prompt, 20, mode, temp, seed=7)
    r = decode.check_stream(CFG, glob, layers, prompt, ref, mode, temp, seed=7, gap=0.0)
    assert r["mismatch"] == [] and r["near_tie"] == []


@pytest.mark.parametrize("depth,width", [(1, 1), (2, 2), (8, 2), (3, 3), (5, 1)])
@pytest.mark.parametrize("mode,temp", [("greedy", 1.0), ("gumbel", 0.6)])
def test_subspec_is_lossless(tiny, depth, width, mode, temp):
    glob, layers, draft, prompt = tiny
    n_new = 24
    ref = decode.generate_plain(CFG, glob, layers, prompt, n_new, mode, temp, seed=7)
    got, emitted = decode.generate_subspec(CFG, glob, layers, draft, prompt, n_new, depth,
                                           width, 0.2, mode, temp, seed=7)
    assert got == ref
    assert all(1 <= e <= depth + 1 for e in emitted)
    assert 1 + sum(emitted) >= n_new


def test_self_draft_chain_accepts_everything(tiny):
    """Draft = target and k = 1: the tree is the target's own greedy chain, so
    every full cycle accepts all D drafted tokens (tau = D + 1)."""
    glob, layers, draft, prompt = tiny
    depth = 4
    got, emitted = decode.generate_subspec(CFG, glob, layers, layers, prompt, 1 + 3 * (depth + 1),
                                           depth, 1)
    assert emitted == [depth + 1] * 3
    assert got == decode.generate_plain(CFG, glob, layers, prompt, len(got))


def test_zero_substitutes_still_lossless(tiny):
    glob, layers, draft, prompt = tiny
    zero = [dict(l) for l in draft]
    for name in synthetic.LAYER_TENSORS:
        zero[1][name] = np.zeros_like(zero[1][name])
    got, emitted = decode.generate_subspec(CFG, glob, layers, zero, prompt, 12, 3, 2)
    assert got == decode.generate_plain(CFG, glob, layers, prompt, 12)
    assert all(e >= 1 for e in emitted)


def test_verify_rows_equal_causal_forward_of_each_path(tiny):
    glob, layers, draft, prompt = tiny
    n = len(prompt)
    _, ks, vs = prefill(CFG, glob, layers, prompt)
    tok, par, dep = synthetic.random_tree(3, 2, 5, CFG.vocab)
    tok, par, dep = tok.numpy(), par.numpy(), dep.numpy()
    lg, _, _ = verify_tree(CFG, glob, layers, tok, par, dep, n, ks, vs)
    for u in (0, 3, len(tok) - 1):
        path = []
        w = u
        while w >= 0:
            path.append(w)
            w = par[w]
        seq = np.concatenate([prompt, tok[path[::-1]]])
        full, _, _ = prefill(CFG, glob, layers, seq)
        assert np.allclose(lg[u], full[-1], atol=1e-5, rtol=1e-5)


def test_check_stream_catches_a_wrong_token(tiny):
    glob, layers, draft, prompt = tiny
    ref = decode.generate_plain(CFG, glob, layers, prompt, 10)
    bad = list(ref)
    bad[6] = (bad[6] + 1) % CFG.vocab
    r = decode.check_stream(CFG, glob, layers, prompt, bad, gap=1e-6)
    # the planted token is caught; later positions see a changed context
    assert r["mismatch"][:1] == [6]
    assert decode.check_stream(CFG, glob, layers, prompt, ref, gap=1e-6)["mismatch"] == []


# ---- adaptive draft depth ("Low-Bit Shadow" report 3.7, 10.1 (3)) ----
@pytest.mark.parametrize("stop", [-1.0, -4.0, -12.0])
@pytest.mark.parametrize("mode,temp", [("greedy", 1.0), ("gumbel", 0.6)])
def test_adaptive_depth_is_lossless(tiny, stop, mode, temp):
    glob, layers, draft, prompt = tiny
    ref = decode.generate_plain(CFG, glob, layers, prompt, 24, mode, temp, seed=7)
    got, emitted = decode.generate_subspec(CFG, glob, layers, draft, prompt, 24, 8, 2, 0.2, mode,
                                           temp, seed=7, stop_logp=stop)
    assert got == ref
    assert all(1 <= e <= 9 for e in emitted)


def test_adaptive_depth_limits(tiny):
    """A threshold below every score changes nothing; one above every score
    (log-probabilities are <= 0) drafts exactly one level per cycle; a higher
    threshold never drafts deeper trees."""
    glob, layers, draft, prompt = tiny
    recs = {}
    for stop in (None, -1e9, -6.0, -2.0, 1.0):
        rec = []
        out, _ = decode.generate_subspec(CFG, glob, layers, draft, prompt, 20, 6, 2,
                                         record=rec, stop_logp=stop)
        recs[stop] = (out, rec)
    base_out, base_rec = recs[None]
    out, rec = recs[-1e9]
    assert out == base_out
    assert all(np.array_equal(a["tokens"], b["tokens"]) and np.array_equal(a["parent"], b["parent"])
               for a, b in zip(rec, base_rec))
    _, rec1 = recs[1.0]
    assert all(len(r["tokens"]) == 1 + 2 and int(max(r["depth"])) == 1 for r in rec1)

    def mean_depth(rec):
        return np.mean([int(max(r["depth"])) for r in rec])
    assert mean_depth(recs[-2.0][1]) <= mean_depth(recs[-6.0][1]) <= mean_depth(base_rec)
    assert mean_depth(recs[-6.0][1]) < 6   # the threshold does stop some cycles early
