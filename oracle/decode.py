"""Plain target decoding and SubSpec draft-and-verify decoding, plus the
teacher-forced stream check (test infrastructure only).

Plain decoding ("Low-Bit Shadow" report, 2.1: the target alone, one token per
forward) is the definition the method must reproduce: SubSpec is lossless, so
its stream equals plain target decoding token for token ("Speculate Deep and
Accurate" abstract; report Critique 1 and 10.2 (4)).

One SubSpec cycle ("Low-Bit Shadow" report 2.2 Step 4, 6.3; card Approach):
  draft : D forwards of the draft (shared resident layers + substitutes) over
          the target's committed KV (KV sharing) and the draft's own KV of the
          tree nodes drafted so far; level l's nodes expand level l+1.
  verify: one target forward over all 1 + D*k nodes with the tree mask.
  accept: walk from the root, emit the accepted tokens and the bonus token,
          commit the target KV of the root and the accepted path.
Emitted tokens per cycle = accepted + 1; the first generated token comes from
the prefill.  Decoding stops once n_new tokens are emitted (the last cycle is
truncated); there is no end-of-sequence token.  tau = emitted tokens per
verify pass (1 <= tau <= D + 1).
"""
import numpy as np

from .model import forward_rows, prefill
from .tree import (expand_level, choice_scores, argmax_first, accept_walk,
                   ancestor_mask)


def _choose(logits_rows, mode, temp, seed, pos_pred):
    return argmax_first(choice_scores(logits_rows, mode, temp, seed, pos_pred))


def generate_plain(cfg, glob, layers, prompt, n_new, mode="greedy", temp=1.0, seed=0):
    """Plain target decoding; returns the n_new generated token ids."""
    prompt = np.asarray(prompt, np.int64)
    p = len(prompt)
    logits, ks, vs = prefill(cfg, glob, layers, prompt)
    out = [int(_choose(logits[-1:], mode, temp, seed, [p])[0])]
    while len(out) < n_new:
        pos = p + len(out) - 1
        lg, nk, nv = forward_rows(cfg, glob, layers, [out[-1]], [pos], ks, vs,
                                  np.ones((1, pos), bool), np.ones((1, 1), bool))
        ks = [np.concatenate([a, b]) for a, b in zip(ks, nk)]
        vs = [np.concatenate([a, b]) for a, b in zip(vs, nv)]
        out.append(int(_choose(lg, mode, temp, seed, [pos + 1])[0]))
    return out


def draft_tree(cfg, glob, draft_layers, root_token, n, ks, vs, depth, width, draft_temp,
               stop_logp=None):
    """Build the static tree for one cycle.  Returns (tokens, parent, depth,
    draft logits per level).  ks/vs: the target's committed KV, length n.

    Adaptive depth (stop_logp not None): after a level is added, drafting stops
    when the best cumulative sharpened log-probability among its nodes is below
    stop_logp -- deeper nodes would hang below a path the draft itself finds
    unlikely ("Low-Bit Shadow" report 3.7 and 10.1 (3): the back half of the
    48-level tree rarely pays off).  The tree then has fewer than `depth`
    levels; everything downstream (verify, accept) takes it as it is."""
    tokens = [int(root_token)]
    parent = [-1]
    dep = [0]
    score = [0.0]
    # draft KV of the tree slots drafted so far, per layer
    dk = [np.zeros((0, cfg.n_heads_kv, cfg.head_dim), np.float32) for _ in range(cfg.n_layers)]
    dv = [np.zeros((0, cfg.n_heads_kv, cfg.head_dim), np.float32) for _ in range(cfg.n_layers)]
    frontier = [0]
    level_logits = []
    for lvl in range(depth):
        n_done = len(dk[0])                       # slots with draft KV so far
        anc = ancestor_mask(np.array(parent))
        rows = frontier
        m = len(rows)
        past_vis = np.zeros((m, n + n_done), bool)
        past_vis[:, :n] = True
        for i, u in enumerate(rows):
            past_vis[i, n:n + n_done] = anc[u, :n_done]
        pk = [np.concatenate([a, b]) for a, b in zip(ks, dk)]
        pv = [np.concatenate([a, b]) for a, b in zip(vs, dv)]
        lg, nk, nv = forward_rows(cfg, glob, draft_layers, [tokens[u] for u in rows],
                                  [n + dep[u] for u in rows], pk, pv, past_vis,
                                  np.eye(m, dtype=bool))
        # frontier slots are exactly the next slots in order: append their KV
        dk = [np.concatenate([a, b]) for a, b in zip(dk, nk)]
        dv = [np.concatenate([a, b]) for a, b in zip(dv, nv)]
        level_logits.append(lg)
        tok, par, sc = expand_level(lg, [score[u] for u in rows], rows, width, draft_temp)
        frontier = []
        for t, pa, s in zip(tok, par, sc):
            frontier.append(len(tokens))
            tokens.append(int(t))
            parent.append(int(pa))
            dep.append(dep[pa] + 1)
            score.append(float(s))
        if stop_logp is not None and max(sc) < stop_logp:
            break
    return (np.array(tokens, np.int64), np.array(parent, np.int64),
            np.array(dep, np.int64), level_logits)


def verify_tree(cfg, glob, layers, tokens, parent, dep, n, ks, vs):
    """One target forward over all tree nodes with the ancestor mask."""
    m = len(tokens)
    return forward_rows(cfg, glob, layers, tokens, n + np.asarray(dep), ks, vs,
                        np.ones((m, n), bool), ancestor_mask(parent))


def generate_subspec(cfg, glob, target_layers, draft_layers, prompt, n_new, depth, width,
                     draft_temp=0.2, mode="greedy", temp=1.0, seed=0, record=None,
                     stop_logp=None):
    """SubSpec decoding; returns (tokens, per-cycle emitted counts).  With
    stop_logp the tree depth adapts per cycle (see draft_tree)."""
    prompt = np.asarray(prompt, np.int64)
    n = len(prompt)
    logits, ks, vs = prefill(cfg, glob, target_layers, prompt)
    root = int(_choose(logits[-1:], mode, temp, seed, [n])[0])
    out = [root]
    emitted = []
    while len(out) < n_new:
        tokens, parent, dep, dl = draft_tree(cfg, glob, draft_layers, root, n, ks, vs,
                                             depth, width, draft_temp, stop_logp)
        lg, nk, nv = verify_tree(cfg, glob, target_layers, tokens, parent, dep, n, ks, vs)
        choice = _choose(lg, mode, temp, seed, n + dep + 1)
        acc, bonus = accept_walk(tokens, parent, choice)
        path = [0] + acc
        ks = [np.concatenate([a, b[path]]) for a, b in zip(ks, nk)]
        vs = [np.concatenate([a, b[path]]) for a, b in zip(vs, nv)]
        new = [int(tokens[s]) for s in acc] + [bonus]
        if record is not None:
            record.append(dict(tokens=tokens, parent=parent, depth=dep, draft_logits=dl,
                               target_logits=lg, accepted=acc, bonus=bonus, n=n))
        emitted.append(len(new))
        out.extend(new)
        n += len(path)
        root = bonus
    return out[:n_new], emitted


def check_stream(cfg, glob, layers, prompt, stream, mode="greedy", temp=1.0, seed=0,
                 gap=1e-2):
    """Teacher-forced losslessness check: one causal target forward over
    prompt + stream[:-1]; at every generated position the emitted token must be
    the target's choice, or lie within `gap` (in choice-score units) of it.
    Returns dict(mismatch=[positions outside the gap], near_tie=[positions where
    a different token won inside the gap], min_gap)."""
    prompt = np.asarray(prompt, np.int64)
    stream = np.asarray(stream, np.int64)
    p = len(prompt)
    seq = np.concatenate([prompt, stream[:-1]])
    logits, _, _ = prefill(cfg, glob, layers, seq)
    rows = logits[p - 1:]
    pos_pred = np.arange(p, p + len(stream))
    sc = choice_scores(rows, mode, temp, seed, pos_pred)
    best = argmax_first(sc)
    bad, near = [], []
    for i, t in enumerate(stream):
        if t != best[i]:
            d = sc[i, best[i]] - sc[i, t]
            (near if d < gap else bad).append(i)
    return dict(mismatch=bad, near_tie=near, n=len(stream))
