"""Static draft tree: expansion from sharpened draft probabilities, the target's
choice per node and the accept walk (test infrastructure only).

Tree shape: deep, narrow and static -- a fixed number k of nodes kept on each
of D levels ("Low-Bit Shadow" report, 6.3 SpecInfer and 6.4 EAGLE-2: k = 6,
D = 48; 3.7: D = 48), verified in one target pass with tree attention
(report, 6.3).  Draft probabilities are sharpened with temperature 0.2
("Speculate Deep and Accurate" card, Approach; report 3.4).

Slot layout: slot 0 is the root (the last committed token, depth 0); level l
(1..D) holds slots 1+(l-1)k .. lk in descending cumulative score.

Reading of the expansion (the pages give only "deep, narrow, static" and
"sharpened probabilities"): for every level-l node j with draft logits z_j,
  lp_j(v) = z_j(v)/T - logsumexp_v(z_j/T)           (float64)
candidates are each node's own top-k tokens (ties -> smaller token id), a
candidate's score is S_j + lp_j(v) with S_j the node's cumulative score, and
level l+1 keeps the global top-k candidates (ties -> smaller parent slot, then
smaller token id).  Siblings therefore carry distinct tokens.

Accept (Leviathan-style verification with a tree, report 6.2 and 6.3): starting
at the root, move to the child whose token equals the target's choice at the
current node while one exists; the visited children are accepted and the
target's choice at the last node is the bonus token.
"""
import numpy as np

from .philox import gumbel


def log_softmax_t(logits, temp: float) -> np.ndarray:
    z = np.asarray(logits, np.float64) / temp
    mx = z.max(axis=-1, keepdims=True)
    lse = mx + np.log(np.exp(z - mx).sum(axis=-1, keepdims=True))
    return z - lse


def expand_level(logits, parent_score, parent_slot, k: int, temp: float):
    """logits [k_prev, V] of the frontier nodes -> (token, parent slot, score)
    arrays of the k children kept, in slot order."""
    lp = log_softmax_t(logits, temp)                      # [k_prev, V]
    cands = []
    for j in range(lp.shape[0]):
        # own top-k, ties to the smaller token id: stable sort on -lp
        order = np.argsort(-lp[j], kind="stable")[:k]
        for v in order:
            cands.append((float(parent_score[j]) + float(lp[j, v]), int(parent_slot[j]), int(v)))
    cands.sort(key=lambda c: (-c[0], c[1], c[2]))
    keep = cands[:k]
    return (np.array([c[2] for c in keep], np.int64),
            np.array([c[1] for c in keep], np.int64),
            np.array([c[0] for c in keep], np.float64))


def choice_scores(logits, mode: str, temp: float, seed: int, pos_pred) -> np.ndarray:
    """Per-row scores whose argmax is the target's token: the logits (greedy)
    or logits/T + Gumbel(seed, predicted position, v) (sampled)."""
    z = np.asarray(logits, np.float64)
    if mode == "greedy":
        return z
    out = np.empty_like(z)
    for i, p in enumerate(np.atleast_1d(pos_pred)):
        out[i] = z[i] / temp + gumbel(seed, int(p), z.shape[1])
    return out


def argmax_first(scores) -> np.ndarray:
    """argmax per row, ties to the smaller index."""
    return np.argmax(np.asarray(scores), axis=-1)


def accept_walk(tokens, parent, choice):
    """tokens, parent: [n] tree arrays; choice: [n] target token per node.
    Returns (accepted slots list, bonus token)."""
    tokens = np.asarray(tokens)
    parent = np.asarray(parent)
    u = 0
    acc = []
    while True:
        kids = np.nonzero(parent == u)[0]
        match = [c for c in kids if tokens[c] == choice[u]]
        if not match:
            break
        u = int(match[0])
        acc.append(u)
    return acc, int(choice[u])


def ancestor_mask(parent) -> np.ndarray:
    """[n, n] bool: entry (u, w) is True when w is u or an ancestor of u."""
    parent = np.asarray(parent)
    n = parent.shape[0]
    m = np.zeros((n, n), bool)
    for u in range(n):
        w = u
        while w >= 0:
            m[u, w] = True
            w = int(parent[w])
    return m


def depth_of(parent) -> np.ndarray:
    parent = np.asarray(parent)
    d = np.zeros(parent.shape[0], np.int64)
    for u in range(parent.shape[0]):
        w = int(parent[u])
        while w >= 0:
            d[u] += 1
            w = int(parent[w])
    return d


def tree_attention(q, k_prefix, v_prefix, k_tree, v_tree, parent, n_heads_kv: int):
    """Tree attention by its definition: node u reads the prefix keys plus the
    keys of its root path (root .. u).  q: [n, Hq, d]; k/v_prefix [P, Hkv, d];
    k/v_tree [n, Hkv, d].  Computed node by node in float64."""
    from .model import attention
    mask = ancestor_mask(parent)
    n = q.shape[0]
    out = np.zeros(q.shape, np.float32)
    for u in range(n):
        path = np.nonzero(mask[u])[0]
        kk = np.concatenate([k_prefix, k_tree[path]], axis=0)
        vv = np.concatenate([v_prefix, v_tree[path]], axis=0)
        vis = np.ones((1, kk.shape[0]), bool)
        out[u] = attention(q[u:u + 1], kk, vv, vis, n_heads_kv)[0]
    return out
