"""Full-size parity harness (shared by the full-size GPU tests).

Drives whole SubSpec decode cycles through the library's public entry points
(target prefill, D draft forwards each followed by an expansion, one verify
pass over the tree, the accept walk, KV compaction) on a full-size decoder,
and checks them against the oracle on the same seeded inputs:

* the emitted stream, by teacher forcing: one causal oracle forward over
  prompt + stream; every emitted token must be the oracle target's choice
  unless the oracle's top-2 gap there is below 1e-2 (counted as near-ties);
* for the checked cycles (the first two and every 16th), the tree level by
  level: the oracle's expansion run on the GPU's own draft logits must pick
  the same slots, tokens and parents, except where its k-th and (k+1)-th
  candidate scores lie within 1e-4 (fp32 against float64 logsumexp);
* the GPU's draft logits of the first levels against the oracle's draft
  forward over the same tree, and a sample of verify rows against the
  oracle's tree-masked target forward (|gpu - oracle| <= 2e-2 + 1e-2 |oracle|);
* the accept walk: the GPU's path and bonus equal the walk of its own choices,
  and its choices equal the oracle's away from near-ties.

Sources: the losslessness claim ("Speculate Deep and Accurate" abstract;
"Low-Bit Shadow" report Critique 1 and 10.2 (4)), tree verification as
per-path causal attention (report 6.3), the expansion reading of the draft
tree (report 6.3/6.4; card, Approach).
"""
from __future__ import annotations

import gc
import time

import numpy as np
import torch

import synthetic
from oracle import quant
from oracle.model import forward_rows, prefill
from oracle.tree import expand_level, choice_scores, argmax_first, accept_walk, ancestor_mask

ATOL, RTOL = 2e-2, 1e-2
DEV = "cuda"
# Full-depth tolerance, calibrated (see tolerance()): the GPU may depart from
# the float64 oracle by at most KAPPA times as much as the oracle itself does
# with float32 GEMM accumulation; the draft path, which folds the RMSNorm row
# scale and the int4 zero/scale into fp32 sums (two more rounding-point
# readings), by at most KAPPA_DRAFT times; token choices may differ where the
# oracle's top-2 gap is below GAP_SIGMAS standard deviations of the calibrated
# difference of two logits' errors (and never below 1e-2).
KAPPA, KAPPA_DRAFT, GAP_SIGMAS = 2.0, 4.0, 6.0


class Float32Gemms:
    """The oracle with its matrix products accumulated in float32 instead of
    float64: a second correct bf16 implementation, used to calibrate how far
    two such implementations drift apart through a deep decoder."""

    def __enter__(self):
        import oracle.model as om
        self.om, self.orig = om, om.mm
        om.mm = lambda a, w: np.asarray(a, np.float32) @ np.asarray(w, np.float32).T
        return self

    def __exit__(self, *exc):
        self.om.mm = self.orig


def tolerance(e_gpu, e_cal, refs, n_elem, viol):
    """Error statistics of the GPU and of the calibration against the oracle
    on the same logits.  Every bf16 rounding stage turns a pre-rounding
    difference d between two implementations into roughly sqrt(d * ulp) of
    flip noise, so after a few stages any two correct bf16 implementations
    differ by about one bf16 ulp per layer, growing like the square root of
    the depth; the calibration measures that floor on the same inputs."""
    e_gpu = np.asarray(e_gpu, np.float64).ravel()
    e_cal = np.asarray(e_cal, np.float64).ravel()
    nref = float(np.linalg.norm(np.asarray(refs, np.float64).ravel()))
    return dict(rms_gpu=float(np.sqrt(np.mean(e_gpu ** 2))),
                rms_cal=float(np.sqrt(np.mean(e_cal ** 2))),
                rel_l2_gpu=float(np.linalg.norm(e_gpu)) / nref,
                rel_l2_cal=float(np.linalg.norm(e_cal)) / nref,
                p999_gpu=float(np.quantile(np.abs(e_gpu), 0.999)),
                p999_cal=float(np.quantile(np.abs(e_cal), 0.999)),
                max_gpu=float(np.abs(e_gpu).max()), max_cal=float(np.abs(e_cal).max()),
                elementwise_violations=f"{viol}/{n_elem}")


def _np(t):
    return t.detach().float().cpu().numpy()


def _substitute(w):
    """The oracle's pack + dequant of one row block (rows quantise
    independently: groups run along K within a row)."""
    q, s, z = quant.w4_pack(w)
    return quant.w4_dequant(q, s, z, w.shape[1])


def oracle_layers(weights, cfg, threads=16, rows_per_task=2048):
    """Target layers (float32 arrays of the bf16 values) and the draft's:
    shared resident layers + oracle-dequantised int4 substitutes (row blocks
    quantised on a thread pool; NumPy releases the GIL in the array work)."""
    from concurrent.futures import ThreadPoolExecutor
    glob = {k: _np(weights[k]) for k in ("embed", "lm_head", "final_norm")}
    target, draft = [], []
    jobs = []
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for i, lw in enumerate(weights["layers"]):
            t = {k: _np(v) for k, v in lw.items()}
            target.append(t)
            if i < cfg.n_resident:
                draft.append(t)
                continue
            d = dict(t)
            for name in synthetic.LAYER_TENSORS:
                w = t[name]
                parts = [ex.submit(_substitute, w[r:r + rows_per_task])
                         for r in range(0, w.shape[0], rows_per_task)]
                jobs.append((d, name, parts))
            draft.append(d)
        for d, name, parts in jobs:
            d[name] = np.concatenate([p.result() for p in parts], axis=0)
    return glob, target, draft


class LazyLayers:
    """Oracle-format layers converted from bf16 host tensors when iterated,
    one at a time (for decoders whose float32 weights do not fit in host
    memory at once)."""

    def __init__(self, layers, draft_from=None):
        self.layers = layers
        self.draft_from = draft_from   # layers >= this index become substitutes

    def __len__(self):
        return len(self.layers)

    def __iter__(self):
        from concurrent.futures import ThreadPoolExecutor
        for i, lw in enumerate(self.layers):
            t = {k: _np(v) for k, v in lw.items()}
            if self.draft_from is not None and i >= self.draft_from:
                with ThreadPoolExecutor(max_workers=16) as ex:
                    for name in synthetic.LAYER_TENSORS:
                        w = t[name]
                        parts = [ex.submit(_substitute, w[r:r + 2048])
                                 for r in range(0, w.shape[0], 2048)]
                        t[name] = np.concatenate([p.result() for p in parts], axis=0)
            yield t


class Cycle:
    """What one GPU decode cycle produced (host copies)."""

    def __init__(self, n, root):
        self.n = n              # committed length; the root sits at position n
        self.root = root
        self.draft_logits = []  # per level: [rows, V] float32
        self.tokens = self.parent = self.depth = None
        self.verify_logits = None
        self.choice = None
        self.accepted = None
        self.bonus = None


def gpu_cycles(sub, model, cfg, prompt, n_new, depth, width, mode, temp, seed, keep_cycles):
    """Decode n_new tokens with cycles driven through the public entry points.
    Returns (stream, [Cycle] with draft/verify logits for the cycles in
    keep_cycles (0-based), cycle count)."""
    V = cfg.vocab
    p = prompt.to(DEV)
    lg = torch.empty((len(p), V), dtype=torch.float32, device=DEV)
    model.forward(0, p, 0, 0, logits=lg)
    acc0 = torch.zeros(max(depth, 1), dtype=torch.int32, device=DEV)
    tr = sub.DeviceTree(depth, width, DEV)
    n = len(p)
    first = sub.verify_accept(lg[-1:].contiguous(), tr, 1, mode=mode, temperature=temp, seed=seed,
                              root_pos=n - 1)
    root = int(first[2].item())
    stream = [root]
    kv = model.kv()
    n_tree = 1 + depth * width
    dl = torch.empty((width, V), dtype=torch.float32, device=DEV)
    vl = torch.empty((n_tree, V), dtype=torch.float32, device=DEV)
    kept, c = [], 0
    while len(stream) < n_new:
        cyc = Cycle(n, root)
        keep = c in keep_cycles
        tr.token[0] = root
        for lvl in range(depth):
            s0 = 0 if lvl == 0 else 1 + (lvl - 1) * width
            m = 1 if lvl == 0 else width
            model.forward(1, tr.token[s0:s0 + m], s0, n, depth=tr.depth[s0:s0 + m],
                          anc=tr.anc[s0:s0 + m], logits=dl[:m])
            if keep:
                cyc.draft_logits.append(_np(dl[:m]))
            sub.draft_expand(dl[:m], 0.2, tr, lvl)
        model.forward(0, tr.token, 0, n, depth=tr.depth, anc=tr.anc, logits=vl)
        acc, na, bonus, choice = sub.verify_accept(vl, tr, n_tree, mode=mode, temperature=temp,
                                                   seed=seed, root_pos=n)
        sub.kv_compact(kv, n, acc, na, depth)
        a = int(na.item())
        toks = tr.token.cpu().numpy()
        new = [int(toks[s]) for s in acc[:a].cpu().tolist()] + [int(bonus.item())]
        if keep:
            cyc.tokens, cyc.parent, cyc.depth = toks, tr.parent.cpu().numpy(), tr.depth.cpu().numpy()
            cyc.verify_logits = _np(vl)
            cyc.choice = choice.cpu().numpy()
            cyc.accepted = acc[:a].cpu().tolist()
            cyc.bonus = int(bonus.item())
            kept.append((c, cyc))
        stream.extend(new)
        n += a + 1
        root = new[-1]
        c += 1
    del acc0
    torch.cuda.synchronize()
    return stream[:n_new], kept, c


def _close(got, ref, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond tolerance, max excess "
                           f"{np.max(err - bound):.3e}, max err {err.max():.3e}")
    return float(err.max())


def check_tree_teacher_forced(cyc, width, temp=0.2):
    """Level by level, the oracle's expansion of the GPU's draft logits picks
    the GPU's slots.  Returns the number of near-tie levels (a k-th/(k+1)-th
    gap < 1e-4 where the two sides may differ; the GPU's tree is kept)."""
    depth_max = len(cyc.draft_logits)
    score = {0: 0.0}
    near = 0
    for lvl in range(depth_max):
        s0 = 0 if lvl == 0 else 1 + (lvl - 1) * width
        rows = list(range(s0, s0 + cyc.draft_logits[lvl].shape[0]))
        tok, par, sc = expand_level(cyc.draft_logits[lvl], [score[u] for u in rows], rows,
                                    width + 1, temp)
        out0 = 1 + lvl * width
        g_tok = cyc.tokens[out0:out0 + width]
        g_par = cyc.parent[out0:out0 + width]
        same = np.array_equal(tok[:width], g_tok) and np.array_equal(par[:width], g_par)
        if not same:
            margin = sc[width - 1] - sc[width] if len(sc) > width else np.inf
            # where the lists first differ, the oracle's own ranking must be a near-tie there
            first = int(np.nonzero((tok[:width] != g_tok) | (par[:width] != g_par))[0][0])
            local = sc[first] - sc[first + 1] if first + 1 < len(sc) else np.inf
            assert min(margin, local) < 1e-4, (f"level {lvl}: GPU tree differs from the oracle's "
                                               f"selection away from a near-tie "
                                               f"(margin {margin:.3e}, local {local:.3e})")
            near += 1
        # carry on along the GPU's tree with float64 scores
        lp = {}
        for t, pa, s in zip(tok, par, sc):
            lp[(int(pa), int(t))] = s
        for j in range(width):
            u = out0 + j
            key = (int(g_par[j]), int(g_tok[j]))
            if key in lp:
                score[u] = lp[key]
            else:   # a near-tie candidate outside the oracle's top k + 1: recompute
                from oracle.tree import log_softmax_t
                r = rows.index(int(g_par[j]))
                score[u] = score[int(g_par[j])] + float(
                    log_softmax_t(cyc.draft_logits[lvl][r:r + 1], temp)[0, int(g_tok[j])])
    return near


def oracle_verify_rows(cfg, glob, target, cyc, ks, vs, sample):
    """The oracle's tree-masked target forward over the ancestor closure of
    the sampled nodes; returns {slot: logits row}."""
    par = cyc.parent
    anc = ancestor_mask(par)
    rows = sorted(set(int(w) for u in sample for w in np.nonzero(anc[u])[0]))
    sub_anc = anc[np.ix_(rows, rows)]
    n = cyc.n
    lg, _, _ = forward_rows(cfg, glob, target, cyc.tokens[rows], n + cyc.depth[rows],
                            [k[:n] for k in ks], [v[:n] for v in vs], np.ones((len(rows), n), bool),
                            sub_anc)
    return {u: lg[rows.index(u)] for u in sample}


def oracle_draft_levels(cfg, glob, draft, cyc, ks, vs, width, levels):
    """The oracle's draft forward over the GPU's tree for the first `levels`
    levels (draft KV of the drafted slots kept, KV sharing with the committed
    prefix); returns the per-level logits."""
    n = cyc.n
    pk = [k[:n] for k in ks]
    pv = [v[:n] for v in vs]
    dk = [np.zeros((0, cfg.n_heads_kv, cfg.head_dim), np.float32) for _ in range(cfg.n_layers)]
    dv = [np.zeros((0, cfg.n_heads_kv, cfg.head_dim), np.float32) for _ in range(cfg.n_layers)]
    anc = ancestor_mask(cyc.parent)
    out = []
    for lvl in range(levels):
        s0 = 0 if lvl == 0 else 1 + (lvl - 1) * width
        rows = list(range(s0, s0 + (1 if lvl == 0 else width)))
        n_done = len(dk[0])
        vis = np.zeros((len(rows), n + n_done), bool)
        vis[:, :n] = True
        for i, u in enumerate(rows):
            vis[i, n:] = anc[u, :n_done]
        lg, nk, nv = forward_rows(cfg, glob, draft, cyc.tokens[rows], n + cyc.depth[rows],
                                  [np.concatenate([a, b]) for a, b in zip(pk, dk)],
                                  [np.concatenate([a, b]) for a, b in zip(pv, dv)], vis,
                                  np.eye(len(rows), dtype=bool))
        dk = [np.concatenate([a, b]) for a, b in zip(dk, nk)]
        dv = [np.concatenate([a, b]) for a, b in zip(dv, nv)]
        out.append(lg)
    return out


def run(sub, cfg, n_new, mode="greedy", temp=1.0, seed=7, depth=48, width=8, staging=0,
        embed_on_host=False, draft_levels=3, verify_sample=40, lazy=False, every=16, log=print):
    """The whole check; returns a dict of counts for the test to report."""
    t0 = time.time()
    mcode = 0 if mode == "greedy" else 1
    weights = synthetic.make_model(cfg, device=DEV)
    prompt = synthetic.make_prompt(cfg)
    model = sub.Model(cfg, weights, max_seq=cfg.prompt_len + n_new + 2 * (depth + 1) + 64,
                      max_depth=depth, max_width=width, max_prompt=cfg.prompt_len,
                      staging_layers=staging, embed_on_host=embed_on_host)
    for i in range(cfg.n_resident, cfg.n_layers):
        for name in synthetic.LAYER_TENSORS:
            weights["layers"][i][name] = weights["layers"][i][name].to("cpu")
    for k in ("embed", "lm_head", "final_norm"):
        weights[k] = weights[k].to("cpu")
    for i in range(cfg.n_resident):
        weights["layers"][i] = {k: v.to("cpu") for k, v in weights["layers"][i].items()}
    torch.cuda.empty_cache()
    # the graph-captured decode loop, then the same decode through the public steps
    gen, st = model.generate(prompt, n_new, depth, width, 0.2, mode=mcode, target_temp=temp,
                             seed=seed)
    gen = gen.tolist()
    n_cyc_est = max(3, int(n_new / max(st.tau, 1.0)) + 2)
    keep = {0, 1} | set(range(every, n_cyc_est + every, every))
    stream, kept, n_cycles = gpu_cycles(sub, model, cfg, prompt, n_new, depth, width, mcode, temp,
                                        seed, keep)
    model.close()
    del model
    torch.cuda.empty_cache()
    t_gpu = time.time() - t0
    log(f"{cfg.name}: GPU done in {t_gpu:.0f}s, {n_cycles} cycles, tau {st.tau:.2f}")

    if lazy:
        glob = {k: _np(weights[k]) for k in ("embed", "lm_head", "final_norm")}
        target = LazyLayers(weights["layers"])
        draft = LazyLayers(weights["layers"], draft_from=cfg.n_resident)
    else:
        glob, target, draft = oracle_layers(weights, cfg)
        del weights
    gc.collect()
    t_or = time.time()
    # one causal oracle forward over prompt + stream gives the stream check and
    # the committed K/V at every cycle's start; the same with float32 GEMMs is
    # the calibration (see tolerance())
    p = prompt.numpy().astype(np.int64)
    seq = np.concatenate([p, np.asarray(stream[:-1], np.int64)])
    logits, ks, vs = prefill(cfg, glob, target, seq)
    with Float32Gemms():
        cal_logits, cks, cvs = prefill(cfg, glob, target, seq)
    rows = logits[len(p) - 1:]
    pos_pred = np.arange(len(p), len(p) + len(stream))
    sc = choice_scores(rows, mode, temp, seed, pos_pred)
    best = argmax_first(sc)
    res = dict(cycles=n_cycles, tau=st.tau, near_tie_stream=0, near_tie_tree=0,
               near_tie_choice=0, checked_cycles=[c for c, _ in kept], gen_vs_steps_first_diff=None)

    # ---- verify rows of the checked cycles: GPU and calibration against the oracle
    e_gpu, e_cal, refs, n_elem, viol = [], [], [], 0, 0
    per_cycle = []
    for c, cyc in kept:
        n_tree = len(cyc.tokens)
        rng = np.random.default_rng(c)
        sample = sorted(set([0] + cyc.accepted +
                            rng.choice(n_tree, size=min(verify_sample, n_tree), replace=False)
                            .tolist()))
        ref = oracle_verify_rows(cfg, glob, target, cyc, ks, vs, sample)
        with Float32Gemms():
            cal = oracle_verify_rows(cfg, glob, target, cyc, cks, cvs, sample)
        for u in sample:
            e_gpu.append(cyc.verify_logits[u] - ref[u])
            e_cal.append(cal[u] - ref[u])
            refs.append(ref[u])
            viol += int((np.abs(e_gpu[-1]) > ATOL + RTOL * np.abs(ref[u])).sum())
            n_elem += ref[u].size
        per_cycle.append((c, cyc, sample, ref))
    tol = tolerance(np.concatenate(e_gpu), np.concatenate(e_cal), np.concatenate(refs), n_elem,
                    viol)
    res["verify"] = tol
    assert tol["rel_l2_gpu"] <= KAPPA * tol["rel_l2_cal"] + 1e-4, f"verify logits: {tol}"
    assert tol["p999_gpu"] <= KAPPA * tol["p999_cal"] + 1e-3, f"verify logits: {tol}"
    gap_tol = max(1e-2, GAP_SIGMAS * np.sqrt(2.0) * tol["rms_cal"] / (temp if mode != "greedy"
                                                                       else 1.0))
    res["gap_tol"] = round(float(gap_tol), 4)

    def stream_check(tokens, label):
        bad, near, worst = [], 0, 0.0
        for i, t in enumerate(tokens):
            if t != best[i]:
                gap = sc[i, best[i]] - sc[i, t]
                if gap < gap_tol:
                    near += 1
                    worst = max(worst, float(gap))
                else:
                    bad.append((i, int(t), int(best[i]), float(gap)))
        assert bad == [], f"{label}: tokens that are not the target's choice: {bad[:5]}"
        res.setdefault("max_near_tie_gap", 0.0)
        res["max_near_tie_gap"] = round(max(res["max_near_tie_gap"], worst), 4)
        return near

    # the calibration's own choices along the stream: how often and by how much
    # a second correct bf16 implementation departs from the oracle's argmax
    csc = choice_scores(cal_logits[len(p) - 1:], mode, temp, seed, pos_pred)
    cbest = argmax_first(csc)
    cflip = np.nonzero(cbest != best)[0]
    res["calibration_flips"] = int(len(cflip))
    res["calibration_max_flip_gap"] = round(float(max((sc[i, best[i]] - sc[i, cbest[i]]
                                                       for i in cflip), default=0.0)), 4)
    res["near_tie_stream"] = stream_check(stream, "step-wise stream")
    # the captured decode loop agrees with the step-wise one up to its first near-tie
    # (past a near-tie the contexts differ); it is checked against the oracle up to there
    diff = next((i for i, (a, b) in enumerate(zip(gen, stream)) if a != b), None)
    res["gen_vs_steps_first_diff"] = diff
    if diff is not None:
        assert sc[diff, best[diff]] - min(sc[diff, gen[diff]], sc[diff, stream[diff]]) < gap_tol, \
            f"captured and step-wise decoding differ at {diff} away from a near-tie"
    stream_check(gen[:diff] if diff is not None else gen, "captured stream")

    for c, cyc, sample, ref in per_cycle:
        res["near_tie_tree"] += check_tree_teacher_forced(cyc, width)
        # accept walk of the GPU's own choices
        acc, bonus = accept_walk(cyc.tokens, cyc.parent, cyc.choice)
        assert acc == cyc.accepted and bonus == cyc.bonus, f"cycle {c}: accept walk differs"
        for u in sample:
            ou = choice_scores(ref[u][None], mode, temp, seed, [cyc.n + cyc.depth[u] + 1])[0]
            o_best = int(np.argmax(ou))
            if o_best != int(cyc.choice[u]):
                gap = ou[o_best] - ou[int(cyc.choice[u])]
                assert gap < gap_tol, f"cycle {c} node {u}: choice differs, oracle gap {gap:.3e}"
                res["near_tie_choice"] += 1
        if c == 0 and draft_levels:
            dref = oracle_draft_levels(cfg, glob, draft, cyc, ks, vs, width, draft_levels)
            eg = np.concatenate([cyc.draft_logits[l] - r for l, r in enumerate(dref)]).ravel()
            refs = np.concatenate(dref).ravel()
            rel = float(np.linalg.norm(eg) / np.linalg.norm(refs))
            res["draft_rel_l2"] = round(rel, 5)
            assert rel <= KAPPA_DRAFT * tol["rel_l2_cal"] + 1e-4, \
                f"draft logits: rel_l2 {rel:.4e} against calibration {tol['rel_l2_cal']:.4e}"
    res["oracle_s"] = round(time.time() - t_or, 1)
    res["gpu_s"] = round(t_gpu, 1)
    log(f"{cfg.name}: {res}")
    return res
