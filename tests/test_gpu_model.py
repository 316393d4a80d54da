"""Model-level parity on the tiny decoder: target prefill logits, tree-verify
logits and draft logits against the oracle (allclose with atol 2e-2, rtol
1e-2), and whole SubSpec decoding checked token by token against the
oracle's target with teacher forcing (an emitted token must be the target's
choice unless the oracle's top-2 gap is below 1e-2)."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import decode
from oracle.model import prefill, forward_rows
from oracle.decode import verify_tree
from helpers import oracle_model, oracle_draft_layers

pytestmark = pytest.mark.gpu
DEV = "cuda"
CFG = synthetic.CONFIGS["tiny"]
ATOL, RTOL = 2e-2, 1e-2


@pytest.fixture(scope="module")
def sub():
    import substitute_speculative_decoding_gb300 as s
    return s


@pytest.fixture(scope="module")
def tiny(sub):
    w = synthetic.make_model(CFG, norm_gain_std=0.1)
    glob, layers = oracle_model(w)
    draft = oracle_draft_layers(CFG, layers)
    prompt = synthetic.make_prompt(CFG)
    model = sub.Model(CFG, w, max_seq=256, max_depth=8, max_width=3, max_prompt=64)
    yield dict(w=w, glob=glob, layers=layers, draft=draft, prompt=prompt, model=model)
    model.close()


def close(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    assert np.all(err <= bound), f"max excess {np.max(err - bound):.3e}, max err {err.max():.3e}"


def _prefill_gpu(t):
    m = t["model"]
    p = t["prompt"].to(DEV)
    logits = torch.empty((len(p), CFG.vocab), dtype=torch.float32, device=DEV)
    m.forward(0, p, 0, 0, logits=logits)
    torch.cuda.synchronize()
    return logits.cpu().numpy()


def test_prefill_logits(tiny):
    got = _prefill_gpu(tiny)
    ref, _, _ = prefill(CFG, tiny["glob"], tiny["layers"], tiny["prompt"].numpy())
    close(got, ref)


def test_verify_logits_on_a_tree(tiny):
    _prefill_gpu(tiny)
    n = len(tiny["prompt"])
    _, ks, vs = prefill(CFG, tiny["glob"], tiny["layers"], tiny["prompt"].numpy())
    tok, par, dep = synthetic.random_tree(4, 3, 9, CFG.vocab)
    anc = synthetic.ancestors(par, dep, 8)
    logits = torch.empty((len(tok), CFG.vocab), dtype=torch.float32, device=DEV)
    tiny["model"].forward(0, tok.to(DEV), 0, n, depth=dep.to(DEV), anc=anc.to(DEV), logits=logits)
    torch.cuda.synchronize()
    ref, _, _ = verify_tree(CFG, tiny["glob"], tiny["layers"], tok.numpy(), par.numpy(),
                            dep.numpy(), n, ks, vs)
    close(logits.cpu().numpy(), ref)


def test_draft_logits_two_levels(tiny):
    """Draft rows read the target's committed KV (shared cache) plus the draft
    KV of their tree ancestors."""
    _prefill_gpu(tiny)
    n = len(tiny["prompt"])
    _, ks, vs = prefill(CFG, tiny["glob"], tiny["layers"], tiny["prompt"].numpy())
    tok, par, dep = synthetic.random_tree(2, 3, 10, CFG.vocab)
    anc = synthetic.ancestors(par, dep, 8)
    m = tiny["model"]
    lg0 = torch.empty((1, CFG.vocab), dtype=torch.float32, device=DEV)
    m.forward(1, tok[:1].to(DEV), 0, n, depth=dep[:1].to(DEV), anc=anc[:1].to(DEV), logits=lg0)
    lg1 = torch.empty((3, CFG.vocab), dtype=torch.float32, device=DEV)
    m.forward(1, tok[1:4].contiguous().to(DEV), 1, n, depth=dep[1:4].contiguous().to(DEV),
              anc=anc[1:4].contiguous().to(DEV), logits=lg1)
    torch.cuda.synchronize()
    draft = tiny["draft"]
    r0, dk, dv = forward_rows(CFG, tiny["glob"], draft, tok[:1].numpy(), [n], ks, vs,
                              np.ones((1, n), bool), np.ones((1, 1), bool))
    close(lg0.cpu().numpy(), r0)
    pk = [np.concatenate([a, b]) for a, b in zip(ks, dk)]
    pv = [np.concatenate([a, b]) for a, b in zip(vs, dv)]
    vis = np.ones((3, n + 1), bool)
    r1, _, _ = forward_rows(CFG, tiny["glob"], draft, tok[1:4].numpy(), n + dep[1:4].numpy(),
                            pk, pv, vis, np.eye(3, dtype=bool))
    close(lg1.cpu().numpy(), r1)


def test_draft_prefill_wide(tiny):
    """The draft over all prompt rows (M > 16): int4 products on the
    tensor-core GEMM, with the FFN's 688 columns ending in a partial group."""
    p = tiny["prompt"].to(DEV)
    lg = torch.empty((len(p), CFG.vocab), dtype=torch.float32, device=DEV)
    tiny["model"].forward(1, p, 0, 0, logits=lg)
    torch.cuda.synchronize()
    ref, _, _ = prefill(CFG, tiny["glob"], tiny["draft"], tiny["prompt"].numpy())
    close(lg.cpu().numpy(), ref)


def _check_lossless(tiny, out, mode="greedy", temp=1.0, seed=7):
    r = decode.check_stream(CFG, tiny["glob"], tiny["layers"], tiny["prompt"].numpy(),
                            out.numpy(), mode, temp, seed, gap=1e-2)
    assert r["mismatch"] == [], r
    return r


@pytest.mark.parametrize("depth,width", [(8, 2), (0, 1), (3, 3), (8, 1)])
def test_generate_greedy_is_lossless(tiny, depth, width):
    out, st = tiny["model"].generate(tiny["prompt"], 64, depth, width)
    r = _check_lossless(tiny, out)
    assert st.cycles >= 1 and 1.0 <= st.tau <= depth + 1
    assert sum(st.accept_hist[i] for i in range(depth + 1)) == st.cycles
    # phase times: the draft (none at depth 0) and the verify pass fit in the decode time
    assert st.t_verify_ms > 0.0 and st.t_draft_ms >= 0.0 and st.t_copy_unhidden_ms >= 0.0
    if depth == 0:   # no draft levels: only the copy-stream fork sits in that span
        assert st.t_draft_ms < 0.05 * st.cycles
    else:
        assert st.t_draft_ms > 0.0
    assert st.t_draft_ms + st.t_verify_ms <= st.t_decode_ms * 1.05 + 0.5
    # the streamed originals of the offloaded layer land within each cycle
    assert 0.0 < st.t_copy_ms <= st.t_decode_ms * 1.05 + 0.5
    # the device's near-ties (its own top-2 gap < 1e-2) cover every position
    # where it picked another token than the oracle within the tie gap, or more
    assert st.near_tie_events >= 0 and st.near_tie_events <= 64


def test_generate_gumbel_is_lossless(tiny):
    out, st = tiny["model"].generate(tiny["prompt"], 48, 8, 2, mode=1, target_temp=0.6, seed=7)
    _check_lossless(tiny, out, "gumbel", 0.6, 7)


def test_graph_and_eager_agree(tiny):
    a, sa = tiny["model"].generate(tiny["prompt"], 40, 6, 2, use_graph=True)
    b, sb = tiny["model"].generate(tiny["prompt"], 40, 6, 2, use_graph=False)
    assert torch.equal(a, b) and sa.cycles == sb.cycles


def test_spec_matches_plain_on_gpu(tiny):
    plain, _ = tiny["model"].generate(tiny["prompt"], 64, 0, 1)
    spec, st = tiny["model"].generate(tiny["prompt"], 64, 8, 2)
    # both are the target's choices: each passes the teacher-forced check, and
    # the two agree token for token up to the first near-tie that either took
    # the other way (past it the contexts differ)
    rp = _check_lossless(tiny, plain)
    rs = _check_lossless(tiny, spec)
    cut = min(rp["near_tie"][:1] + rs["near_tie"][:1] + [len(plain)])
    assert torch.equal(plain[:cut], spec[:cut]), (cut, rp, rs)


def test_all_resident_chain_accepts_nearly_everything(sub):
    """With every layer resident the draft is the target itself; a width-1
    tree is then the target's own greedy chain and almost every drafted token
    is accepted (only kernel rounding differences at near-ties reject)."""
    cfg = CFG.replace(n_resident=CFG.n_layers)
    w = synthetic.make_model(cfg, norm_gain_std=0.1)
    m = sub.Model(cfg, w, max_seq=256, max_depth=6, max_width=1, max_prompt=64)
    out, st = m.generate(synthetic.make_prompt(cfg), 120, 6, 1)
    m.close()
    assert st.tau >= 0.85 * 7, st.tau
