"""The model's draft path on the TMA-streamed GEMV, int4 substitutes included,
against the oracle.  The decoder here has widths whose int4 rows hold a
multiple of 8 groups (hidden 512, FFN 1536), so its substitute layers take the
TMA kernel; the tiny decoder of the other model tests has 4- and 11-group
rows, which take the register-streamed kernel."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import decode
from oracle.model import prefill, forward_rows

from helpers import oracle_model, oracle_draft_layers

DEV = "cuda"
CFG = synthetic.DecoderConfig("tma4", n_layers=4, hidden=512, n_heads_q=8, n_heads_kv=2,
                              head_dim=64, ffn=1536, vocab=1024, rope_theta=1e4, rms_eps=1e-6,
                              n_resident=2, prompt_len=32, n_new=48, depth=6, width=3)
ATOL, RTOL = 2e-2, 1e-2


@pytest.fixture(scope="module")
def sub():
    import substitute_speculative_decoding_gb300 as s
    return s


@pytest.fixture(scope="module")
def small(sub):
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


@pytest.mark.gpu
def test_tma_draft_logits_two_levels(small):
    m = small["model"]
    p = small["prompt"].to(DEV)
    n = len(p)
    lp = torch.empty((n, CFG.vocab), dtype=torch.float32, device=DEV)
    m.forward(0, p, 0, 0, logits=lp)
    _, ks, vs = prefill(CFG, small["glob"], small["layers"], small["prompt"].numpy())
    tok, par, dep = synthetic.random_tree(2, 3, 10, CFG.vocab)
    anc = synthetic.ancestors(par, dep, 8)
    lg0 = torch.empty((1, CFG.vocab), dtype=torch.float32, device=DEV)
    m.forward(1, tok[:1].to(DEV), 0, n, depth=dep[:1].to(DEV), anc=anc[:1].to(DEV), logits=lg0)
    lg1 = torch.empty((3, CFG.vocab), dtype=torch.float32, device=DEV)
    m.forward(1, tok[1:4].contiguous().to(DEV), 1, n, depth=dep[1:4].contiguous().to(DEV),
              anc=anc[1:4].contiguous().to(DEV), logits=lg1)
    torch.cuda.synchronize()
    draft = small["draft"]
    r0, dk, dv = forward_rows(CFG, small["glob"], draft, tok[:1].numpy(), [n], ks, vs,
                              np.ones((1, n), bool), np.ones((1, 1), bool))
    close(lg0.cpu().numpy(), r0)
    pk = [np.concatenate([a, b]) for a, b in zip(ks, dk)]
    pv = [np.concatenate([a, b]) for a, b in zip(vs, dv)]
    r1, _, _ = forward_rows(CFG, small["glob"], draft, tok[1:4].numpy(), n + dep[1:4].numpy(),
                            pk, pv, np.ones((3, n + 1), bool), np.eye(3, dtype=bool))
    close(lg1.cpu().numpy(), r1)


@pytest.mark.gpu
def test_tma_draft_prefill_wide(small):
    """The draft over all 32 prompt rows: its int4 products are tree-width
    (M > 16) and run on the tensor-core GEMM with the dequantising stage."""
    p = small["prompt"].to(DEV)
    lg = torch.empty((len(p), CFG.vocab), dtype=torch.float32, device=DEV)
    small["model"].forward(1, p, 0, 0, logits=lg)
    torch.cuda.synchronize()
    ref, _, _ = prefill(CFG, small["glob"], small["draft"], small["prompt"].numpy())
    close(lg.cpu().numpy(), ref)


@pytest.mark.gpu
def test_tma_generate_is_lossless(small):
    out, st = small["model"].generate(small["prompt"], 40, 6, 3)
    r = decode.check_stream(CFG, small["glob"], small["layers"], small["prompt"].numpy(),
                            out.numpy(), "greedy", 1.0, 7, gap=1e-2)
    assert r["mismatch"] == [], r
    assert st.cycles >= 1 and 1.0 <= st.tau <= 7


@pytest.mark.gpu
def test_tma_graph_replays_match_eager(small):
    a, sa = small["model"].generate(small["prompt"], 32, 6, 3, use_graph=True)
    b, sb = small["model"].generate(small["prompt"], 32, 6, 3, use_graph=False)
    assert torch.equal(a, b) and sa.cycles == sb.cycles
