"""Verify reuse of the draft's leading layers (layer and KV sharing, "Low-Bit
Shadow" report 4.1 point 2): the verify starts at layer n_resident from the
residual stream the draft left for every tree node.  Decoding must stay the
target's (teacher-forced check against the oracle) in both modes, with and
without adaptive depth; graph and eager cycles agree; and the stream matches
decoding without reuse up to the first near-tie either run took."""
import pytest
import torch

import synthetic
from oracle import decode
from helpers import oracle_model

pytestmark = pytest.mark.gpu
TMA4 = synthetic.DecoderConfig("tma4", n_layers=4, hidden=512, n_heads_q=8, n_heads_kv=2,
                               head_dim=64, ffn=1536, vocab=1024, rope_theta=1e4, rms_eps=1e-6,
                               n_resident=2, prompt_len=32, n_new=48, depth=6, width=3)
CASES = {"tiny": synthetic.CONFIGS["tiny"], "tma4": TMA4}


@pytest.fixture(scope="module", params=sorted(CASES))
def mdl(request):
    import substitute_speculative_decoding_gb300 as s
    cfg = CASES[request.param]
    w = synthetic.make_model(cfg, norm_gain_std=0.1)
    glob, layers = oracle_model(w)
    prompt = synthetic.make_prompt(cfg)
    model = s.Model(cfg, w, max_seq=256, max_depth=8, max_width=3, max_prompt=64)
    yield dict(cfg=cfg, glob=glob, layers=layers, prompt=prompt, model=model)
    model.close()


def _check(t, out, mode, temp):
    r = decode.check_stream(t["cfg"], t["glob"], t["layers"], t["prompt"].numpy(), out.numpy(),
                            mode, temp, 7, gap=1e-2)
    assert r["mismatch"] == [], r
    return r


@pytest.mark.parametrize("mode,temp", [("greedy", 1.0), ("gumbel", 0.6)])
@pytest.mark.parametrize("stop", [None, -4.0])
def test_reuse_is_lossless(mdl, mode, temp, stop):
    out, st = mdl["model"].generate(mdl["prompt"], 48, 8, 3, mode=int(mode == "gumbel"),
                                    target_temp=temp, seed=7, stop_logp=stop, verify_reuse=True)
    _check(mdl, out, mode, temp)
    assert st.cycles >= 1 and 1.0 <= st.tau <= 9


def test_graph_and_eager_agree(mdl):
    a, sa = mdl["model"].generate(mdl["prompt"], 40, 6, 3, verify_reuse=True)
    b, sb = mdl["model"].generate(mdl["prompt"], 40, 6, 3, verify_reuse=True, use_graph=False)
    assert torch.equal(a, b) and sa.cycles == sb.cycles


def test_same_stream_as_without_reuse(mdl):
    plain, sp = mdl["model"].generate(mdl["prompt"], 64, 8, 3)
    reuse, sr = mdl["model"].generate(mdl["prompt"], 64, 8, 3, verify_reuse=True)
    rp = _check(mdl, plain, "greedy", 1.0)
    rr = _check(mdl, reuse, "greedy", 1.0)
    cut = min(rp["near_tie"][:1] + rr["near_tie"][:1] + [len(plain)])
    assert torch.equal(plain[:cut], reuse[:cut]), (cut, rp, rr)
