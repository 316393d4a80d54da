"""The decode options together on one model: a staging ring with fewer slots
than offloaded layers, adaptive depth (conditional graph levels), verify
reuse of the leading layers, mixed 4/2/3-bit substitutes, greedy and Gumbel
sampling.  Every combination must stay the target's stream (teacher-forced
against the oracle), and graph replay must equal eager cycles."""
import pytest
import torch

import synthetic
from oracle import decode
from helpers import oracle_model

pytestmark = pytest.mark.gpu
CFG = synthetic.DecoderConfig("combo5", n_layers=5, hidden=512, n_heads_q=8, n_heads_kv=2,
                              head_dim=64, ffn=1536, vocab=1024, rope_theta=1e4, rms_eps=1e-6,
                              n_resident=2, prompt_len=32, n_new=48, depth=6, width=3)
BITS = [4, 4, 4, 2, 3]   # resident layers' entries are ignored


@pytest.fixture(scope="module")
def combo():
    import substitute_speculative_decoding_gb300 as s
    w = synthetic.make_model(CFG, norm_gain_std=0.1)
    glob, layers = oracle_model(w)
    prompt = synthetic.make_prompt(CFG)
    model = s.Model(CFG, w, max_seq=256, max_depth=8, max_width=3, max_prompt=64,
                    staging_layers=1, bits=BITS)
    yield dict(glob=glob, layers=layers, prompt=prompt, model=model)
    model.close()


def _lossless(t, out, mode, temp):
    r = decode.check_stream(CFG, t["glob"], t["layers"], t["prompt"].numpy(), out.numpy(), mode,
                            temp, 7, gap=1e-2)
    assert r["mismatch"] == [], r


@pytest.mark.parametrize("mode,temp", [("greedy", 1.0), ("gumbel", 0.6)])
@pytest.mark.parametrize("stop", [None, -3.0])
@pytest.mark.parametrize("reuse", [False, True])
def test_combinations_are_lossless(combo, mode, temp, stop, reuse):
    out, st = combo["model"].generate(combo["prompt"], 48, 8, 3, mode=int(mode == "gumbel"),
                                      target_temp=temp, seed=7, stop_logp=stop,
                                      verify_reuse=reuse)
    _lossless(combo, out, mode, temp)
    assert st.cycles >= 1 and st.t_copy_ms > 0.0
    assert st.cycles <= st.drafted_levels <= st.cycles * 8


@pytest.mark.parametrize("stop,reuse", [(-3.0, True), (None, True), (-3.0, False)])
def test_graph_equals_eager(combo, stop, reuse):
    a, sa = combo["model"].generate(combo["prompt"], 40, 8, 3, stop_logp=stop, verify_reuse=reuse)
    b, sb = combo["model"].generate(combo["prompt"], 40, 8, 3, stop_logp=stop, verify_reuse=reuse,
                                    use_graph=False)
    assert torch.equal(a, b)
    assert (sa.cycles, sa.drafted_levels) == (sb.cycles, sb.drafted_levels)
