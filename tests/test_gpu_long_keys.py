"""Draft attention over long key ranges in the decode loop: with 8k keys or
more and few query rows, a draft level's tree attention splits the keys 32
ways, as four thread-block clusters of 8 whose partials meet in the model's
cross-cluster scratch.  Two models exercise it end to end and are checked
against the oracle by teacher forcing: one whose prompt alone is past 8k keys
(eager and graph cycles both take 32 splits), and one sized for a long
context but given a short prompt (the captured graphs take 32 splits from the
capacity, so most key splits and whole clusters are empty)."""
import pytest

import synthetic
from oracle import decode
from helpers import oracle_model

pytestmark = pytest.mark.gpu


def _cfg(name, prompt_len):
    return synthetic.DecoderConfig(name, n_layers=2, hidden=512, n_heads_q=4, n_heads_kv=1,
                                   head_dim=128, ffn=1024, vocab=512, rope_theta=1e6,
                                   rms_eps=1e-6, n_resident=1, prompt_len=prompt_len, n_new=24,
                                   depth=6, width=3)


@pytest.fixture(scope="module")
def sub():
    import substitute_speculative_decoding_gb300 as s
    return s


@pytest.mark.parametrize("prompt_len,use_graph", [(8256, True), (8256, False), (40, True)])
def test_long_key_draft_attention_is_lossless(sub, prompt_len, use_graph):
    cfg = _cfg(f"long{prompt_len}", prompt_len)
    w = synthetic.make_model(cfg, norm_gain_std=0.1)
    glob, layers = oracle_model(w)
    prompt = synthetic.make_prompt(cfg)
    model = sub.Model(cfg, w, max_seq=8400, max_depth=6, max_width=3, max_prompt=8256)
    try:
        out, st = model.generate(prompt, 24, 6, 3, use_graph=use_graph)
    finally:
        model.close()
    assert st.cycles >= 1
    r = decode.check_stream(cfg, glob, layers, prompt.numpy(), out.numpy(), "greedy", 1.0, 0,
                            gap=1e-2)
    assert r["mismatch"] == [], r
