"""The staging ring of the streamed originals ("Low-Bit Shadow" report 2.1
and 2.2 Step 4; "Speculate Deep and Accurate" card, measured effects:
asynchronous transfer): with fewer device slots than offloaded layers, a
verify pass copies layer j + ring into the slot of layer j as soon as layer j's
kernels are done.  The result must not depend on the ring size: logits
bit-equal and token streams identical to a ring that holds every offloaded
layer, and the device memory the model holds must shrink by one layer per slot
given up.  A host-resident embedding (read in place over the host link) must
give the same results too."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import decode
from helpers import oracle_model

pytestmark = pytest.mark.gpu
DEV = "cuda"
# tiny widths, five layers of which four are offloaded
CFG = synthetic.DecoderConfig("ring5", n_layers=5, hidden=256, n_heads_q=4, n_heads_kv=2,
                              head_dim=64, ffn=768, vocab=1024, rope_theta=1e4, rms_eps=1e-6,
                              n_resident=1, prompt_len=32, n_new=48, depth=6, width=2)


@pytest.fixture(scope="module")
def sub():
    import substitute_speculative_decoding_gb300 as s
    return s


@pytest.fixture(scope="module")
def weights():
    return synthetic.make_model(CFG, norm_gain_std=0.1)


def _model(sub, w, ring, embed_on_host=False):
    return sub.Model(CFG, w, max_seq=256, max_depth=8, max_width=3, max_prompt=64,
                     staging_layers=ring, embed_on_host=embed_on_host)


def _target_logits(m, prompt):
    p = prompt.to(DEV)
    lg = torch.empty((len(p), CFG.vocab), dtype=torch.float32, device=DEV)
    m.forward(0, p, 0, 0, logits=lg)
    torch.cuda.synchronize()
    return lg.cpu()


def test_ring_sizes_give_identical_results(sub, weights):
    prompt = synthetic.make_prompt(CFG)
    runs = {}
    for ring in (0, 1, 2, 3):
        m = _model(sub, weights, ring)
        lg = _target_logits(m, prompt)
        greedy, sg = m.generate(prompt, 48, 6, 2)
        gumbel, su = m.generate(prompt, 40, 6, 2, mode=1, target_temp=0.6, seed=7)
        eager, _ = m.generate(prompt, 40, 4, 3, use_graph=False)
        runs[ring] = (lg, greedy, gumbel, eager, m.device_bytes(), sg)
        m.close()
    lg0, g0, u0, e0, b0, _ = runs[0]
    layer_bytes = sum(a * b for a, b in synthetic.layer_shapes(CFG).values()) * 2
    for ring in (1, 2, 3):
        lg, g, u, e, b, st = runs[ring]
        assert torch.equal(lg, lg0), f"ring {ring}: target logits differ"
        assert torch.equal(g, g0) and torch.equal(u, u0) and torch.equal(e, e0), ring
        # four offloaded layers: a ring of r slots holds (4 - r) layers fewer
        assert b0 - b >= (4 - ring) * layer_bytes, (ring, b0, b)
        assert st.t_copy_unhidden_ms >= 0.0 and st.t_verify_ms > 0.0 and st.t_draft_ms > 0.0


def test_small_ring_is_lossless(sub, weights):
    glob, layers = oracle_model(weights)
    prompt = synthetic.make_prompt(CFG)
    m = _model(sub, weights, 1)
    for mode, temp in (("greedy", 1.0), ("gumbel", 0.6)):
        out, st = m.generate(prompt, 40, 6, 2, mode=0 if mode == "greedy" else 1,
                             target_temp=temp, seed=7)
        r = decode.check_stream(CFG, glob, layers, prompt.numpy(), out.numpy(), mode, temp, 7,
                                gap=1e-2)
        assert r["mismatch"] == [], (mode, r)
        assert 0 <= st.near_tie_events <= 40
    m.close()


def test_host_embedding_matches_device_embedding(sub, weights):
    prompt = synthetic.make_prompt(CFG)
    a = _model(sub, weights, 2)
    b = _model(sub, weights, 2, embed_on_host=True)
    assert torch.equal(_target_logits(a, prompt), _target_logits(b, prompt))
    ta, _ = a.generate(prompt, 40, 6, 2)
    tb, _ = b.generate(prompt, 40, 6, 2)
    assert torch.equal(ta, tb)
    a.close()
    b.close()
