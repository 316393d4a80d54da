"""Adaptive draft depth on the device ("Low-Bit Shadow" report 3.7 and 10.1
(3)): the stream stays the target's (teacher-forced check against the
oracle), the values that leave it off draft every level, graph replay and
eager cycles agree, and the number of levels drafted follows the oracle's
decisions on the same workload."""
import math

import numpy as np
import pytest
import torch

import synthetic
from oracle import decode
from helpers import oracle_model, oracle_draft_layers

pytestmark = pytest.mark.gpu
CFG = synthetic.CONFIGS["tiny"]
DEPTH, WIDTH, N_NEW = 8, 2, 64


@pytest.fixture(scope="module")
def tiny():
    import substitute_speculative_decoding_gb300 as s
    w = synthetic.make_model(CFG, norm_gain_std=0.1)
    glob, layers = oracle_model(w)
    draft = oracle_draft_layers(CFG, layers)
    prompt = synthetic.make_prompt(CFG)
    model = s.Model(CFG, w, max_seq=256, max_depth=DEPTH, max_width=WIDTH, max_prompt=64)
    yield dict(glob=glob, layers=layers, draft=draft, prompt=prompt, model=model)
    model.close()


def _lossless(t, out, mode="greedy", temp=1.0, seed=7):
    r = decode.check_stream(CFG, t["glob"], t["layers"], t["prompt"].numpy(), out.numpy(), mode,
                            temp, seed, gap=1e-2)
    assert r["mismatch"] == [], r


@pytest.mark.parametrize("stop", [0.0, 1.0, -math.inf, math.nan])
def test_values_that_leave_it_off(tiny, stop):
    base, sb = tiny["model"].generate(tiny["prompt"], N_NEW, DEPTH, WIDTH)
    out, st = tiny["model"].generate(tiny["prompt"], N_NEW, DEPTH, WIDTH, stop_logp=stop)
    assert torch.equal(out, base) and st.cycles == sb.cycles
    assert st.drafted_levels == st.cycles * DEPTH


@pytest.mark.parametrize("stop", [-1.0, -4.0, -12.0])
@pytest.mark.parametrize("mode,temp", [("greedy", 1.0), ("gumbel", 0.6)])
def test_adaptive_is_lossless(tiny, stop, mode, temp):
    m = 0 if mode == "greedy" else 1
    out, st = tiny["model"].generate(tiny["prompt"], N_NEW, DEPTH, WIDTH, mode=m,
                                     target_temp=temp, seed=7, stop_logp=stop)
    _lossless(tiny, out, mode, temp, 7)
    assert st.cycles <= st.drafted_levels <= st.cycles * DEPTH
    # an accepted path never runs past the levels drafted
    assert st.emitted - 1 <= st.drafted_levels + st.cycles
    assert sum(st.accept_hist[i] for i in range(DEPTH + 1)) == st.cycles


@pytest.mark.parametrize("stop", [-1.0, -4.0])
def test_graph_and_eager_agree(tiny, stop):
    a, sa = tiny["model"].generate(tiny["prompt"], 40, DEPTH, WIDTH, stop_logp=stop)
    b, sb = tiny["model"].generate(tiny["prompt"], 40, DEPTH, WIDTH, stop_logp=stop,
                                   use_graph=False)
    assert torch.equal(a, b)
    assert (sa.cycles, sa.drafted_levels) == (sb.cycles, sb.drafted_levels)


def test_levels_follow_the_oracle(tiny):
    """The oracle's SubSpec decode with the same threshold on the same weights:
    the device drafts about as many levels per cycle.  Exact equality is not
    required -- a draft near-tie at T = 0.2 can send a cycle down another
    branch, and a best score within rounding of the threshold can go either
    way -- but a level counted wrong in every cycle would miss by far more
    than the 15% allowed."""
    stop = -4.0
    rec = []
    _, emitted = decode.generate_subspec(CFG, tiny["glob"], tiny["layers"], tiny["draft"],
                                         tiny["prompt"].numpy(), N_NEW, DEPTH, WIDTH,
                                         record=rec, stop_logp=stop)
    ref_levels = np.mean([int(max(r["depth"])) for r in rec])
    assert ref_levels < DEPTH     # the threshold does stop cycles early here
    _, st = tiny["model"].generate(tiny["prompt"], N_NEW, DEPTH, WIDTH, stop_logp=stop)
    got_levels = st.drafted_levels / st.cycles
    assert abs(got_levels - ref_levels) <= 0.15 * ref_levels, (got_levels, ref_levels)
