"""Failure handling without any device fault.

* A bounded device wait that nothing completes gives up, its kernel ends
  normally, the call reports SUB_ETIMEOUT, and the context stays usable.
* Host-side fault injection (SUB_FAULT): a device allocation that fails in
  sub_model_create returns SUB_ENOMEM and frees what was allocated; a failed
  streamed copy returns SUB_ECUDA and leaves the model usable.
* Ordering of the public calls on one stream with no synchronisation between
  them: an expansion that writes the tree, then tree attention that reads it
  (programmatic launch must not let the attention read a half-written tree).
* The mma.sync fallback of the tree-shaped products (SUB_GEMM_TC=0) and of the
  draft GEMV (SUB_GEMV_TMA=0) still decode losslessly (subprocess: the
  switches are read once per process).
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import synthetic
from oracle import tree as otree

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sub():
    import substitute_speculative_decoding_gb300 as s
    return s


def test_bounded_wait_gives_up_and_the_context_survives(sub):
    before = sub.pipeline_timeouts()
    assert sub.bounded_wait_check(1024) == sub.SUB_ETIMEOUT
    assert b"gave up" in sub._lib.sub_last_error()
    # the context still runs work, and the pipelines' own count is untouched
    w = synthetic.randn_bf16((64, 256), 3, std=0.02).to(DEV)
    q, s, z = sub.w4_pack(w)
    torch.cuda.synchronize()
    assert q.shape == (64, 128)
    assert sub.pipeline_timeouts() == before
    with pytest.raises(sub.SubError):
        sub._check(sub._bounded_wait_check(0))   # argument check on the host


def _tiny(sub, max_seq=256, **kw):
    cfg = synthetic.CONFIGS["tiny"]
    w = synthetic.make_model(cfg, norm_gain_std=0.1)
    return cfg, w, sub.Model(cfg, w, max_seq=max_seq, max_depth=8, max_width=2, max_prompt=64,
                             **kw)


def test_injected_allocation_failure_frees_everything(sub, monkeypatch):
    cfg = synthetic.CONFIGS["tiny"]
    w = synthetic.make_model(cfg, norm_gain_std=0.1)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    # allocation 2 (the page table) fails after the K and V pools (~100 MB
    # each at this max_seq) were allocated
    monkeypatch.setenv("SUB_FAULT", "alloc:2")
    for _ in range(4):
        with pytest.raises(sub.SubError) as e:
            sub.Model(cfg, w, max_seq=200000, max_depth=8, max_width=2, max_prompt=64)
        assert e.value.code == sub.SUB_ENOMEM
        assert "injected" in str(e.value)
    monkeypatch.delenv("SUB_FAULT")
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free0 - free1 < 64 << 20, (free0, free1)


def test_injected_copy_failure_leaves_the_model_usable(sub, monkeypatch):
    cfg, w, m = _tiny(sub)
    prompt = synthetic.make_prompt(cfg)
    ref, _ = m.generate(prompt, 24, 4, 2)
    monkeypatch.setenv("SUB_FAULT", "h2d")
    with pytest.raises(sub.SubError) as e:
        m.generate(prompt, 24, 4, 2)
    assert e.value.code == sub.SUB_ECUDA and "injected" in str(e.value)
    monkeypatch.delenv("SUB_FAULT")
    out, st = m.generate(prompt, 24, 4, 2)
    assert torch.equal(out, ref)
    m.close()


def test_expand_then_attention_on_one_stream(sub):
    """sub_draft_expand writes the tree's levels and sub_tree_attn reads the
    ancestor lists right after, on one stream with no synchronisation."""
    depth, width, vocab = 5, 4, 4096
    hq, hkv, d, n_prefix = 8, 2, 128, 200
    n = 1 + depth * width
    tree_base = n_prefix
    kv, (k, v, pt) = sub.make_kv(1, hkv, d, n_prefix + n + 64, page_size=64, shuffle_seed=5)
    k.copy_(torch.randn_like(k, dtype=torch.float32).to(torch.bfloat16))
    v.copy_(torch.randn_like(v, dtype=torch.float32).to(torch.bfloat16))
    q = synthetic.randn_bf16((n, hq, d), 17).to(DEV)
    rng = np.random.default_rng(9)
    logits = [torch.tensor((rng.standard_normal((1 if l == 0 else width, vocab)) * 2)
                           .astype(np.float32), device=DEV) for l in range(depth)]
    tr = sub.DeviceTree(depth, width, DEV)
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for lvl in range(depth):
            sub.draft_expand(logits[lvl], 0.2, tr, lvl, stream=st)
        o = sub.tree_attn(q, kv, 0, n_prefix, tree_base, n, anc=tr.anc, depth=tr.depth, stream=st)
    st.synchronize()
    par = tr.parent.cpu().numpy()

    def rows(t, positions):
        return torch.stack([t[0, pt[p // 64], :, p % 64, :] for p in positions]).float().cpu()

    kp, vp = rows(k, range(n_prefix)), rows(v, range(n_prefix))
    kt, vt = rows(k, range(tree_base, tree_base + n)), rows(v, range(tree_base, tree_base + n))
    ref = otree.tree_attention(q.float().cpu().numpy(), kp.numpy(), vp.numpy(), kt.numpy(),
                               vt.numpy(), par, hkv)
    got = o.float().cpu().numpy()
    err = np.abs(got - ref)
    assert np.all(err <= 2e-2 + 2 ** -7 * np.abs(ref)), err.max()


_FALLBACK = r"""
import sys
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
import synthetic
import substitute_speculative_decoding_gb300 as sub
from oracle import decode
from helpers import oracle_model
cfg = synthetic.CONFIGS["tiny"]
w = synthetic.make_model(cfg, norm_gain_std=0.1)
glob, layers = oracle_model(w)
prompt = synthetic.make_prompt(cfg)
m = sub.Model(cfg, w, max_seq=256, max_depth=8, max_width=3, max_prompt=64)
for depth, width in ((8, 2), (3, 3)):
    out, st = m.generate(prompt, 48, depth, width)
    r = decode.check_stream(cfg, glob, layers, prompt.numpy(), out.numpy(), gap=1e-2)
    assert r["mismatch"] == [], r
m.close()
print("fallback ok")
"""


@pytest.mark.parametrize("env", [{"SUB_GEMM_TC": "0"}, {"SUB_GEMV_TMA": "0"},
                                 {"SUB_PDL": "0"}])
def test_fallback_paths_decode_losslessly(env):
    code = _FALLBACK.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env={**os.environ, **env},
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "fallback ok" in r.stdout, r.stdout + r.stderr
