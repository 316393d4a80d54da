"""2- and 3-bit and per-layer mixed-precision substitutes on the device
("Low-Bit Shadow" report 5.1 point 2, 10.1 (2), 10.2 (10)), and HQQ zero
points (Critique 3, 6.2), against the oracle: packed codes, scales, zeros
and dequantised values bit-exact; the GEMV and the wide product within the
bf16 output rounding; draft logits of mixed-precision and HQQ models within
the stated tolerance; and decoding that stays lossless with any of them."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import quant, decode
from oracle.model import prefill, forward_rows
from helpers import oracle_model, oracle_draft_layers

pytestmark = pytest.mark.gpu
DEV = "cuda"
ATOL, RTOL = 2e-2, 1e-2


@pytest.fixture(scope="module")
def sub():
    import substitute_speculative_decoding_gb300 as s
    return s


def np32(t):
    return t.detach().float().cpu().numpy()


def close(got, ref, atol=ATOL, rtol=RTOL):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    assert np.all(err <= bound), f"max excess {np.max(err - bound):.3e}, max err {err.max():.3e}"


# ------------------------------------------------------------------ kernels --
@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("n,k", [(48, 688), (64, 3584), (16, 64), (40, 200)])
def test_wq_pack_and_dequant_bit_exact(sub, bits, n, k):
    w = synthetic.randn_bf16((n, k), n * 7 + k + bits, std=0.02)
    w[3, :64] = 0.25                       # a constant group
    w[5, 64:128] = -0.0078125
    q, s, z = sub.wq_pack(w.to(DEV), bits)
    rq, rs, rz = quant.wq_pack(np32(w), bits)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(np32(s), rs) and np.array_equal(np32(z), rz)
    deq = sub.wq_dequant(q, s, z, k, bits)
    assert np.array_equal(np32(deq), quant.wq_dequant(rq, rs, rz, k, bits))


@pytest.mark.parametrize("bits", [2, 3])
@pytest.mark.parametrize("m", [1, 8, 13, 16, 17, 48])
@pytest.mark.parametrize("n,k", [(256, 688), (4608, 3584), (96, 512)])
def test_wq_gemm(sub, bits, m, n, k):
    w = synthetic.randn_bf16((n, k), 3 + n + k + bits, std=0.02)
    q, s, z = sub.wq_pack(w.to(DEV), bits)
    x = synthetic.randn_bf16((m, k), 11 + m + k)
    y = sub.wq_gemm(x.to(DEV), q, s, z, n, k, bits)
    ref = quant.wq_gemm(np32(x), q.cpu().numpy(), np32(s), np32(z), k, bits)
    # bf16 output rounding (2^-8 relative) + the GEMV's unrounded dequant
    scale = np.abs(ref).max()
    close(np32(y), ref, atol=3e-3 * scale, rtol=2 ** -8)


@pytest.mark.parametrize("bits", [2, 3])
@pytest.mark.parametrize("k", [256, 1024])
def test_wq_gemm_identity_is_exact_dequant(sub, bits, k):
    """Identity rows through the GEMV give s (q - z) in fp32, rounded once to
    bf16 on output: the dequantised values exactly (K = 256: the
    register-streamed kernel; K = 1024, whole stages of 8 groups: the
    TMA-streamed one)."""
    w = synthetic.randn_bf16((64, k), 5 + bits, std=0.02)
    q, s, z = sub.wq_pack(w.to(DEV), bits)
    deq = sub.wq_dequant(q, s, z, k, bits)
    eye = torch.eye(k, dtype=torch.bfloat16, device=DEV)
    for r0 in range(0, k, 16):
        y = sub.wq_gemm(eye[r0:r0 + 16].contiguous(), q, s, z, 64, k, bits)
        assert torch.equal(y.t().contiguous(), deq[:, r0:r0 + 16])
    y = sub.wq_gemm(eye, q, s, z, 64, k, bits)            # M = 256: dequant + bf16 GEMM
    assert torch.equal(y.t().contiguous(), deq)


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("iters", [1, 20])
@pytest.mark.parametrize("n,k", [(48, 688), (64, 3584), (40, 200)])
def test_hqq_pack_bit_exact(sub, bits, iters, n, k):
    """HQQ zero optimisation: codes, scales and zeros equal the oracle's bit
    for bit (fp32 steps and one summation order on both sides)."""
    w = synthetic.randn_bf16((n, k), n + k + bits, std=0.02)
    w[3, :64] = 0.25                       # a constant group
    q, s, z = sub.wq_pack_hqq(w.to(DEV), bits, iters)
    rq, rs, rz = quant.wq_pack_hqq(np32(w), bits, iters)
    assert np.array_equal(np32(s), rs)
    assert np.array_equal(np32(z), rz)
    assert np.array_equal(q.cpu().numpy(), rq)


def test_bad_bits_rejected(sub):
    w = torch.zeros((16, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(sub.SubError):
        sub.wq_pack(w, 5)
    with pytest.raises(sub.SubError):
        sub.wq_pack(w, 1)


# -------------------------------------------------------------------- model --
TMA4 = synthetic.DecoderConfig("tma4", n_layers=4, hidden=512, n_heads_q=8, n_heads_kv=2,
                               head_dim=64, ffn=1536, vocab=1024, rope_theta=1e4, rms_eps=1e-6,
                               n_resident=1, prompt_len=32, n_new=48, depth=6, width=3)
TINY = synthetic.CONFIGS["tiny"]
CASES = {
    "tiny-2bit": (TINY, 2, 0),
    "tiny-3bit": (TINY, 3, 0),
    "tma4-mixed": (TMA4, [4, 4, 2, 3], 0),   # layer 0 resident; substitutes 4, 2, 3 bits
    "tma4-hqq": (TMA4, 4, 20),               # 4-bit substitutes with HQQ zero points
}


@pytest.fixture(scope="module", params=sorted(CASES))
def lowbit(sub, request):
    cfg, bits, hqq = CASES[request.param]
    w = synthetic.make_model(cfg, norm_gain_std=0.1)
    glob, layers = oracle_model(w)
    draft = oracle_draft_layers(cfg, layers, bits, hqq_iters=hqq)
    prompt = synthetic.make_prompt(cfg)
    model = sub.Model(cfg, w, max_seq=256, max_depth=8, max_width=3, max_prompt=64, bits=bits,
                      hqq_iters=hqq)
    yield dict(cfg=cfg, glob=glob, layers=layers, draft=draft, prompt=prompt, model=model)
    model.close()


def test_draft_logits_two_levels(lowbit):
    cfg, m = lowbit["cfg"], lowbit["model"]
    p = lowbit["prompt"].to(DEV)
    n = len(p)
    lp = torch.empty((n, cfg.vocab), dtype=torch.float32, device=DEV)
    m.forward(0, p, 0, 0, logits=lp)
    _, ks, vs = prefill(cfg, lowbit["glob"], lowbit["layers"], lowbit["prompt"].numpy())
    tok, par, dep = synthetic.random_tree(2, 3, 10, cfg.vocab)
    anc = synthetic.ancestors(par, dep, 8)
    lg0 = torch.empty((1, cfg.vocab), dtype=torch.float32, device=DEV)
    m.forward(1, tok[:1].to(DEV), 0, n, depth=dep[:1].to(DEV), anc=anc[:1].to(DEV), logits=lg0)
    lg1 = torch.empty((3, cfg.vocab), dtype=torch.float32, device=DEV)
    m.forward(1, tok[1:4].contiguous().to(DEV), 1, n, depth=dep[1:4].contiguous().to(DEV),
              anc=anc[1:4].contiguous().to(DEV), logits=lg1)
    torch.cuda.synchronize()
    draft = lowbit["draft"]
    r0, dk, dv = forward_rows(cfg, lowbit["glob"], draft, tok[:1].numpy(), [n], ks, vs,
                              np.ones((1, n), bool), np.ones((1, 1), bool))
    close(lg0.cpu().numpy(), r0)
    pk = [np.concatenate([a, b]) for a, b in zip(ks, dk)]
    pv = [np.concatenate([a, b]) for a, b in zip(vs, dv)]
    r1, _, _ = forward_rows(cfg, lowbit["glob"], draft, tok[1:4].numpy(), n + dep[1:4].numpy(),
                            pk, pv, np.ones((3, n + 1), bool), np.eye(3, dtype=bool))
    close(lg1.cpu().numpy(), r1)


@pytest.mark.parametrize("mode,temp", [("greedy", 1.0), ("gumbel", 0.6)])
def test_generate_is_lossless(lowbit, mode, temp):
    out, st = lowbit["model"].generate(lowbit["prompt"], 40, 6, 3, mode=int(mode == "gumbel"),
                                       target_temp=temp, seed=7)
    r = decode.check_stream(lowbit["cfg"], lowbit["glob"], lowbit["layers"],
                            lowbit["prompt"].numpy(), out.numpy(), mode, temp, 7, gap=1e-2)
    assert r["mismatch"] == [], r
    assert st.cycles >= 1 and 1.0 <= st.tau <= 7


def test_wide_draft_needs_four_bits(sub, lowbit):
    """A draft forward over more than 16 rows with 2- or 3-bit substitutes is
    refused (those widths have the GEMV only on the model path); with 4-bit
    HQQ substitutes it runs the tensor-core GEMM and matches the oracle."""
    p = lowbit["prompt"].to(DEV)
    if lowbit["model"].w4 and all(q.shape[1] * 2 == 64 * s.shape[1]
                                  for q, s, _ in lowbit["model"].w4.values()):
        lg = torch.empty((len(p), lowbit["cfg"].vocab), dtype=torch.float32, device=DEV)
        lowbit["model"].forward(1, p, 0, 0, logits=lg)
        torch.cuda.synchronize()
        ref, _, _ = prefill(lowbit["cfg"], lowbit["glob"], lowbit["draft"],
                            lowbit["prompt"].numpy())
        close(lg.cpu().numpy(), ref)
        return
    lg = torch.empty((len(p), lowbit["cfg"].vocab), dtype=torch.float32, device=DEV)
    with pytest.raises(sub.SubError):
        lowbit["model"].forward(1, p, 0, 0, logits=lg)
    torch.cuda.synchronize()
