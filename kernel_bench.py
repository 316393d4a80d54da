"""Kernel micro-benchmarks on single shapes of the decode path (for timing and
for profiler captures on a small case), a measurement tool beside bench.py.

    python kernel_bench.py <case> [--iters N]

Cases (Qwen2.5-7B draft/verify shapes; operand sets rotate over more memory
than the 129 MB L2):
  gemv_bf16   bf16 weights 18944x3584, M = 8 (a resident FFN matrix)
  gemv_w4     int4 weights 37888x3584, M = 8 (a substitute gate+up pair)
  attn_draft  8 tree queries, 28/4 heads, d 128, 640 committed keys
  attn_verify 385 tree queries, same heads and keys
  attn32      the Qwen2.5-32B attention sweep (40/8 heads; 385 or 8 queries over 1k, 4k
              and 16k committed keys)
  attn32_draft16k  its draft-shaped 16k-key point alone
  gemm_bf16   bf16 weights 18944x3584, M = 385 (a verify FFN matrix, tcgen05)
  gemm_w4     int4 weights 18944x3584, M = 385 (tcgen05 with the dequantising stage)
  gemv_{bf16,w4}_{down,o}  down projection 3584x18944 / o projection 3584x3584, M = 8
  w4_wide     int4 37888x3584 at M = 8, 16, 24, 32, 48 (TMA GEMV to 32 rows, then tcgen05)
  w4_mix      the four int4 substitute matrices of one layer (o, gate, up, down)
              in turn, M = 8
  wq_mix2, wq_mix3  the same with 2- or 3-bit substitutes
  draft_level one draft forward of 8 tree nodes through the whole Qwen2.5-7B-shaped
              model (11 resident + 17 int4 layers, lm_head), inside the NVTX range
              "draft_level" (the second of two runs)
  verify_pass one target forward over a 385-node tree (offloaded layers streamed),
              inside the NVTX range "verify_pass"
Prints one JSON line: milliseconds per launch and algorithmic GB/s, TFLOP/s.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import synthetic  # noqa: E402
import substitute_speculative_decoding_gb300 as sub  # noqa: E402


def _time(fn, iters):
    """Milliseconds per call, device-side: the calls are captured once in a
    CUDA graph and the graph is replayed, so host launch cost drops out."""
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(iters):
            fn(i)
    g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(3):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (3 * iters)


def _model_pass(case):
    """One draft level (8 rows at the deepest level) or one verify pass of the
    Qwen2.5-7B-shaped model after a 512-token prefill."""
    cfg = synthetic.CONFIGS["qwen7b"]
    dev = torch.device("cuda", torch.cuda.current_device())
    w = synthetic.make_model(cfg, device=dev)
    m = sub.Model(cfg, w, max_seq=2048, max_depth=48, max_width=8, max_prompt=512)
    for i in range(cfg.n_resident, cfg.n_layers):
        for n in synthetic.LAYER_TENSORS:
            w["layers"][i][n] = w["layers"][i][n].to("cpu")
    torch.cuda.empty_cache()
    dcfg = sub.Model.decode_cfg(48, 8, 0.2)
    m.prefill(synthetic.make_prompt(cfg), dcfg)
    tok, par, dep = synthetic.random_tree(48, 8, 1, cfg.vocab)
    anc = synthetic.ancestors(par, dep, 48).to(dev)
    tok, dep = tok.to(dev), dep.to(dev)
    logits = torch.empty(385, cfg.vocab, device=dev)
    s0 = 1 + 46 * 8
    out = {}
    for it in range(2):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if it == 1:
            torch.cuda.nvtx.range_push(case)
        e0.record()
        if case == "draft_level":
            m.forward(1, tok[s0:s0 + 8], s0, 600, depth=dep[s0:s0 + 8], anc=anc[s0:s0 + 8],
                      logits=logits)
        else:
            m.forward(0, tok, 0, 600, depth=dep, anc=anc, logits=logits)
        e1.record()
        torch.cuda.synchronize()
        if it == 1:
            torch.cuda.nvtx.range_pop()
        out["ms"] = e0.elapsed_time(e1)
    m.close()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--iters", type=int, default=20)
    a = ap.parse_args()
    dev = "cuda"
    res = {"case": a.case}
    if a.case in ("gemv_bf16_down", "gemv_bf16_o", "gemv_w4_down", "gemv_w4_o"):
        n, k = (3584, 18944) if a.case.endswith("down") else (3584, 3584)
        reps = 4
        x = torch.randn(8, k, device=dev).to(torch.bfloat16)
        y = torch.empty(8, n, device=dev, dtype=torch.bfloat16)
        if "w4" in a.case:
            packs = [synthetic.random_w4(n, k, s, dev) for s in range(reps)]
            ms = _time(lambda i: sub.w4_gemm(x, *packs[i % reps], n, k, out=y), a.iters)
            byt = n * (k // 64) * 36 + 8 * (n + k) * 2
        else:
            ws = [synthetic.randn_bf16((n, k), s, 0.02, dev) for s in range(reps)]
            ms = _time(lambda i: sub.bf16_gemm(x, ws[i % reps], out=y), a.iters)
            byt = n * k * 2 + 8 * (n + k) * 2
        res.update(ms=ms, gbs=byt / ms / 1e6)
    elif a.case == "w4_wide":
        # int4 37888 x 3584 (a Qwen2.5-7B gate+up pair, 4 packed copies rotate
        # past L2) at M = 8, 16, 24, 32, 48: the TMA GEMV with 1, 2, 4, 4 token
        # tiles of 8, then the tensor-core GEMM
        n, k, reps = 37888, 3584, 4
        packs = [synthetic.random_w4(n, k, s, dev) for s in range(reps)]
        for m in (8, 16, 24, 32, 48):
            x = torch.randn(m, k, device=dev).to(torch.bfloat16)
            y = torch.empty(m, n, device=dev, dtype=torch.bfloat16)
            ms = _time(lambda i: sub.w4_gemm(x, *packs[i % reps], n, k, out=y), a.iters)
            byt = n * (k // 64) * 36 + m * (n + k) * 2
            res[f"M{m}"] = dict(ms=round(ms, 5), gbs=round(byt / ms / 1e6, 1),
                                tflops=round(2 * m * n * k / ms / 1e9, 2))
    elif a.case == "w4_mix":
        # the four int4 substitute matrices of a Qwen2.5-7B layer in turn (o,
        # gate, up, down), M = 8: the shapes bench.py's roofline cycles through
        shapes = [(3584, 3584), (18944, 3584), (18944, 3584), (3584, 18944)]
        packs = [synthetic.random_w4(n, k, 11 + i, dev) for i, (n, k) in enumerate(shapes)]
        xs = {k: torch.randn(8, k, device=dev).to(torch.bfloat16) for _, k in shapes}
        ys = {n: torch.empty(8, n, device=dev, dtype=torch.bfloat16) for n, _ in shapes}

        def run(i):
            n, k = shapes[i % 4]
            sub.w4_gemm(xs[k], *packs[i % 4], n, k, out=ys[n])
        ms = _time(run, a.iters)
        byt = sum(n * ((k + 63) // 64) * 36 + 8 * (n + k) * 2 for n, k in shapes) / 4
        res.update(ms=ms, gbs=byt / ms / 1e6, bytes_per_launch=byt)
    elif a.case in ("wq_mix2", "wq_mix3"):
        # the same four shapes with 2- or 3-bit substitutes (random bf16 weights
        # packed on the device; 4 copies of each shape rotate past L2)
        bits = 2 if a.case == "wq_mix2" else 3
        shapes = [(3584, 3584), (18944, 3584), (18944, 3584), (3584, 18944)]
        packs = [sub.wq_pack(synthetic.randn_bf16((n, k), 11 + 4 * i + r, 0.02, dev), bits)
                 for i, (n, k) in enumerate(shapes) for r in range(4)]
        xs = {k: torch.randn(8, k, device=dev).to(torch.bfloat16) for _, k in shapes}
        ys = {n: torch.empty(8, n, device=dev, dtype=torch.bfloat16) for n, _ in shapes}

        def run(i):
            n, k = shapes[i % 4]
            sub.wq_gemm(xs[k], *packs[(i % 4) * 4 + (i // 4) % 4], n, k, bits, out=ys[n])
        ms = _time(run, a.iters)
        byt = sum(n * ((k + 63) // 64) * (8 * bits + 4) + 8 * (n + k) * 2 for n, k in shapes) / 4
        res.update(ms=ms, gbs=byt / ms / 1e6, bytes_per_launch=byt)
    elif a.case in ("gemv_bf16", "gemm_bf16"):
        m = 8 if a.case == "gemv_bf16" else 385
        ws = [synthetic.randn_bf16((18944, 3584), s, 0.02, dev) for s in range(4)]
        x = torch.randn(m, 3584, device=dev).to(torch.bfloat16)
        y = torch.empty(m, 18944, device=dev, dtype=torch.bfloat16)
        ms = _time(lambda i: sub.bf16_gemm(x, ws[i % 4], out=y), a.iters)
        byt = 18944 * 3584 * 2 + m * (3584 + 18944) * 2
        res.update(ms=ms, gbs=byt / ms / 1e6, tflops=2 * m * 18944 * 3584 / ms / 1e9)
    elif a.case == "gemm_w4":
        m, n, k = 385, 18944, 3584
        packs = [synthetic.random_w4(n, k, s, dev) for s in range(4)]
        x = torch.randn(m, k, device=dev).to(torch.bfloat16)
        y = torch.empty(m, n, device=dev, dtype=torch.bfloat16)
        ms = _time(lambda i: sub.w4_gemm(x, *packs[i % 4], n, k, out=y), a.iters)
        byt = n * (k // 64) * 36 + m * (n + k) * 2
        res.update(ms=ms, gbs=byt / ms / 1e6, tflops=2 * m * n * k / ms / 1e9)
    elif a.case == "gemv_w4":
        packs = [synthetic.random_w4(37888, 3584, s, dev) for s in range(4)]
        x = torch.randn(8, 3584, device=dev).to(torch.bfloat16)
        y = torch.empty(8, 37888, device=dev, dtype=torch.bfloat16)
        ms = _time(lambda i: sub.w4_gemm(x, *packs[i % 4], 37888, 3584, out=y), a.iters)
        byt = 37888 * 56 * 36 + 8 * (3584 + 37888) * 2
        res.update(ms=ms, gbs=byt / ms / 1e6)
    elif a.case in ("attn_draft", "attn_verify"):
        depth, width, hq, hkv, d, n_prefix = 48, 8, 28, 4, 128, 640
        tok, par, dep = synthetic.random_tree(depth, width, 1, 1000)
        anc = synthetic.ancestors(par, dep, depth).to(dev)
        dep = dep.to(dev)
        n_tree = len(par)
        kv, keep = sub.make_kv(1, hkv, d, n_prefix + n_tree + 64)
        keep[0].normal_()
        keep[1].normal_()
        nq = width if a.case == "attn_draft" else n_tree
        q = torch.randn(nq, hq, d, device=dev).to(torch.bfloat16)
        an, dp = anc[-nq:].contiguous(), dep[-nq:].contiguous()
        ms = _time(lambda i: sub.tree_attn(q, kv, 0, n_prefix, n_prefix, n_tree, anc=an,
                                           depth=dp), a.iters)
        byt = (n_prefix + n_tree) * hkv * d * 4 + 2 * nq * hq * d * 2
        res.update(ms=ms, gbs=byt / ms / 1e6)
    elif a.case == "attn32":
        # the Qwen2.5-32B attention sweep of bench.py: 40/8 heads, d 128, a
        # depth-48 width-8 tree over 1k/4k/16k committed keys, 385 or 8 queries,
        # key/value copies rotated over at least 4x L2
        import math
        hq, hkv, d = 40, 8, 128
        tok, par, dep = synthetic.random_tree(48, 8, 3, 1000)
        anc = synthetic.ancestors(par, dep, 48).to(dev)
        dep = dep.to(dev)
        n_tree = len(par)
        for lkv in (1024, 4096, 16384):
            kv_bytes = (lkv + n_tree) * hkv * d * 4
            nc = max(2, math.ceil(4 * 129 * 2 ** 20 / kv_bytes))
            caches = []
            for _ in range(nc):
                kv, keep = sub.make_kv(1, hkv, d, lkv + n_tree + 64)
                keep[0].normal_()
                keep[1].normal_()
                caches.append((kv, keep))
            for nq, tag in ((n_tree, "verify385"), (8, "draft8")):
                q = torch.randn(nq, hq, d, device=dev).to(torch.bfloat16)
                an, dp = anc[-nq:].contiguous(), dep[-nq:].contiguous()
                ms = _time(lambda i: sub.tree_attn(q, caches[i % nc][0], 0, lkv, lkv, n_tree,
                                                   anc=an, depth=dp), max(a.iters, nc))
                byt = kv_bytes + 4 * nq * hq * d
                res[f"{tag}_kv{lkv}"] = dict(ms=round(ms, 5), gbs=round(byt / ms / 1e6, 1))
            del caches
    elif a.case == "attn32_draft16k":
        # one shape of that sweep alone, for a profiler capture: 8 draft
        # queries of a depth-48 width-8 tree over 16384 committed keys
        import math
        hq, hkv, d, lkv = 40, 8, 128, 16384
        tok, par, dep = synthetic.random_tree(48, 8, 3, 1000)
        anc = synthetic.ancestors(par, dep, 48).to(dev)
        dep = dep.to(dev)
        n_tree = len(par)
        kv_bytes = (lkv + n_tree) * hkv * d * 4
        nc = max(2, math.ceil(4 * 129 * 2 ** 20 / kv_bytes))
        caches = []
        for _ in range(nc):
            kv, keep = sub.make_kv(1, hkv, d, lkv + n_tree + 64)
            keep[0].normal_()
            keep[1].normal_()
            caches.append((kv, keep))
        q = torch.randn(8, hq, d, device=dev).to(torch.bfloat16)
        an, dp = anc[-8:].contiguous(), dep[-8:].contiguous()
        ms = _time(lambda i: sub.tree_attn(q, caches[i % nc][0], 0, lkv, lkv, n_tree, anc=an,
                                           depth=dp), max(a.iters, nc))
        byt = kv_bytes + 4 * 8 * hq * d
        res.update(ms=ms, gbs=byt / ms / 1e6)
    elif a.case in ("draft_level", "verify_pass"):
        res.update(_model_pass(a.case))
    else:
        raise SystemExit(f"unknown case {a.case}")
    print(json.dumps(res))


if __name__ == "__main__":
    main()
