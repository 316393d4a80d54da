#!/usr/bin/env python
"""SubSpec decode benchmark on GB300.

One step = one SubSpec decode cycle: D = 48 draft levels (shared resident bf16
layers + int4 substitutes, width 8, draft temperature 0.2) -> one target pass
verifying all 385 tree nodes (the offloaded layers' bf16 originals streamed
from pinned host memory on a copy stream) -> accept -> KV compaction.
`value` is the generated tokens/s of K device-timed cycles with every input
resident; `e2e` is sub_generate (host prompt in, host tokens out, prefill
included).

Workloads (--workload):
  qwen7b   Qwen2.5-7B-shaped decoder, 11 resident + 17 int4 layers, prompt 512,
           greedy (the default; 256 tokens for e2e)
  llama8b  Llama-3.1-8B-shaped decoder (RoPE theta 5e5, eps 1e-5), 8 resident +
           24 int4 layers, prompt 1024, greedy (512 tokens for e2e)
  qwen32b  Qwen2.5-32B-shaped decoder under a 24 GB device budget: 1 resident
           layer, 63 int4 substitutes, a 2-slot staging ring for the streamed
           originals, the embedding in pinned host memory; prompt 256,
           Gumbel-max sampling at T = 0.6 with seed 7 (e2e: --new tokens, 256
           by default; the workload's full length is 4096)

Flags: --gpus N (replicas; one process per GPU under torchrun), --steps K,
--warmup W, --impl reference (the CPU oracle arm), --quick (skip the kernel
sweep, e2e and the CPU baseline: for profiler launch lists), --new N,
--stop-logp X (adaptive depth for the timed cycles and the e2e run; the
default line is the fixed-depth workload).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synthetic  # noqa: E402

METRIC = "generated tokens/s and τ (1 GB300); W4 GEMM + tree-attn GB/s vs 8 TB/s"
DEPTH, WIDTH, DRAFT_T = 48, 8, 0.2
# adaptive-depth thresholds (cumulative sharpened log-probability) and the
# tokens each of their decodes generates
ADAPTIVE_STOPS, ADAPTIVE_NEW = (-0.5, -2.0, -6.0, -16.0), 128
# fixed tree depths of the depth sweep (the model is built for the deepest)
DEPTH_SWEEP = (8, 16, 32, 48, 64)
L2_BYTES = 129 * 2 ** 20
ROTATE_BYTES = 4 * L2_BYTES      # operand sets rotated per timed sweep point

WORKLOADS = {
    "qwen7b": dict(cfg="qwen7b", staging=0, embed_on_host=False, e2e_new=256,
                   text="Qwen2.5-7B-shaped decoder (28 layers, hidden 3584, 28/4 heads, FFN "
                        "18944, vocab 152064), random bf16 init; 11 resident layers + 17 int4 "
                        "g64 substitutes with pinned-host bf16 originals streamed per verify; "
                        "prompt 512; SubSpec tree depth 48, width 8, draft T 0.2, greedy; "
                        "step = one draft/verify/accept cycle"),
    "llama8b": dict(cfg="llama8b", staging=0, embed_on_host=False, e2e_new=512,
                    text="Llama-3.1-8B-shaped decoder (32 layers, hidden 4096, 32/8 heads, FFN "
                         "14336, vocab 128256, RoPE theta 5e5), random bf16 init; 8 resident + "
                         "24 int4 g64 substitutes with pinned-host originals; prompt 1024; "
                         "depth 48, width 8, greedy; step = one cycle"),
    "qwen32b": dict(cfg="qwen32b", staging=2, embed_on_host=True, e2e_new=256, sweep_new=32,
                    lowbit=False,
                    text="Qwen2.5-32B-shaped decoder (64 layers, hidden 5120, 40/8 heads, FFN "
                         "27648, vocab 152064), random bf16 init, 24 GB device budget: 1 resident "
                         "layer + 63 int4 g64 substitutes, 2-slot staging ring for the pinned-host "
                         "originals, host-resident embedding; prompt 256; depth 48, width 8, "
                         "Gumbel-max T 0.6 seed 7; step = one cycle"),
}


# ------------------------------------------------------------------ setup --
def dist_setup():
    """Rank, world size and local rank from the launcher's environment; with
    more than one rank, a process group (NCCL on GPUs, gloo without them:
    replicas exchange only their timings and counts, no data)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce(world, value, op):
    """max or sum of one number over the ranks."""
    if world == 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(world, tokens, ms):
    """Whole-job throughput of N replicas: every rank's tokens over the
    slowest rank's time -> (tokens over all ranks, max ms, tokens/s)."""
    ms_max = reduce(world, ms, "max")
    tokens_all = reduce(world, tokens, "sum")
    return tokens_all, ms_max, tokens_all / (ms_max / 1e3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sus=p["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class Clocks:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm = [float(r[1]) for r in self.rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            if len(r) < 9:
                continue
            for i, n in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        pw = [float(r[3]) for r in self.rows if len(r) >= 9 and r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_median": statistics.median(pw) if pw else None,
                "power_w_max": max(pw) if pw else None}


def gpu_index(local):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return int(vis.split(",")[local])
    return local


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


# ------------------------------------------------------------ workload --
def layer_bytes_bf16(cfg):
    return cfg.params_per_layer() * 2


def layer_bytes_w4(cfg):
    return sum(n * ((k + 63) // 64) * (32 + 4) for n, k in synthetic.layer_shapes(cfg).values())


def cycle_bound(cfg, pk, tau, n_ctx, link_gbs, ring):
    """Roofline-derived lower bound on one cycle (ms) and the tokens/s it allows."""
    lm = cfg.vocab * cfg.hidden * 2
    kv = cfg.n_layers * n_ctx * cfg.kv_dim * 2 * 2
    level_bytes = (cfg.n_resident * layer_bytes_bf16(cfg)
                   + (cfg.n_layers - cfg.n_resident) * layer_bytes_w4(cfg) + lm + kv)
    t_draft = DEPTH * level_bytes / (pk["hbm"] * 1e9) * 1e3
    n_tree = 1 + DEPTH * WIDTH
    flops = 2 * n_tree * (cfg.n_layers * cfg.params_per_layer() + lm // 2)
    t_verify = flops / (pk["bf16_sus"] * 1e12) * 1e3
    n_off = cfg.n_layers - cfg.n_resident
    t_layer = layer_bytes_bf16(cfg) / (link_gbs * 1e9) * 1e3 if link_gbs else 0.0
    t_link = n_off * t_layer
    # a ring of every offloaded layer streams them all under the draft; a ring
    # of r slots stages r layers there and the other n_off - r during the verify
    r = n_off if ring <= 0 else min(ring, n_off)
    link_after_draft = max(0.0, r * t_layer - t_draft) + (n_off - r) * t_layer
    t = t_draft + max(t_verify, link_after_draft)
    return dict(cycle_ms=t, draft_ms=t_draft, verify_ms=t_verify, link_ms=t_link,
                level_bytes=level_bytes, tokens_per_s=tau / t * 1e3 if t else None)


def measure_link(dev):
    """Pinned host -> device copy bandwidth (GB/s), 1 GiB, best of 3."""
    n = 1 << 30
    h = torch.empty(n, dtype=torch.uint8).pin_memory()
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    best = 0.0
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        d.copy_(h, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, n / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del h, d
    return best


def time_launches(fn, iters, stream):
    """Milliseconds per call: `iters` calls captured once in a CUDA graph (on
    a side stream) and replayed three times between CUDA events on the
    replaying stream (host launch cost drops out; each call's own scratch
    allocation stays in)."""
    fn(0)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(iters):
                fn(i)
    # replays run on the current stream: the events go there too
    cur = torch.cuda.current_stream()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(3):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (3 * iters)


def copies_for(nbytes):
    """Operand sets to rotate so that one sweep point streams >= 4x L2."""
    return max(2, math.ceil(ROTATE_BYTES / max(nbytes, 1)))


def kernel_measurements(sub, cfg, weights, model, pk, dev, quick):
    """Dominant-kernel roofline and the kernel sweep (CUDA events on the
    launching stream; every timed point rotates operands over >= 4x L2)."""
    st = torch.cuda.current_stream()
    out = {}
    # --- dominant kernel: int4 GEMV of the substitutes at draft width M=8
    subs = model.w4_mats
    xs = {s[4]: torch.randn(WIDTH, s[4], device=dev).to(torch.bfloat16) for s in subs}
    ys = {s[3]: torch.empty(WIDTH, s[3], device=dev, dtype=torch.bfloat16) for s in subs}

    def run_w4(i):
        q, s_, z, n, k = subs[i % len(subs)]
        sub.w4_gemm(xs[k], q, s_, z, n, k, out=ys[n])
    ms4 = time_launches(run_w4, len(subs) * 2, st)
    b4 = sum(q.numel() + s_.numel() * 2 + z.numel() * 2 + WIDTH * (n + k) * 2
             for q, s_, z, n, k in subs) / len(subs)
    out["w4_gemv_m8"] = dict(ms_per_launch=ms4, bytes_per_launch=b4,
                             gbs=b4 / (ms4 / 1e3) / 1e9,
                             rotated_bytes=sum(q.numel() for q, *_ in subs),
                             what="int4 substitutes (o, gate, up, down of every offloaded "
                                  "layer) in turn, M=8")
    # --- bf16 GEMV of the resident layers at M=8
    mats = []
    for i in range(cfg.n_resident):
        for n in ("wo", "wg", "wu", "wd"):
            mats.append(weights["layers"][i][n])
    x = {m.shape[1]: torch.randn(WIDTH, m.shape[1], device=dev).to(torch.bfloat16) for m in mats}
    y = {m.shape[0]: torch.empty(WIDTH, m.shape[0], device=dev, dtype=torch.bfloat16) for m in mats}
    ms = time_launches(lambda i: sub.bf16_gemm(x[mats[i % len(mats)].shape[1]], mats[i % len(mats)],
                                               out=y[mats[i % len(mats)].shape[0]]),
                       len(mats) * 2, st)
    nbytes = sum(m.numel() * 2 + WIDTH * (m.shape[0] + m.shape[1]) * 2 for m in mats) / len(mats)
    out["gemv_bf16_m8"] = dict(ms_per_launch=ms, bytes_per_launch=nbytes,
                               gbs=nbytes / (ms / 1e3) / 1e9)
    # --- verify GEMM on the tensor cores: all tree nodes through resident matrices
    n_tree = 1 + DEPTH * WIDTH
    xv = {m.shape[1]: torch.randn(n_tree, m.shape[1], device=dev).to(torch.bfloat16) for m in mats}
    yv = {m.shape[0]: torch.empty(n_tree, m.shape[0], device=dev, dtype=torch.bfloat16) for m in mats}
    msv = time_launches(lambda i: sub.bf16_gemm(xv[mats[i % len(mats)].shape[1]], mats[i % len(mats)],
                                                out=yv[mats[i % len(mats)].shape[0]]),
                        len(mats), st)
    fl = sum(2 * n_tree * m.numel() for m in mats) / len(mats)
    out["verify_gemm_bf16"] = dict(ms_per_launch=msv, flops_per_launch=fl,
                                   tflops=fl / (msv / 1e3) / 1e12,
                                   frac_of_peak=fl / (msv / 1e3) / 1e12 / pk["bf16"],
                                   what=f"tcgen05 GEMM, M={n_tree} tree nodes, resident o/gate/up/down")
    del xv, yv
    if quick:
        return out
    # --- 2-, 3- and 4-bit substitutes at M=8 on this workload's o/gate/up/down
    # shapes (random bf16 weights packed on the device), rotated over >= 4x L2
    h, f = cfg.hidden, cfg.ffn
    low = {}
    for bits in (2, 3, 4):
        mats_b = []
        for n, k in ((h, h), (f, h), (f, h), (h, f)):
            wbytes = n * ((k + 63) // 64) * (8 * bits + 4)
            for c in range(copies_for(wbytes)):
                w = (torch.randn(n, k, device=dev) * 0.02).to(torch.bfloat16)
                mats_b.append((*sub.wq_pack(w, bits), n, k))
                del w
        xb = {k: torch.randn(WIDTH, k, device=dev).to(torch.bfloat16) for *_, k in mats_b}
        yb = {n: torch.empty(WIDTH, n, device=dev, dtype=torch.bfloat16) for *_, n, _k in mats_b}

        def run_b(i, bits=bits, mats_b=mats_b, xb=xb, yb=yb):
            q, s_, z, n, k = mats_b[i % len(mats_b)]
            sub.wq_gemm(xb[k], q, s_, z, n, k, bits, out=yb[n])
        msb = time_launches(run_b, len(mats_b), st)
        bb = sum(q.numel() + s_.numel() * 2 + z.numel() * 2 + WIDTH * (n + k) * 2
                 for q, s_, z, n, k in mats_b) / len(mats_b)
        low[f"bits{bits}"] = dict(ms_per_launch=round(msb, 5), bytes_per_launch=int(bb),
                                  gbs=round(bb / (msb / 1e3) / 1e9, 1),
                                  frac_hbm=round(bb / (msb / 1e3) / 1e9 / pk["hbm"], 3),
                                  kernel="gemv_tma_kernel" if all(k % 512 == 0 for *_, k in mats_b)
                                  else "gemv_kernel (K not a multiple of 512)")
        del mats_b, xb, yb
    out["wq_gemv_m8"] = low
    # --- substitute construction: min-max and HQQ (20 iterations) packing of
    # one gate matrix, 4 bits
    wg = (torch.randn(f, h, device=dev) * 0.02).to(torch.bfloat16)
    ms_mm = time_launches(lambda i: sub.wq_pack(wg, 4), 4, st)
    ms_hq = time_launches(lambda i: sub.wq_pack_hqq(wg, 4, 20), 4, st)
    out["pack_gate_4bit"] = dict(shape=[f, h], minmax_ms=round(ms_mm, 4), hqq20_ms=round(ms_hq, 4),
                                 hqq20_gweights_per_s=round(f * h / (ms_hq / 1e3) / 1e9, 2))
    del wg
    # --- int4 sweep on Qwen2.5-32B layer shapes, operands rotated over >= 4x L2
    shapes = {"qkv": (7168, 5120), "o": (5120, 5120), "gate_up": (55296, 5120),
              "down": (5120, 27648)}
    sweep = {}
    for name, (n, k) in shapes.items():
        wbytes = n * ((k + 63) // 64) * 36
        nc = copies_for(wbytes)
        packs = [synthetic.random_w4(n, k, seed, device=dev) for seed in range(nc)]
        for mrows in (1, 8, 32, 48, 128, 384):
            xx = torch.randn(mrows, k, device=dev).to(torch.bfloat16)
            yy = torch.empty(mrows, n, device=dev, dtype=torch.bfloat16)
            msx = time_launches(lambda i: sub.w4_gemm(xx, *packs[i % nc], n, k, out=yy),
                                max(20, nc), st)
            byt = wbytes + 2 * mrows * (n + k)
            sweep.setdefault(f"M{mrows}", {})[name] = dict(
                ms=round(msx, 5), gbs=round(byt / (msx / 1e3) / 1e9, 1),
                frac_hbm=round(byt / (msx / 1e3) / 1e9 / pk["hbm"], 3),
                tflops=round(2 * mrows * n * k / (msx / 1e3) / 1e12, 2), copies=nc)
        del packs
    out["w4_sweep_qwen32b"] = sweep
    # --- tree attention, Qwen2.5-32B heads (40 q / 8 kv, d 128); KV rotated over >= 4x L2
    attn = {}
    hq, hkv, d = 40, 8, 128
    tok, par, dep = synthetic.random_tree(DEPTH, WIDTH, 3, 1000)
    anc = synthetic.ancestors(par, dep, DEPTH).to(dev)
    depd = dep.to(dev)
    n_tree = len(par)
    for lkv in (1024, 4096, 16384):
        cap = lkv + n_tree + 64
        kv_bytes = (lkv + n_tree) * hkv * d * 2 * 2
        nc = copies_for(kv_bytes)
        caches = []
        for _ in range(nc):
            kv, keep = sub.make_kv(1, hkv, d, cap, page_size=64)
            keep[0].normal_()
            keep[1].normal_()
            caches.append((kv, keep))
        for nq, tag in ((n_tree, "verify385"), (WIDTH, "draft8")):
            q = torch.randn(nq, hq, d, device=dev).to(torch.bfloat16)
            a_ = anc[-nq:].contiguous()
            dd = depd[-nq:].contiguous()
            msa = time_launches(lambda i: sub.tree_attn(q, caches[i % nc][0], 0, lkv, lkv, n_tree,
                                                        anc=a_, depth=dd), max(20, nc), st)
            byt = kv_bytes + 2 * nq * hq * d * 2
            fl = 4 * nq * hq * (lkv + DEPTH) * d
            attn[f"{tag}_kv{lkv}"] = dict(ms=round(msa, 5), gbs=round(byt / (msa / 1e3) / 1e9, 1),
                                          frac_hbm=round(byt / (msa / 1e3) / 1e9 / pk["hbm"], 3),
                                          tflops=round(fl / (msa / 1e3) / 1e12, 2), copies=nc)
        del caches
    out["tree_attn_qwen32b_heads"] = attn
    return out


# ------------------------------------------------------------ CPU oracle --
def oracle_weights(weights, layers):
    """Oracle-format (float32 NumPy, exact bf16 values) globals and layers."""
    glob = {k: weights[k].float().cpu().numpy() for k in ("embed", "lm_head", "final_norm")}
    lay = [{k: v.float().cpu().numpy() for k, v in weights["layers"][i].items()} for i in layers]
    return glob, lay


def oracle_token(cfg, glob, layers, n_ctx, seed=0):
    """Seconds for the oracle's plain target decoding of one token at context
    n_ctx over the given layers (a random bf16 KV prefix stands in for the
    prompt's cache), lm_head included."""
    import numpy as np
    from oracle.bf16 import round_bf16
    from oracle.model import forward_rows
    rng = np.random.default_rng(seed)
    ks = [round_bf16(rng.standard_normal((n_ctx, cfg.n_heads_kv, cfg.head_dim)).astype(np.float32))
          for _ in layers]
    t0 = time.perf_counter()
    forward_rows(cfg, glob, layers, [7], [n_ctx], ks, ks, np.ones((1, n_ctx), bool),
                 np.ones((1, 1), bool))
    return time.perf_counter() - t0


_ONE_THREAD = r"""
import os, sys, time, json
sys.path.insert(0, {root!r})
import numpy as np
import torch
import synthetic
from oracle.bf16 import round_bf16
from oracle.model import forward_rows
cfg = synthetic.CONFIGS[{cfg!r}]
g = synthetic.make_globals(cfg)
glob = {{k: v.float().numpy() for k, v in g.items()}}
lay = [{{k: v.float().numpy() for k, v in synthetic.make_layer(cfg, i).items()}}
       for i in range({nl})]
rng = np.random.default_rng(0)
ks = [round_bf16(rng.standard_normal(({ctx}, cfg.n_heads_kv, cfg.head_dim)).astype(np.float32))
      for _ in lay]
vis = np.ones((1, {ctx}), bool)
t0 = time.perf_counter()
forward_rows(cfg, glob, lay, [7], [{ctx}], ks, ks, vis, np.ones((1, 1), bool))
t1 = time.perf_counter()
forward_rows(cfg, glob, [], [7], [{ctx}], [], [], np.ones((1, 0), bool), np.ones((1, 1), bool))
t2 = time.perf_counter()
print(json.dumps(dict(layers_s=t1 - t0, head_s=t2 - t1)))
"""


def oracle_one_thread(cfg, n_layers_sample=2):
    """The oracle on one host thread (BLAS pinned to one thread in a child
    process): seconds for n_layers_sample layers and for the head alone."""
    env = {**os.environ, "OPENBLAS_NUM_THREADS": "1", "OMP_NUM_THREADS": "1",
           "MKL_NUM_THREADS": "1", "CUDA_VISIBLE_DEVICES": ""}
    code = _ONE_THREAD.format(root=ROOT, cfg=cfg.name, nl=n_layers_sample, ctx=cfg.prompt_len)
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=600)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:   # reported, not fatal: the baseline is context only
        return {"error": f"{type(e).__name__}: {e}"}


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, as it stands, on the host cores.
    One step = the oracle's plain target decoding of one token through every
    layer and the head at the workload's prompt length."""
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    cfg = synthetic.CONFIGS[wl["cfg"]]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t0 = time.perf_counter()
    weights = synthetic.make_model(cfg, device=dev)
    glob, layers = oracle_weights(weights, range(cfg.n_layers))
    del weights
    setup = time.perf_counter() - t0
    times = []
    for i in range(args.warmup + args.steps):
        t = oracle_token(cfg, glob, layers, cfg.prompt_len, seed=i)
        if i >= args.warmup:
            times.append(t)
    t = statistics.mean(times)
    value = 1.0 / t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": wl["text"], "prompt": cfg.prompt_len, "depth": DEPTH,
                   "width": WIDTH},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(),
                         "cpu": cpu_model(), "kind": "oracle",
                         "sample": f"per step: the oracle's plain target decoding of one token "
                                   f"through all {cfg.n_layers} layers and the lm_head at context "
                                   f"{cfg.prompt_len} (random bf16 KV prefix); float64 GEMMs on "
                                   f"NumPy's threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "step_ms": {"median": statistics.median(times) * 1e3,
                    "std": (statistics.stdev(times) * 1e3 if len(times) > 1 else 0.0)},
        "setup_s": round(setup, 1),
    }
    print(json.dumps(line))


# ------------------------------------------------------------------ main --
def build_model(sub, cfg, wl, dev, max_seq):
    weights = synthetic.make_model(cfg, device=dev)
    model = sub.Model(cfg, weights, max_seq=max_seq, max_depth=max(DEPTH_SWEEP), max_width=WIDTH,
                      max_prompt=cfg.prompt_len, staging_layers=wl["staging"],
                      embed_on_host=wl["embed_on_host"])
    # the substitutes' device tensors, for the kernel measurement
    model.w4_mats = []
    for i in range(cfg.n_resident, cfg.n_layers):
        for name in ("wo", "wg", "wu", "wd"):
            q, s_, z = model.w4[(i, name)]
            n, k = weights["layers"][i][name].shape
            model.w4_mats.append((q, s_, z, n, k))
    # offloaded originals now live pinned on the host; free their device copies
    for i in range(cfg.n_resident, cfg.n_layers):
        for name in synthetic.LAYER_TENSORS:
            weights["layers"][i][name] = weights["layers"][i][name].to("cpu")
    if wl["embed_on_host"]:
        weights["embed"] = weights["embed"].to("cpu")
    torch.cuda.empty_cache()
    return weights, model


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen7b", choices=sorted(WORKLOADS))
    ap.add_argument("--new", type=int, default=None, help="tokens generated by the e2e leg")
    ap.add_argument("--quick", action="store_true")
    ap.add_argument("--stop-logp", type=float, default=None,
                    help="adaptive depth for the timed cycles and the e2e run (default: off)")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    import substitute_speculative_decoding_gb300 as sub

    assert args.warmup >= 0 and args.steps >= 1
    wl = WORKLOADS[args.workload]
    cfg = synthetic.CONFIGS[wl["cfg"]]
    mode = 1 if cfg.mode == "gumbel" else 0
    e2e_new = args.new or wl["e2e_new"]
    sweep_new = wl.get("sweep_new", ADAPTIVE_NEW)   # tokens per sweep run
    dev = torch.device("cuda", torch.cuda.current_device())
    pk = peaks()
    t_setup = time.perf_counter()
    max_seq = cfg.prompt_len + max(e2e_new, (args.warmup + args.steps + 2) * (DEPTH + 1),
                                   sweep_new + max(DEPTH_SWEEP) + 1) + 64
    weights, model = build_model(sub, cfg, wl, dev, max_seq)
    t_setup = time.perf_counter() - t_setup
    timeouts0 = sub.pipeline_timeouts()

    prompt = synthetic.make_prompt(cfg)
    dcfg = sub.Model.decode_cfg(DEPTH, WIDTH, DRAFT_T, mode=mode, target_temp=cfg.target_temp,
                                seed=cfg.seed, stop_logp=args.stop_logp)
    kernels_per_cycle, h2d_per_cycle = model.cycle_info(dcfg)
    stream = torch.cuda.current_stream()
    model.prefill(prompt, dcfg, stream)
    model.decode_cycles(dcfg, args.warmup, stream)
    _, e0, c0 = model.decode_read()

    clocks = Clocks(gpu_index(local))
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs[0].record(stream)
    torch.cuda.nvtx.range_push("timed_cycles")   # lets a profiler select exactly the steps
    for i in range(args.steps):
        model.decode_cycles(dcfg, 1, stream)
        evs[i + 1].record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    barrier(world)
    ms = evs[0].elapsed_time(evs[-1])
    cyc = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    clk = clocks.stop()
    _, e1, c1 = model.decode_read()
    tokens = e1 - e0
    tau = tokens / args.steps
    tokens_all, ms_max, value = aggregate(world, tokens, ms)

    # clocks and throttle reasons over the e2e run and the sweeps as well
    clocks_sweeps = Clocks(gpu_index(local))
    if not args.quick:
        clocks_sweeps.start()
    # e2e: the public call with host buffers, prefill included
    e2e = None
    if not args.quick:
        t0 = time.perf_counter()
        out, st = model.generate(prompt, e2e_new, DEPTH, WIDTH, DRAFT_T, mode=mode,
                                 target_temp=cfg.target_temp, seed=cfg.seed,
                                 stop_logp=args.stop_logp)
        t_e2e = time.perf_counter() - t0
        cycles = max(int(st.cycles), 1)
        h2d_total = prompt.numel() * 4 + h2d_per_cycle * (st.cycles + 1)
        d2h_total = e2e_new * 4 + 32 * (st.cycles + 1)
        e2e = {"value": e2e_new / t_e2e, "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d_total / cycles),
               "d2h_bytes_per_step": int(d2h_total / cycles),
               "tokens": e2e_new, "seconds": t_e2e, "prefill_ms": st.t_prefill_ms,
               "decode_ms": st.t_decode_ms, "tau": st.tau, "cycles": st.cycles,
               "per_cycle_ms": {"draft": st.t_draft_ms / cycles,
                                "verify": st.t_verify_ms / cycles,
                                "copy_unhidden": st.t_copy_unhidden_ms / cycles,
                                "copy": st.t_copy_ms / cycles},
               "h2d_gbs": (h2d_per_cycle * cycles / (st.t_copy_ms / 1e3) / 1e9
                           if st.t_copy_ms > 0 else None),
               "draft_over_target": (st.t_draft_ms / st.t_verify_ms
                                     if st.t_verify_ms > 0 else None),
               "near_tie_events": st.near_tie_events,
               "note": "per step = per decode cycle: the run's host-to-device bytes (prompt, the "
                       "offloaded originals streamed for the prefill and every verify) and "
                       "device-to-host bytes (state reads, tokens) over its cycles; "
                       "draft_over_target is the denominator term D*t_draft/t_target"}

    # adaptive depth: the same decode with drafting stopped per cycle once the
    # best cumulative sharpened log-probability of a new level falls below a
    # threshold (decode tokens/s over the cycles, prefill excluded)
    adaptive = depth_sweep = None
    if not args.quick:
        depth_sweep = []
        for dd in DEPTH_SWEEP:
            # capture the cycle graph first: the decode time is then steady-state
            model.cycle_info(sub.Model.decode_cfg(dd, WIDTH, DRAFT_T, mode=mode,
                                                  target_temp=cfg.target_temp, seed=cfg.seed))
            _, sd = model.generate(prompt, sweep_new, dd, WIDTH, DRAFT_T, mode=mode,
                                   target_temp=cfg.target_temp, seed=cfg.seed)
            cyc_d = max(int(sd.cycles), 1)
            depth_sweep.append({"depth": dd,
                                "decode_tokens_per_s": (sweep_new - 1) / (sd.t_decode_ms / 1e3),
                                "tau": sd.tau, "cycle_ms": sd.t_decode_ms / cyc_d,
                                "cycles": sd.cycles, **phase_ms(sd, h2d_per_cycle)})
        adaptive = []
        for stop in ADAPTIVE_STOPS:
            model.cycle_info(sub.Model.decode_cfg(DEPTH, WIDTH, DRAFT_T, mode=mode,
                                                  target_temp=cfg.target_temp, seed=cfg.seed,
                                                  stop_logp=stop))
            _, sa = model.generate(prompt, sweep_new, DEPTH, WIDTH, DRAFT_T, mode=mode,
                                   target_temp=cfg.target_temp, seed=cfg.seed, stop_logp=stop)
            cyc_a = max(int(sa.cycles), 1)
            adaptive.append({"stop_logp": stop,
                             "decode_tokens_per_s": (sweep_new - 1) / (sa.t_decode_ms / 1e3),
                             "tau": sa.tau, "mean_depth": sa.drafted_levels / cyc_a,
                             "cycle_ms": sa.t_decode_ms / cyc_a, "cycles": sa.cycles,
                             **phase_ms(sa, h2d_per_cycle)})

    # verify reuse of the draft's leading (resident) layers, fixed depth and
    # adaptive depth at stop_logp -6
    reuse = None
    if not args.quick:
        reuse = []
        for stop in (None, -6.0):
            model.cycle_info(sub.Model.decode_cfg(DEPTH, WIDTH, DRAFT_T, mode=mode,
                                                  target_temp=cfg.target_temp, seed=cfg.seed,
                                                  stop_logp=stop, verify_reuse=True))
            _, sr = model.generate(prompt, sweep_new, DEPTH, WIDTH, DRAFT_T, mode=mode,
                                   target_temp=cfg.target_temp, seed=cfg.seed, stop_logp=stop,
                                   verify_reuse=True)
            cr = max(int(sr.cycles), 1)
            reuse.append({"stop_logp": stop,
                          "decode_tokens_per_s": (sweep_new - 1) / (sr.t_decode_ms / 1e3),
                          "tau": sr.tau, "mean_depth": sr.drafted_levels / cr,
                          "cycle_ms": sr.t_decode_ms / cr, **phase_ms(sr, h2d_per_cycle)})

    clk_sweeps = clocks_sweeps.stop() if not args.quick else None
    # host link and kernel measurements come after this model's decode runs
    link = measure_link(dev)
    bound = cycle_bound(cfg, pk, tau, cfg.prompt_len + tokens, link, wl["staging"])
    kern = kernel_measurements(sub, cfg, weights, model, pk, dev, args.quick)

    g = kern["w4_gemv_m8"]
    traffic = profile_traffic("gemv_w4")
    roof = {"kernel": "gemv_tma_kernel (int4 substitutes, M=8: the draft's substitute layers)",
            "bound": "hbm", "achieved": round(g["gbs"], 1), "peak": pk["hbm"],
            "unit": "GB/s", "frac": round(g["gbs"] / pk["hbm"], 4),
            "traffic": traffic, "peak_source": pk["src"] + " (burst copy)",
            "bytes_per_launch": int(g["bytes_per_launch"])}

    model_bytes = model.device_bytes()
    device_total = int(torch.cuda.memory_allocated() + model_bytes)
    # lower and mixed-precision substitutes: the same workload rebuilt with
    # 3-bit, 2-bit and half-and-half (first half of the substituted layers
    # 4-bit, the rest 2-bit) substitutes; decode tokens/s, tau and the draft's
    # share, at the fixed depth and with adaptive depth at stop_logp -6
    lowbit = None
    if not args.quick and wl.get("lowbit", True):
        model.close()
        model = None
        torch.cuda.empty_cache()
        n_sub = cfg.n_layers - cfg.n_resident
        mixed = [4] * cfg.n_resident + [4 if j < n_sub // 2 else 2 for j in range(n_sub)]
        lowbit = []
        for tag, bits, hq in (("4-bit HQQ zeros", 4, 20), ("3-bit", 3, 0), ("2-bit", 2, 0),
                              ("4/2-bit mixed", mixed, 0)):
            mb = sub.Model(cfg, weights, max_seq=max_seq, max_depth=max(DEPTH_SWEEP),
                           max_width=WIDTH, max_prompt=cfg.prompt_len,
                           staging_layers=wl["staging"], embed_on_host=wl["embed_on_host"],
                           bits=bits, hqq_iters=hq)
            entry = {"substitutes": tag}
            for key, stop in (("fixed", None), ("adaptive_m6", -6.0)):
                mb.cycle_info(sub.Model.decode_cfg(DEPTH, WIDTH, DRAFT_T, mode=mode,
                                                   target_temp=cfg.target_temp, seed=cfg.seed,
                                                   stop_logp=stop))
                _, sb = mb.generate(prompt, sweep_new, DEPTH, WIDTH, DRAFT_T, mode=mode,
                                    target_temp=cfg.target_temp, seed=cfg.seed, stop_logp=stop)
                cb = max(int(sb.cycles), 1)
                entry[key] = {"decode_tokens_per_s": (sweep_new - 1) / (sb.t_decode_ms / 1e3),
                              "tau": sb.tau, "mean_depth": sb.drafted_levels / cb,
                              "draft_ms_per_level": sb.t_draft_ms / max(sb.drafted_levels, 1),
                              **phase_ms(sb, h2d_per_cycle)}
            mb.close()
            lowbit.append(entry)
            torch.cuda.empty_cache()

    # the oracle baseline last: its host memory and threads touch no GPU measurement
    cpu = None
    if rank == 0 and world == 1 and not args.quick:
        # one full token through every layer and the head on all host cores,
        # then a one-thread sample (2 layers + head, scaled) in a child process
        glob, layers = oracle_weights(weights, range(cfg.n_layers)) \
            if args.workload != "qwen32b" else (None, None)
        one = oracle_one_thread(cfg)
        if glob is not None:
            t_tok = oracle_token(cfg, glob, layers, cfg.prompt_len)
            del glob, layers
            cpu = {"value": 1.0 / t_tok, "unit": "tokens/s", "cores": cpu_cores(),
                   "cpu": cpu_model(), "kind": "oracle",
                   "sample": f"the oracle's plain target decoding of one token through all "
                             f"{cfg.n_layers} layers and the lm_head at context {cfg.prompt_len} "
                             f"(random bf16 KV prefix), float64 GEMMs on NumPy's threads"}
        else:
            cpu = {"value": None, "unit": "tokens/s", "cores": cpu_cores(), "cpu": cpu_model(),
                   "kind": "oracle", "sample": "all-core token skipped (the 32B oracle weights "
                                               "do not fit beside the pinned originals)"}
        if "layers_s" in one:
            t1 = one["layers_s"] * cfg.n_layers / 2 + one["head_s"]
            cpu["one_thread"] = {"value": 1.0 / t1, "unit": "tokens/s", "cores": 1,
                                 "sample": "2 layers and the lm_head timed on one thread, "
                                           f"layers scaled to {cfg.n_layers}"}
        else:
            cpu["one_thread"] = one

    timeouts = sub.pipeline_timeouts() - timeouts0
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl["text"], "prompt": cfg.prompt_len, "depth": DEPTH,
                   "width": WIDTH, "parallelism": f"replicas x{world}",
                   **({"stop_logp": args.stop_logp,
                       "gpu_launches": "upper bound: every conditional draft level counted"}
                      if args.stop_logp is not None else {}),
                   "l2": "inputs larger than L2 (every draft level reads all weights: "
                         f"{bound['level_bytes'] / 1e9:.2f} GB)"},
        "tau": tau, "tokens_timed": tokens_all,
        "cycle_ms": {"median": statistics.median(cyc),
                     "std": statistics.stdev(cyc) if len(cyc) > 1 else 0.0,
                     "min": min(cyc), "max": max(cyc)},
        "bound": {k: (round(v, 3) if isinstance(v, float) else v) for k, v in bound.items()},
        "frac_of_bound": value / world / bound["tokens_per_s"] if bound["tokens_per_s"] else None,
        "host_link_gbs": round(link, 1),
        "roofline": roof, "kernels": kern, "cpu_baseline": cpu, "e2e": e2e,
        "adaptive": adaptive, "depth_sweep": depth_sweep, "lowbit": lowbit, "verify_reuse": reuse,
        "gpu_launches": kernels_per_cycle * args.steps, "kernels_per_cycle": kernels_per_cycle,
        "clocks": clk, "clocks_e2e_and_sweeps": clk_sweeps, "setup_s": round(t_setup, 1),
        "model_device_bytes": model_bytes,
        "device_bytes_total": device_total,
        "pipeline_timeouts": timeouts, "valid": timeouts == 0,
    }
    if rank == 0:
        print(json.dumps(line))
    if model is not None:
        model.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if timeouts:
        raise SystemExit(f"{timeouts} bounded pipeline wait(s) ran out: the numbers are invalid")


def phase_ms(st, h2d_per_cycle=None):
    """Per-cycle device time of a generate call's phases (sub_stats), and the
    host link rate its streamed copies got."""
    c = max(int(st.cycles), 1)
    out = {"per_cycle_ms": {"draft": round(st.t_draft_ms / c, 3),
                            "verify": round(st.t_verify_ms / c, 3),
                            "copy_unhidden": round(st.t_copy_unhidden_ms / c, 3),
                            "copy": round(st.t_copy_ms / c, 3)}}
    if h2d_per_cycle and st.t_copy_ms > 0:
        out["h2d_gbs"] = round(h2d_per_cycle * c / (st.t_copy_ms / 1e3) / 1e9, 1)
    return out


def profile_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, valid only while
    the kernel's source is unchanged; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path)).get(kernel)
    if not d:
        return None
    src = os.path.join(ROOT, "substitute_speculative_decoding_gb300", "csrc", d["source"])
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return d["dram_bytes_per_launch"] if sha == d["source_sha"] else None


if __name__ == "__main__":
    main()
