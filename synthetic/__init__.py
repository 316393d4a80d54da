"""Seeded synthetic inputs for the SubSpec decode step.

This module only *draws* inputs: model shapes, random bf16 weights, prompts,
random trees and random packed int4 tensors.  It holds none of the method's
arithmetic (no quantiser, no forward pass, no tree selection), so both the
CUDA path and the CPU oracle can take their inputs from it without sharing any
code of the method.

The pages measure on MT-Bench and four other prompt suites ("Speculate Deep and
Accurate" summary card, Experimental setup); none of them is available here, so
prompts are uniform random token ids and weights are N(0, 0.02) draws rounded
to bf16 (random initialisation of the decoder shapes the pages evaluate:
Qwen2.5-7B, Llama-3.1-8B, Qwen2.5-32B).
"""
from __future__ import annotations

import dataclasses
import hashlib

import torch


@dataclasses.dataclass(frozen=True)
class DecoderConfig:
    """Shape of a dense Llama/Qwen-style decoder plus the decode settings."""
    name: str
    n_layers: int
    hidden: int
    n_heads_q: int
    n_heads_kv: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float
    rms_eps: float
    n_resident: int          # layers [0, n_resident) stay on the GPU in bf16
    prompt_len: int
    n_new: int
    depth: int               # draft tree depth (levels below the root)
    width: int               # nodes kept per level
    draft_temp: float = 0.2
    mode: str = "greedy"     # "greedy" or "gumbel"
    target_temp: float = 1.0
    seed: int = 7            # sampling seed (gumbel mode)

    @property
    def q_dim(self) -> int:
        return self.n_heads_q * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_heads_kv * self.head_dim

    @property
    def n_tree(self) -> int:
        return 1 + self.depth * self.width

    def params_per_layer(self) -> int:
        h = self.hidden
        return h * (self.q_dim + 2 * self.kv_dim) + self.q_dim * h + 3 * h * self.ffn

    def replace(self, **kw) -> "DecoderConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    # Tiny decoder: the oracle runs the whole decode in seconds.
    "tiny": DecoderConfig("tiny", n_layers=2, hidden=256, n_heads_q=4, n_heads_kv=2,
                          head_dim=64, ffn=688, vocab=1024, rope_theta=1e4, rms_eps=1e-6,
                          n_resident=1, prompt_len=32, n_new=64, depth=8, width=2),
    # Qwen2.5-7B shapes, 11 resident layers, 17 substitutes.
    "qwen7b": DecoderConfig("qwen7b", n_layers=28, hidden=3584, n_heads_q=28, n_heads_kv=4,
                            head_dim=128, ffn=18944, vocab=152064, rope_theta=1e6, rms_eps=1e-6,
                            n_resident=11, prompt_len=512, n_new=256, depth=48, width=8),
    # Llama-3.1-8B shapes, 8 resident layers, 24 substitutes.
    "llama8b": DecoderConfig("llama8b", n_layers=32, hidden=4096, n_heads_q=32, n_heads_kv=8,
                             head_dim=128, ffn=14336, vocab=128256, rope_theta=5e5, rms_eps=1e-5,
                             n_resident=8, prompt_len=1024, n_new=512, depth=48, width=8),
    # Qwen2.5-32B shapes, sampled decoding at T=0.6 with a fixed seed.
    "qwen32b": DecoderConfig("qwen32b", n_layers=64, hidden=5120, n_heads_q=40, n_heads_kv=8,
                             head_dim=128, ffn=27648, vocab=152064, rope_theta=1e6, rms_eps=1e-6,
                             n_resident=1, prompt_len=256, n_new=4096, depth=48, width=8,
                             mode="gumbel", target_temp=0.6, seed=7),
}

WEIGHT_SEED = 1234
PROMPT_SEED = 42
WEIGHT_STD = 0.02

LAYER_TENSORS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def _seed_of(*parts) -> int:
    """Stable 63-bit seed from a tuple of labels."""
    h = hashlib.sha256(repr(parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _randn_bf16(shape, seed, std, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (t * std).to(torch.bfloat16)


def layer_shapes(cfg: DecoderConfig) -> dict:
    h, f = cfg.hidden, cfg.ffn
    return {"wq": (cfg.q_dim, h), "wk": (cfg.kv_dim, h), "wv": (cfg.kv_dim, h),
            "wo": (h, cfg.q_dim), "wg": (f, h), "wu": (f, h), "wd": (h, f)}


def make_layer(cfg: DecoderConfig, layer: int, seed: int = WEIGHT_SEED, device="cpu",
               norm_gain_std: float = 0.0) -> dict:
    """bf16 weights of one decoder layer (out_features x in_features, row-major)."""
    out = {}
    for name, shape in layer_shapes(cfg).items():
        out[name] = _randn_bf16(shape, _seed_of(cfg.name, seed, layer, name), WEIGHT_STD, device)
    for name in ("attn_norm", "ffn_norm"):
        out[name] = _gain(cfg.hidden, _seed_of(cfg.name, seed, layer, name), norm_gain_std, device)
    return out


def _gain(n, seed, std, device):
    if std == 0.0:
        return torch.ones(n, dtype=torch.bfloat16, device=device)
    return (1.0 + _randn_bf16((n,), seed, std, device).float()).to(torch.bfloat16)


def make_globals(cfg: DecoderConfig, seed: int = WEIGHT_SEED, device="cpu",
                 norm_gain_std: float = 0.0) -> dict:
    """Embedding, untied lm_head and final norm gain."""
    return {
        "embed": _randn_bf16((cfg.vocab, cfg.hidden), _seed_of(cfg.name, seed, "embed"),
                             WEIGHT_STD, device),
        "lm_head": _randn_bf16((cfg.vocab, cfg.hidden), _seed_of(cfg.name, seed, "lm_head"),
                               WEIGHT_STD, device),
        "final_norm": _gain(cfg.hidden, _seed_of(cfg.name, seed, "final_norm"), norm_gain_std,
                            device),
    }


def make_model(cfg: DecoderConfig, seed: int = WEIGHT_SEED, device="cpu",
               norm_gain_std: float = 0.0) -> dict:
    m = make_globals(cfg, seed, device, norm_gain_std)
    m["layers"] = [make_layer(cfg, i, seed, device, norm_gain_std) for i in range(cfg.n_layers)]
    return m


def make_prompt(cfg: DecoderConfig, seed: int = PROMPT_SEED, n: int | None = None) -> torch.Tensor:
    g = torch.Generator().manual_seed(_seed_of(cfg.name, "prompt", seed))
    n = cfg.prompt_len if n is None else n
    return torch.randint(0, cfg.vocab, (n,), generator=g, dtype=torch.int64).to(torch.int32)


def randn_bf16(shape, seed: int, std: float = 1.0, device="cpu") -> torch.Tensor:
    return _randn_bf16(shape, _seed_of("randn", seed, tuple(shape)), std, device)


def randn_f32(shape, seed: int, std: float = 1.0, device="cpu") -> torch.Tensor:
    g = torch.Generator(device=device).manual_seed(_seed_of("randnf", seed, tuple(shape)))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def random_tree(depth: int, width: int, seed: int, vocab: int):
    """A static tree of 1 + depth*width slots: slot 0 is the root, level l
    (1..depth) holds slots 1+(l-1)*width .. l*width, and each level-l node picks
    a uniformly random parent on level l-1.  Returns (tokens, parent, depth) as
    int32 tensors.  Siblings get distinct tokens."""
    g = torch.Generator().manual_seed(_seed_of("tree", depth, width, seed))
    n = 1 + depth * width
    parent = torch.full((n,), -1, dtype=torch.int32)
    dep = torch.zeros(n, dtype=torch.int32)
    tok = torch.zeros(n, dtype=torch.int32)
    tok[0] = int(torch.randint(0, vocab, (1,), generator=g))
    for lvl in range(1, depth + 1):
        lo = 1 + (lvl - 1) * width
        prev_lo, prev_n = (0, 1) if lvl == 1 else (1 + (lvl - 2) * width, width)
        pars = torch.randint(0, prev_n, (width,), generator=g) + prev_lo
        toks = torch.randperm(vocab, generator=g)[:width]
        for j in range(width):
            parent[lo + j] = int(pars[j])
            dep[lo + j] = lvl
            tok[lo + j] = int(toks[j])
    return tok, parent, dep


def ancestors(parent: torch.Tensor, dep: torch.Tensor, max_depth: int) -> torch.Tensor:
    """[n, max_depth+1] int32 slot lists root->self, padded with -1.  A pure
    re-indexing of the parent links (no arithmetic of the method)."""
    n = parent.numel()
    anc = torch.full((n, max_depth + 1), -1, dtype=torch.int32)
    for s in range(n):
        chain = []
        u = s
        while u >= 0:
            chain.append(u)
            u = int(parent[u])
        chain.reverse()
        anc[s, :len(chain)] = torch.tensor(chain, dtype=torch.int32)
    return anc


def random_w4(n: int, k: int, seed: int, device="cpu"):
    """Uniform random packed nibbles with scales/zeros derived from min-max of
    N(0, 0.02) groups of 64: the kernel-sweep input.  Returns (qbytes uint8
    [n, ceil(k/64)*32], scale bf16 [n, G], zero bf16 [n, G])."""
    gcount = (k + 63) // 64
    g = torch.Generator(device=device).manual_seed(_seed_of("w4", n, k, seed))
    q = torch.randint(0, 256, (n, gcount * 32), generator=g, device=device, dtype=torch.int32)
    q = q.to(torch.uint8)
    # scale ~ range of 64 normals / 15, zero ~ mid code: typical of N(0,0.02) groups
    s = (torch.rand((n, gcount), generator=g, device=device) * 0.002 + 0.0055).to(torch.bfloat16)
    z = (torch.rand((n, gcount), generator=g, device=device) * 2.0 + 6.5).to(torch.bfloat16)
    return q, s, z
