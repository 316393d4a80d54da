"""Python binding of the SubSpec CUDA library (libsubspec.so, sm_103a).

Argument marshalling only: every step of the decode path runs in the
library's kernels.  PyTorch provides device memory, pinned host memory and
streams.  There is no CPU fallback: importing this package fails loudly when
the library has not been built (run ``substitute_speculative_decoding_gb300/build.py``
or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsubspec.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                      "(python substitute_speculative_decoding_gb300/build.py)")
_lib = C.CDLL(LIB_PATH)

SUB_OK, SUB_EINVAL, SUB_ENOMEM, SUB_ECUDA, SUB_EUNSUPPORTED, SUB_ETIMEOUT = range(6)
_NAMES = {1: "EINVAL", 2: "ENOMEM", 3: "ECUDA", 4: "EUNSUPPORTED", 5: "ETIMEOUT"}


class SubError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"SUB_{_NAMES.get(code, code)}: {msg}")
        self.code = code


_vp = C.c_void_p
_i32, _i64, _u64, _f32 = C.c_int32, C.c_int64, C.c_uint64, C.c_float


class KVCache(C.Structure):
    _fields_ = [("k", _vp), ("v", _vp), ("page_table", _vp), ("n_layers", _i32),
                ("n_heads_kv", _i32), ("head_dim", _i32), ("page_size", _i32),
                ("n_pages", _i32), ("capacity", _i64)]


class Tree(C.Structure):
    _fields_ = [("token", _vp), ("parent", _vp), ("depth", _vp), ("score", _vp), ("anc", _vp),
                ("width", _i32), ("max_depth", _i32)]


class W4(C.Structure):
    _fields_ = [("q", _vp), ("scale", _vp), ("zero", _vp), ("bits", _i32)]


class LayerDesc(C.Structure):
    _fields_ = [(n, _vp) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd",
                                   "attn_norm", "ffn_norm")] + \
               [(n, W4) for n in ("q4", "k4", "v4", "o4", "g4", "u4", "d4")]


class ModelDesc(C.Structure):
    _fields_ = [(n, _i32) for n in ("n_layers", "hidden", "n_heads_q", "n_heads_kv", "head_dim",
                                    "ffn", "vocab", "n_resident")] + \
               [("rope_theta", _f32), ("rms_eps", _f32), ("embed", _vp), ("lm_head", _vp),
                ("final_norm", _vp), ("layers", C.POINTER(LayerDesc))] + \
               [(n, _i32) for n in ("max_seq", "max_depth", "max_width", "staging_layers",
                                    "max_prompt")]


class DecodeCfg(C.Structure):
    _fields_ = [("depth", _i32), ("width", _i32), ("draft_temp", _f32), ("mode", _i32),
                ("target_temp", _f32), ("seed", _u64), ("use_graph", _i32),
                ("stop_logp", _f32), ("verify_reuse", _i32)]


class Stats(C.Structure):
    _fields_ = [("cycles", _i64), ("emitted", _i64), ("tau", C.c_double),
                ("t_prefill_ms", C.c_double), ("t_decode_ms", C.c_double),
                ("accept_hist", _i64 * 65), ("t_draft_ms", C.c_double),
                ("t_verify_ms", C.c_double), ("t_copy_unhidden_ms", C.c_double),
                ("near_tie_events", _i64), ("drafted_levels", _i64), ("t_copy_ms", C.c_double)]


def _decl(name, args):
    f = getattr(_lib, name)
    f.argtypes = args
    f.restype = _i32
    return f


_lib.sub_last_error.restype = C.c_char_p
_lib.sub_last_error.argtypes = []
_lib.sub_version.restype = C.c_char_p
_lib.sub_version.argtypes = []
_pipeline_timeouts = _decl("sub_pipeline_timeouts", [_vp])
_bounded_wait_check = _decl("sub_bounded_wait_check", [C.c_uint32])

_w4_pack = _decl("sub_w4_pack", [_vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp])
_w4_dequant = _decl("sub_w4_dequant", [_vp, _vp, _vp, _i64, _i64, _i32, _vp, _vp])
_w4_gemm = _decl("sub_w4_gemm", [_vp, _i64, _vp, _vp, _vp, _i64, _i64, _i32, _vp, _vp])
_bf16_gemm = _decl("sub_bf16_gemm", [_vp, _i64, _vp, _i64, _i64, _vp, _vp])
_wq_pack = _decl("sub_wq_pack", [_vp, _i64, _i64, _i32, _i32, _vp, _vp, _vp, _vp])
_wq_dequant = _decl("sub_wq_dequant", [_vp, _vp, _vp, _i64, _i64, _i32, _i32, _vp, _vp])
_wq_pack_hqq = _decl("sub_wq_pack_hqq", [_vp, _i64, _i64, _i32, _i32, _i32, _vp, _vp, _vp, _vp])
_wq_gemm = _decl("sub_wq_gemm", [_vp, _i64, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _vp, _vp])
_tree_attn = _decl("sub_tree_attn", [_vp, _i32, _i32, C.POINTER(KVCache), _i32, _i64, _i64, _i32,
                                     _vp, _i32, _vp, _f32, _vp, _vp])
_draft_expand = _decl("sub_draft_expand", [_vp, _i64, _f32, C.POINTER(Tree), _i32, _vp])
_verify_accept = _decl("sub_verify_accept", [_vp, C.POINTER(Tree), _i32, _i64, _i32, _f32, _u64,
                                             _i64, _vp, _vp, _vp, _vp, _vp])
_verify_accept_static = _decl("sub_verify_accept_static",
                              [_vp, C.POINTER(Tree), _i32, _i64, _i32, _f32, _u64, _i64, _vp, _vp,
                               _vp, _vp, _vp])
_kv_compact = _decl("sub_kv_compact", [C.POINTER(KVCache), _i64, _vp, _vp, _i32, _vp])
_model_create = _decl("sub_model_create", [C.POINTER(ModelDesc), C.POINTER(_vp)])
_model_destroy = _decl("sub_model_destroy", [_vp])
_model_memory = _decl("sub_model_memory", [_vp, C.POINTER(_i64)])
_model_forward = _decl("sub_model_forward", [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _i32, _i64,
                                             _vp, _vp])
_model_kv = _decl("sub_model_kv", [_vp, C.POINTER(KVCache)])
_generate = _decl("sub_generate", [_vp, _vp, _i32, _i32, C.POINTER(DecodeCfg), _vp,
                                   C.POINTER(Stats)])
_prefill = _decl("sub_prefill", [_vp, _vp, _i32, C.POINTER(DecodeCfg), _vp])
_decode_cycles = _decl("sub_decode_cycles", [_vp, C.POINTER(DecodeCfg), _i32, _vp])
_decode_read = _decl("sub_decode_read", [_vp, _vp, _i32, C.POINTER(_i32), C.POINTER(_i64)])
_cycle_info = _decl("sub_cycle_info", [_vp, C.POINTER(DecodeCfg), C.POINTER(_i64),
                                       C.POINTER(_i64)])

EXPORTED = ["sub_last_error", "sub_version", "sub_pipeline_timeouts", "sub_bounded_wait_check",
            "sub_w4_pack", "sub_w4_dequant", "sub_w4_gemm",
            "sub_wq_pack", "sub_wq_dequant", "sub_wq_gemm", "sub_wq_pack_hqq",
            "sub_bf16_gemm", "sub_tree_attn", "sub_draft_expand", "sub_verify_accept",
            "sub_verify_accept_static",
            "sub_kv_compact", "sub_model_create", "sub_model_destroy", "sub_model_memory",
            "sub_model_forward", "sub_model_kv", "sub_generate", "sub_prefill",
            "sub_decode_cycles", "sub_decode_read", "sub_cycle_info"]


def _check(code):
    if code != SUB_OK:
        raise SubError(code, _lib.sub_last_error().decode())


def version() -> str:
    return _lib.sub_version().decode()


def pipeline_timeouts() -> int:
    """Bounded pipeline waits that ran out on this device (0 in a correct run)."""
    n = C.c_uint32(0)
    _check(_pipeline_timeouts(C.byref(n)))
    return int(n.value)


def bounded_wait_check(max_polls: int) -> int:
    """Run the bounded-wait check kernel; returns its status code
    (SUB_ETIMEOUT when the wait gave up, as it must)."""
    return int(_bounded_wait_check(max_polls))


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _bf16(t):
    assert t.dtype == torch.bfloat16 and t.is_contiguous()
    return t


# ------------------------------------------------------------------ kernels --
def w4_pack(w: torch.Tensor, stream=None):
    """Group-64 min-max int4 pack of a bf16 [N, K] device matrix -> (q, scale, zero)."""
    n, k = w.shape
    g = (k + 63) // 64
    q = torch.empty((n, g * 32), dtype=torch.uint8, device=w.device)
    s = torch.empty((n, g), dtype=torch.bfloat16, device=w.device)
    z = torch.empty((n, g), dtype=torch.bfloat16, device=w.device)
    _check(_w4_pack(_p(_bf16(w)), n, k, 64, _p(q), _p(s), _p(z), _stream(stream)))
    return q, s, z


def w4_dequant(q, s, z, k: int, stream=None):
    n = q.shape[0]
    out = torch.empty((n, k), dtype=torch.bfloat16, device=q.device)
    _check(_w4_dequant(_p(q), _p(s), _p(z), n, k, 64, _p(out), _stream(stream)))
    return out


def w4_gemm(x, q, s, z, n: int, k: int, out=None, stream=None):
    m = x.shape[0]
    y = out if out is not None else torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    _check(_w4_gemm(_p(_bf16(x)), m, _p(q), _p(s), _p(z), n, k, 64, _p(y), _stream(stream)))
    return y


def wq_pack(w: torch.Tensor, bits: int, stream=None):
    """Group-64 min-max pack with 2, 3 or 4 code bits of a bf16 [N, K] device
    matrix -> (q uint8 [N, G * 8 * bits], scale, zero)."""
    n, k = w.shape
    g = (k + 63) // 64
    q = torch.empty((n, g * 8 * bits), dtype=torch.uint8, device=w.device)
    s = torch.empty((n, g), dtype=torch.bfloat16, device=w.device)
    z = torch.empty((n, g), dtype=torch.bfloat16, device=w.device)
    _check(_wq_pack(_p(_bf16(w)), n, k, 64, bits, _p(q), _p(s), _p(z), _stream(stream)))
    return q, s, z


def wq_pack_hqq(w: torch.Tensor, bits: int, iters: int = 20, stream=None):
    """wq_pack with the HQQ-optimised zero point -> (q, scale, zero)."""
    n, k = w.shape
    g = (k + 63) // 64
    q = torch.empty((n, g * 8 * bits), dtype=torch.uint8, device=w.device)
    s = torch.empty((n, g), dtype=torch.bfloat16, device=w.device)
    z = torch.empty((n, g), dtype=torch.bfloat16, device=w.device)
    _check(_wq_pack_hqq(_p(_bf16(w)), n, k, 64, bits, iters, _p(q), _p(s), _p(z),
                        _stream(stream)))
    return q, s, z


def wq_dequant(q, s, z, k: int, bits: int, stream=None):
    n = q.shape[0]
    out = torch.empty((n, k), dtype=torch.bfloat16, device=q.device)
    _check(_wq_dequant(_p(q), _p(s), _p(z), n, k, 64, bits, _p(out), _stream(stream)))
    return out


def wq_gemm(x, q, s, z, n: int, k: int, bits: int, out=None, stream=None):
    m = x.shape[0]
    y = out if out is not None else torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    _check(_wq_gemm(_p(_bf16(x)), m, _p(q), _p(s), _p(z), n, k, 64, bits, _p(y),
                    _stream(stream)))
    return y


def bf16_gemm(x, w, out=None, stream=None):
    m, k = x.shape
    n = w.shape[0]
    y = out if out is not None else torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    _check(_bf16_gemm(_p(_bf16(x)), m, _p(_bf16(w)), n, k, _p(y), _stream(stream)))
    return y


def tree_attn(q, kv: KVCache, layer: int, n_prefix: int, tree_base: int, n_slots: int,
              anc=None, depth=None, scale=None, out=None, stream=None):
    n_q, hq, d = q.shape
    o = out if out is not None else torch.empty_like(q)
    scale = scale if scale is not None else d ** -0.5
    _check(_tree_attn(_p(_bf16(q)), n_q, hq, C.byref(kv), layer, n_prefix, tree_base, n_slots,
                      _p(anc), 0 if anc is None else anc.shape[1], _p(depth), scale, _p(o),
                      _stream(stream)))
    return o


class DeviceTree:
    """Device arrays of a static tree with 1 + depth*width slots."""

    def __init__(self, depth: int, width: int, device="cuda"):
        n = 1 + depth * width
        self.depth_max, self.width = depth, width
        self.token = torch.zeros(n, dtype=torch.int32, device=device)
        self.parent = torch.full((n,), -1, dtype=torch.int32, device=device)
        self.depth = torch.zeros(n, dtype=torch.int32, device=device)
        self.score = torch.zeros(n, dtype=torch.float32, device=device)
        self.anc = torch.full((n, depth + 1), -1, dtype=torch.int32, device=device)
        self.anc[0, 0] = 0

    def struct(self) -> Tree:
        return Tree(self.token.data_ptr(), self.parent.data_ptr(), self.depth.data_ptr(),
                    self.score.data_ptr(), self.anc.data_ptr(), self.width, self.depth_max)


def draft_expand(logits, temperature: float, tree: DeviceTree, level: int, stream=None):
    t = tree.struct()
    _check(_draft_expand(_p(logits), logits.shape[1], temperature, C.byref(t), level,
                         _stream(stream)))


def verify_accept(logits, tree: DeviceTree, n_nodes: int, mode=0, temperature=1.0, seed=0,
                  root_pos=0, stream=None, out=None, with_choice=True):
    """Returns device tensors (accepted slots [D], n_accepted [1], bonus [1],
    choice [n] or None).  `out` reuses those four tensors."""
    return _accept(_verify_accept, logits, tree, n_nodes, mode, temperature, seed, root_pos,
                   stream, out, with_choice)


def verify_accept_static(logits, tree: DeviceTree, n_nodes: int, mode=0, temperature=1.0,
                         seed=0, root_pos=0, stream=None, out=None, with_choice=True):
    """verify_accept on the library's fixed per-device scratch (no device
    allocation inside the call; calls on one device must be ordered)."""
    return _accept(_verify_accept_static, logits, tree, n_nodes, mode, temperature, seed,
                   root_pos, stream, out, with_choice)


def _accept(fn, logits, tree, n_nodes, mode, temperature, seed, root_pos, stream, out,
            with_choice):
    dev = logits.device
    if out is None:
        out = (torch.zeros(max(tree.depth_max, 1), dtype=torch.int32, device=dev),
               torch.zeros(1, dtype=torch.int32, device=dev),
               torch.zeros(1, dtype=torch.int32, device=dev),
               torch.zeros(n_nodes, dtype=torch.int32, device=dev) if with_choice else None)
    acc, na, bonus, choice = out
    t = tree.struct()
    _check(fn(_p(logits), C.byref(t), n_nodes, logits.shape[1], mode, temperature, seed, root_pos,
              _p(acc), _p(na), _p(bonus), _p(choice),
              _stream(stream)))
    return acc, na, bonus, choice


def kv_compact(kv: KVCache, root_pos: int, accepted, n_accepted, max_accept: int, stream=None):
    _check(_kv_compact(C.byref(kv), root_pos, _p(accepted), _p(n_accepted), max_accept,
                       _stream(stream)))


def make_kv(n_layers, n_heads_kv, head_dim, capacity, page_size=64, device="cuda",
            shuffle_seed=None):
    """A paged cache owned by torch tensors (pages optionally permuted)."""
    n_pages = (capacity + page_size - 1) // page_size
    k = torch.zeros((n_layers, n_pages, n_heads_kv, page_size, head_dim), dtype=torch.bfloat16,
                    device=device)
    v = torch.zeros_like(k)
    if shuffle_seed is None:
        pt = torch.arange(n_pages, dtype=torch.int32)
    else:
        pt = torch.randperm(n_pages, generator=torch.Generator().manual_seed(shuffle_seed))
        pt = pt.to(torch.int32)
    pt = pt.to(device)
    st = KVCache(k.data_ptr(), v.data_ptr(), pt.data_ptr(), n_layers, n_heads_kv, head_dim,
                 page_size, n_pages, n_pages * page_size)
    return st, (k, v, pt)


# -------------------------------------------------------------------- model --
class Model:
    """A decoder for SubSpec decoding: resident layers on the device, offloaded
    layers as pinned host originals (streamed for the target) plus device int4
    substitutes (packed here with the library's w4_pack) for the draft."""

    def __init__(self, cfg, weights: dict, max_seq: int, max_depth: int, max_width: int,
                 max_prompt: int | None = None, staging_layers: int = 0, device="cuda",
                 embed_on_host: bool = False, bits=4, hqq_iters: int = 0):
        """bits: code bits of the substitutes (2, 3 or 4), or one entry per
        layer (entries of resident layers are ignored) for mixed precision.
        hqq_iters > 0 packs them with the HQQ-optimised zero point."""
        self.cfg = cfg
        self.keep = []          # tensors the library points into
        self.w4 = {}            # (layer, name) -> (q, scale, zero) device substitutes
        dev = torch.device(device)

        def dev_t(t):
            t = t.to(dev, non_blocking=False).contiguous()
            self.keep.append(t)
            return t

        # the offloaded originals live in one pinned host arena (one large
        # page-locked allocation), each matrix 256-byte aligned inside it
        names = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")
        off_mats = [(i, n) for i in range(cfg.n_resident, cfg.n_layers) for n in names]
        sizes = [weights["layers"][i][n].numel() * 2 for i, n in off_mats]
        total = sum((b + 255) // 256 * 256 for b in sizes)
        arena = torch.empty(max(total, 256), dtype=torch.uint8, pin_memory=True)
        self.keep.append(arena)
        host_of, pos = {}, 0
        for (i, n), b in zip(off_mats, sizes):
            w = weights["layers"][i][n]
            view = arena[pos:pos + b].view(torch.bfloat16).view(w.shape)
            view.copy_(w)
            host_of[(i, n)] = view
            pos += (b + 255) // 256 * 256

        layers = (LayerDesc * cfg.n_layers)()
        for i, lw in enumerate(weights["layers"]):
            L = layers[i]
            L.attn_norm = dev_t(lw["attn_norm"]).data_ptr()
            L.ffn_norm = dev_t(lw["ffn_norm"]).data_ptr()
            w4n = ("q4", "k4", "v4", "o4", "g4", "u4", "d4")
            for name, qn in zip(names, w4n):
                w = lw[name]
                if i < cfg.n_resident:
                    setattr(L, name, dev_t(w).data_ptr())
                else:
                    b = bits[i] if isinstance(bits, (list, tuple)) else bits
                    wd = w.to(dev).contiguous()
                    if hqq_iters > 0:
                        q, s, z = wq_pack_hqq(wd, b, hqq_iters)
                    else:
                        q, s, z = w4_pack(wd) if b == 4 else wq_pack(wd, b)
                    self.w4[(i, name)] = (q, s, z)
                    setattr(L, qn, W4(q.data_ptr(), s.data_ptr(), z.data_ptr(), b))
                    setattr(L, name, host_of[(i, name)].data_ptr())
                    del wd
        torch.cuda.synchronize(dev)
        d = ModelDesc()
        for f in ("n_layers", "hidden", "n_heads_q", "n_heads_kv", "head_dim", "ffn", "vocab",
                  "n_resident"):
            setattr(d, f, getattr(cfg, f))
        d.rope_theta = cfg.rope_theta
        d.rms_eps = cfg.rms_eps
        if embed_on_host:   # read in place from pinned host memory
            emb = weights["embed"].to("cpu").contiguous().pin_memory()
            self.keep.append(emb)
            d.embed = emb.data_ptr()
        else:
            d.embed = dev_t(weights["embed"]).data_ptr()
        d.lm_head = dev_t(weights["lm_head"]).data_ptr()
        d.final_norm = dev_t(weights["final_norm"]).data_ptr()
        d.layers = layers
        d.max_seq = max_seq
        d.max_depth = max_depth
        d.max_width = max_width
        d.staging_layers = staging_layers
        d.max_prompt = max_prompt if max_prompt is not None else max_seq
        self._layers = layers
        h = _vp()
        _check(_model_create(C.byref(d), C.byref(h)))
        self.handle = h

    def close(self):
        """Destroy the model and drop the tensors it pointed into (the pinned
        originals and the device substitutes)."""
        if getattr(self, "handle", None) and self.handle.value:
            _model_destroy(self.handle)
            self.handle = _vp()
        self.keep = []
        self.w4 = {}

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def device_bytes(self) -> int:
        b = _i64()
        _check(_model_memory(self.handle, C.byref(b)))
        return b.value

    def kv(self) -> KVCache:
        kv = KVCache()
        _check(_model_kv(self.handle, C.byref(kv)))
        return kv

    def forward(self, which: int, tokens, slot0: int, n_prefix: int, depth=None, anc=None,
                logits=None, stream=None):
        n = tokens.shape[0]
        _check(_model_forward(self.handle, which, _p(tokens), n, slot0, _p(depth), _p(anc),
                              0 if anc is None else anc.shape[1], n_prefix, _p(logits),
                              _stream(stream)))
        return logits

    @staticmethod
    def decode_cfg(depth, width, draft_temp=0.2, mode=0, target_temp=1.0, seed=0,
                   use_graph=True, stop_logp=None, verify_reuse=False) -> DecodeCfg:
        """stop_logp: None (every level drafted) or a negative threshold for adaptive
        depth; verify_reuse: the verify starts from the draft's leading layers."""
        return DecodeCfg(depth, width, draft_temp, mode, target_temp, seed, int(use_graph),
                         0.0 if stop_logp is None else float(stop_logp), int(verify_reuse))

    def prefill(self, prompt, cfg: DecodeCfg, stream=None):
        self._prompt = prompt.to(torch.int32).contiguous()
        _check(_prefill(self.handle, C.c_void_p(self._prompt.data_ptr()), self._prompt.numel(),
                        C.byref(cfg), _stream(stream)))

    def decode_cycles(self, cfg: DecodeCfg, n_cycles: int, stream=None):
        _check(_decode_cycles(self.handle, C.byref(cfg), n_cycles, _stream(stream)))

    def decode_read(self, n: int = 0):
        """-> (emitted tokens int32 CPU tensor [min(n, emitted)], emitted, cycles)."""
        out = torch.zeros(max(n, 1), dtype=torch.int32)
        e, c = _i32(), _i64()
        _check(_decode_read(self.handle, C.c_void_p(out.data_ptr()), n, C.byref(e), C.byref(c)))
        return out[:min(n, e.value)], e.value, c.value

    def cycle_info(self, cfg: DecodeCfg):
        k, b = _i64(), _i64()
        _check(_cycle_info(self.handle, C.byref(cfg), C.byref(k), C.byref(b)))
        return k.value, b.value

    def generate(self, prompt, n_new: int, depth: int, width: int, draft_temp=0.2, mode=0,
                 target_temp=1.0, seed=0, use_graph=True, stop_logp=None, verify_reuse=False):
        """prompt: int32 CPU tensor -> (int32 CPU tensor [n_new], Stats)."""
        p = prompt.to(torch.int32).contiguous()
        out = torch.zeros(n_new, dtype=torch.int32)
        cfg = self.decode_cfg(depth, width, draft_temp, mode, target_temp, seed, use_graph,
                              stop_logp, verify_reuse)
        st = Stats()
        _check(_generate(self.handle, C.c_void_p(p.data_ptr()), p.numel(), n_new, C.byref(cfg),
                         C.c_void_p(out.data_ptr()), C.byref(st)))
        return out, st
