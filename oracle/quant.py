"""Group-64 min-max int4 substitutes (test infrastructure only).

The pages build the draft's substitute layers by quantising each offloaded
target layer to 4 bits, data-free ("Low-Bit Shadow" report, 2.2 Step 4;
"Speculate Deep and Accurate" card, Approach and Problem).  They use HQQ;
this library's quantiser is the plainer min-max one with the dequant rule
W = (q - z) * s, one (s, z) pair per row and group of 64 consecutive inputs
along the reduction dimension K, s and z stored as bf16.

Reading of the steps (the pages give none of them):
  lo, hi = min, max of the group's real elements (a last group may be short)
  s = bf16(fp32(hi - lo) / 15); if s == 0 then s = 1   (covers hi == lo)
  z = bf16(fp32(-lo) / s)                              (a bf16 float, not an int)
  q = clamp(rint_even(fp32(w / s) + z), 0, 15)
  deq = bf16((q - z) * s)   -- exact in fp32, one rounding to bf16
Packing: byte j of a group holds element 2j in the low nibble and 2j+1 in the
high nibble; the 32 bytes of a group are contiguous; nibbles past K are 0.
All fp32 steps are single IEEE operations (NumPy float32 arithmetic).
"""
import numpy as np

from .bf16 import round_bf16, mm

GROUP = 64


def n_groups(k: int) -> int:
    return (k + GROUP - 1) // GROUP


def w4_pack(w) -> tuple:
    """w: float32 [N, K] of bf16 values -> (q uint8 [N, G*32], s, z float32 [N, G]
    holding bf16 values)."""
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    g_count = n_groups(k)
    codes = np.zeros((n, g_count * GROUP), dtype=np.uint8)
    s_all = np.zeros((n, g_count), dtype=np.float32)
    z_all = np.zeros((n, g_count), dtype=np.float32)
    fifteen = np.float32(15.0)
    for g in range(g_count):
        blk = w[:, g * GROUP:min(k, (g + 1) * GROUP)]
        lo = blk.min(axis=1)
        hi = blk.max(axis=1)
        s = round_bf16((hi - lo) / fifteen)
        s = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
        z = round_bf16((-lo) / s)
        t = (blk / s[:, None]) + z[:, None]          # two fp32 ops, each rounded
        q = np.clip(np.rint(t), 0, 15).astype(np.uint8)
        codes[:, g * GROUP:g * GROUP + blk.shape[1]] = q
        s_all[:, g] = s
        z_all[:, g] = z
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, s_all, z_all


def unpack_codes(q, k: int) -> np.ndarray:
    """uint8 [N, G*32] -> int codes [N, K] (low nibble = even element)."""
    q = np.asarray(q, dtype=np.uint8)
    n = q.shape[0]
    codes = np.empty((n, q.shape[1] * 2), dtype=np.uint8)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    return codes[:, :k]


def w4_dequant(q, s, z, k: int) -> np.ndarray:
    """bf16((q - z) * s) per element, as float32 [N, K].  (q - z) and the
    product are exact in float64 and in fp32 (q has 4 bits, z and s 8
    significant bits), so the only rounding is the final one to bf16."""
    codes = unpack_codes(q, k).astype(np.float64)
    gidx = np.arange(k) // GROUP
    s64 = np.asarray(s, np.float64)[:, gidx]
    z64 = np.asarray(z, np.float64)[:, gidx]
    return round_bf16(((codes - z64) * s64).astype(np.float32))


def w4_gemm(x, q, s, z, k: int) -> np.ndarray:
    """Y[M, N] = X[M, K] . deq(W)^T, accumulated in float64, rounded to fp32."""
    return mm(x, w4_dequant(q, s, z, k))


# ---------------------------------------------------------------------------
# 2-, 3- and 4-bit substitutes (lower and mixed precision for the draft's
# substitute layers: "Low-Bit Shadow" report 5.1 point 2 and 10.1 (2), which
# leave 2/3-bit substitutes untested, and 10.2 (10), per-layer precision
# chosen by sensitivity).  The quantiser is the min-max one above with
# L = 2^bits - 1 levels in place of 15:
#   s = bf16(fp32(hi - lo) / L); if s == 0 then s = 1;  z = bf16(fp32(-lo) / s)
#   q = clamp(rint_even(fp32(w / s) + z), 0, L);   deq = bf16((q - z) * s)
# Code layout of one 64-element group (8 * bits bytes, groups contiguous):
#   bits 4: 32 bytes, byte j = element 2j (low nibble) | element 2j+1 << 4
#   bits 2: 16 bytes, byte j = elements 4j .. 4j+3 at bits 0-1, 2-3, 4-5, 6-7
#   bits 3: 24 bytes, bytes 0..15 the 2-bit layout of (code & 3), bytes
#           16..23 the high bits: bit i of byte 16 + j = code(8j + i) >> 2
# Codes past K are 0.
# ---------------------------------------------------------------------------
BITS = (2, 3, 4)


def group_bytes(bits: int) -> int:
    return 8 * bits


def wq_codes(w, bits: int) -> tuple:
    """w: float32 [N, K] of bf16 values -> (codes uint8 [N, K], s, z float32
    [N, G] holding bf16 values), the min-max quantiser with 2^bits - 1 levels."""
    assert bits in BITS
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    g_count = n_groups(k)
    levels = np.float32(2 ** bits - 1)
    codes = np.zeros((n, k), dtype=np.uint8)
    s_all = np.zeros((n, g_count), dtype=np.float32)
    z_all = np.zeros((n, g_count), dtype=np.float32)
    for g in range(g_count):
        c0, c1 = g * GROUP, min(k, (g + 1) * GROUP)
        blk = w[:, c0:c1]
        lo = blk.min(axis=1)
        hi = blk.max(axis=1)
        s = round_bf16((hi - lo) / levels)
        s = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
        z = round_bf16((-lo) / s)
        t = (blk / s[:, None]) + z[:, None]          # two fp32 ops, each rounded
        codes[:, c0:c1] = np.clip(np.rint(t), 0, levels).astype(np.uint8)
        s_all[:, g] = s
        z_all[:, g] = z
    return codes, s_all, z_all


def wq_pack_codes(codes, bits: int) -> np.ndarray:
    """codes uint8 [N, K] (each < 2^bits) -> packed uint8 [N, G * 8 * bits]."""
    codes = np.asarray(codes, dtype=np.uint8)
    n, k = codes.shape
    g_count = n_groups(k)
    full = np.zeros((n, g_count * GROUP), dtype=np.uint8)
    full[:, :k] = codes
    grp = full.reshape(n, g_count, GROUP)
    if bits == 4:
        out = grp[:, :, 0::2] | (grp[:, :, 1::2] << 4)
    else:
        lo2 = grp & 3
        out = lo2[:, :, 0::4] | (lo2[:, :, 1::4] << 2) | (lo2[:, :, 2::4] << 4) | (lo2[:, :, 3::4] << 6)
        if bits == 3:
            hb = (grp >> 2) & 1
            plane = np.zeros((n, g_count, 8), dtype=np.uint8)
            for i in range(8):
                plane |= (hb[:, :, i::8] << i).astype(np.uint8)
            out = np.concatenate([out, plane], axis=2)
    return out.reshape(n, g_count * group_bytes(bits)).astype(np.uint8)


def wq_unpack_codes(q, k: int, bits: int) -> np.ndarray:
    """packed uint8 [N, G * 8 * bits] -> codes [N, K]."""
    q = np.asarray(q, dtype=np.uint8)
    n = q.shape[0]
    gb = group_bytes(bits)
    g_count = q.shape[1] // gb
    grp = q.reshape(n, g_count, gb)
    codes = np.zeros((n, g_count, GROUP), dtype=np.uint8)
    if bits == 4:
        codes[:, :, 0::2] = grp & 0xF
        codes[:, :, 1::2] = grp >> 4
    else:
        for i in range(4):
            codes[:, :, i::4] = (grp[:, :, :16] >> (2 * i)) & 3
        if bits == 3:
            for i in range(8):
                codes[:, :, i::8] |= ((grp[:, :, 16:24] >> i) & 1) << 2
    return codes.reshape(n, g_count * GROUP)[:, :k]


def wq_pack(w, bits: int) -> tuple:
    """w: float32 [N, K] of bf16 values -> (q uint8 [N, G * 8 * bits], s, z)."""
    codes, s, z = wq_codes(w, bits)
    return wq_pack_codes(codes, bits), s, z


def wq_dequant(q, s, z, k: int, bits: int) -> np.ndarray:
    """bf16((q - z) * s) per element, as float32 [N, K] (exact before the
    rounding, as for 4 bits: fewer code bits only shorten q - z)."""
    codes = wq_unpack_codes(q, k, bits).astype(np.float64)
    gidx = np.arange(k) // GROUP
    s64 = np.asarray(s, np.float64)[:, gidx]
    z64 = np.asarray(z, np.float64)[:, gidx]
    return round_bf16(((codes - z64) * s64).astype(np.float32))


def wq_gemm(x, q, s, z, k: int, bits: int) -> np.ndarray:
    """Y[M, N] = X[M, K] . deq(W)^T, accumulated in float64, rounded to fp32."""
    return mm(x, wq_dequant(q, s, z, k, bits))


# ---------------------------------------------------------------------------
# HQQ zero-point optimisation (the pages build their substitutes with HQQ,
# "Low-Bit Shadow" report Critique 3 and 6.2, and give none of its steps).
# Restated here from the published half-quadratic method: keep the min-max
# scale s and, per group, alternate
#   q  = clamp(rint(w / s + z), 0, L)            codes for the current zero
#   r  = w - s (q - z)                            the residual
#   e  = sign(r) max(|r| - |r|^(p-1) / beta, 0)   the l_p shrinkage of r
#   z  = mean(q - (w - e) / s)                    the zero minimising
#                                                 sum (w - e - s (q - z))^2
#   beta = beta * kappa
# for a fixed number of iterations, keeping the zero with the smallest
# sum |r| seen (the first one, the min-max zero, included; ties keep the
# earlier).  Parameters: p = 1/2 (HQQ's default is 0.7; at 1/2,
# |r|^(p-1) = 1 / sqrt|r| is two correctly rounded fp32 operations),
# beta = 10, kappa = 1.01, 20 iterations (HQQ's defaults).  The kept zero is
# rounded to bf16 and the codes are formed with it, as in the min-max rule.
# All arithmetic is fp32, each operation rounded; the sums over a group run
# in one fixed pairwise order (pair_sum64), and the mean divides by the
# group's element count.
# ---------------------------------------------------------------------------
HQQ_ITERS, HQQ_BETA, HQQ_KAPPA, HQQ_P = 20, 10.0, 1.01, 0.5


def pair_sum64(x) -> np.ndarray:
    """Sum over the last axis (64 entries) in a fixed order: a_l = x[2l] +
    x[2l+1], then five rounds of a_l = a_l + a_(l xor o), o = 16, 8, 4, 2, 1;
    the result is a_0.  fp32, every addition rounded."""
    x = np.asarray(x, np.float32)
    a = x[..., 0::2] + x[..., 1::2]
    idx = np.arange(32)
    for o in (16, 8, 4, 2, 1):
        a = a + a[..., idx ^ o]
    return a[..., 0]


def shrink_lp(r, beta, p=HQQ_P) -> np.ndarray:
    """sign(r) max(|r| - |r|^(p-1) / beta, 0) in fp32; 0 where r == 0."""
    r = np.asarray(r, np.float32)
    ar = np.abs(r)
    safe = np.where(ar > 0, ar, np.float32(1))
    if p == 0.5:
        pw = np.float32(1) / np.sqrt(safe)
    else:
        pw = np.power(safe, np.float32(p - 1)).astype(np.float32)
    th = np.where(ar > 0, pw / np.float32(beta), np.float32(0)).astype(np.float32)
    return (np.sign(r) * np.maximum(ar - th, np.float32(0))).astype(np.float32)


def hqq_codes(w, bits: int, iters=HQQ_ITERS, beta0=HQQ_BETA, kappa=HQQ_KAPPA, p=HQQ_P) -> tuple:
    """w: float32 [N, K] of bf16 values -> (codes uint8 [N, K], s, z) with the
    min-max scale and the HQQ-optimised zero (see above)."""
    assert bits in BITS and iters >= 1
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    g_count = n_groups(k)
    levels = np.float32(2 ** bits - 1)
    codes = np.zeros((n, k), dtype=np.uint8)
    s_all = np.zeros((n, g_count), dtype=np.float32)
    z_all = np.zeros((n, g_count), dtype=np.float32)
    for g in range(g_count):
        c0, c1 = g * GROUP, min(k, (g + 1) * GROUP)
        cnt = c1 - c0
        blk = np.zeros((n, GROUP), np.float32)
        blk[:, :cnt] = w[:, c0:c1]
        valid = np.zeros(GROUP, bool)
        valid[:cnt] = True
        lo = blk[:, :cnt].min(axis=1)
        hi = blk[:, :cnt].max(axis=1)
        s = round_bf16((hi - lo) / levels)
        s = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
        z = ((-lo) / s).astype(np.float32)
        beta = np.float32(beta0)
        best_z, best_err = z.copy(), None
        for _ in range(iters):
            q = np.clip(np.rint((blk / s[:, None]) + z[:, None]), 0, levels).astype(np.float32)
            r = (blk - s[:, None] * (q - z[:, None])).astype(np.float32)
            r = np.where(valid, r, np.float32(0))
            err = pair_sum64(np.abs(r))
            if best_err is None:
                best_err = err
            else:
                better = err < best_err
                best_err = np.where(better, err, best_err)
                best_z = np.where(better, z, best_z)
            e = shrink_lp(r, beta, p)
            t = np.where(valid, q - (blk - e) / s[:, None], np.float32(0)).astype(np.float32)
            z = (pair_sum64(t) / np.float32(cnt)).astype(np.float32)
            beta = np.float32(beta * np.float32(kappa))
        zb = round_bf16(best_z)
        t = (blk[:, :cnt] / s[:, None]) + zb[:, None]
        codes[:, c0:c1] = np.clip(np.rint(t), 0, levels).astype(np.uint8)
        s_all[:, g] = s
        z_all[:, g] = zb
    return codes, s_all, z_all


def wq_pack_hqq(w, bits: int, iters=HQQ_ITERS) -> tuple:
    """HQQ-zero substitutes in the wq layouts: (q, s, z); dequantise with
    wq_dequant like any other."""
    codes, s, z = hqq_codes(w, bits, iters)
    return wq_pack_codes(codes, bits), s, z
