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
