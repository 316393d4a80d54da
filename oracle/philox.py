"""Philox4x32-10 and the Gumbel noise of sampled verification (test
infrastructure only).

Sampled verification: the pages verify at T > 0 ("Low-Bit Shadow" report,
3.6; "Speculate Deep and Accurate" card, measured effects at temperature 0.6)
and insist the output stays identical to plain target sampling (report,
Critique 1 and 10.2 (4): tokenwise agreement under fixed seeds).  This
library reads that as a coupled sampler: the target's token at absolute
position p is argmax_v (z_v / T + g(seed, p, v)) with Gumbel noise g that
depends only on (seed, p, v).  Plain sampled decoding and SubSpec then pick the
same token at every position, so the stream is lossless token for token.

Philox4x32-10 follows Salmon, Moraes, Dror and Shaw, "Parallel random numbers:
as easy as 1, 2, 3" (SC'11): 10 rounds of two 32x32->64 multiplies with the
key bumped by the Weyl constants between rounds.

Noise for (seed, p, v): counter = (v // 4, p, 0, 0), key = (seed & 0xffffffff,
seed >> 32), word r = output[v % 4];  x = ((r >> 9) + 0.5) * 2^-23, which is
exact in fp32 and lies strictly inside (0, 1);  g = -log(-log(x)).
"""
import numpy as np

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """ctr: 4 arrays (or ints) of uint32, key: 2 of uint32 -> 4 uint32 arrays."""
    c = [np.asarray(v, dtype=np.uint64) & MASK32 for v in ctr]
    k0 = np.asarray(key[0], dtype=np.uint64) & MASK32
    k1 = np.asarray(key[1], dtype=np.uint64) & MASK32
    for rnd in range(10):
        if rnd:
            k0 = (k0 + PHILOX_W0) & MASK32
            k1 = (k1 + PHILOX_W1) & MASK32
        p0 = np.uint64(PHILOX_M0) * c[0]
        p1 = np.uint64(PHILOX_M1) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return [v.astype(np.uint32) for v in c]


def uniform_words(seed: int, pos: int, vocab: int) -> np.ndarray:
    """The 32-bit word r(seed, pos, v) for v in [0, vocab)."""
    v = np.arange(vocab, dtype=np.uint64)
    blocks = v // 4
    zeros = np.zeros_like(blocks)
    out = philox4x32_10((blocks, np.full_like(blocks, pos), zeros, zeros),
                        (seed & MASK32, (seed >> 32) & MASK32))
    stacked = np.stack(out, axis=1)              # [vocab, 4]
    return stacked[np.arange(vocab), (v % 4).astype(np.int64)]


def gumbel(seed: int, pos: int, vocab: int) -> np.ndarray:
    """Gumbel(0,1) noise g(seed, pos, v) in float64."""
    r = uniform_words(seed, pos, vocab).astype(np.float64)
    x = (np.floor(r / 512.0) + 0.5) * 2.0 ** -23
    return -np.log(-np.log(x))
