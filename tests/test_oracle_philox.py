"""Pins of the oracle's Philox4x32-10 and Gumbel noise: the known-answer
vectors published with the Random123 library (Salmon et al., SC'11) and the
Gumbel-max property (argmax of logits/T + Gumbel noise is distributed as
softmax(logits/T)), checked statistically."""
import numpy as np

from oracle import philox


def _one(ctr, key):
    out = philox.philox4x32_10([np.uint64(c) for c in ctr], [np.uint64(k) for k in key])
    return [int(v) for v in out]


def test_philox_known_answers():
    assert _one((0, 0, 0, 0), (0, 0)) == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    f = 0xFFFFFFFF
    assert _one((f, f, f, f), (f, f)) == [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]
    assert _one((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0)) == \
        [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]


def test_uniform_words_layout():
    # word for token v is output word v % 4 of the block counter (v // 4, pos, 0, 0)
    seed = (5 << 32) | 9
    w = philox.uniform_words(seed, 17, 10)
    blk2 = _one((2, 17, 0, 0), (9, 5))
    assert [int(x) for x in w[8:10]] == blk2[:2]


def test_gumbel_max_is_softmax_sampling():
    logits = np.array([0.3, -0.4, 1.1, 0.0])
    temp = 0.6
    n = 40000
    counts = np.zeros(4)
    for p in range(n):
        g = philox.gumbel(1234, p, 4)
        counts[np.argmax(logits / temp + g)] += 1
    probs = np.exp(logits / temp) / np.exp(logits / temp).sum()
    sd = np.sqrt(n * probs * (1 - probs))
    assert np.all(np.abs(counts - n * probs) < 5 * sd), (counts / n, probs)


def test_gumbel_uniform_open_interval():
    r = np.array([0, 511, 512, 0xFFFFFFFF], dtype=np.float64)
    x = (np.floor(r / 512.0) + 0.5) * 2.0 ** -23
    assert np.all((x > 0) & (x < 1))
    g = philox.gumbel(7, 3, 1000)
    assert np.all(np.isfinite(g))
    # Gumbel(0,1) mean is the Euler-Mascheroni constant
    big = np.concatenate([philox.gumbel(7, p, 4096) for p in range(8)])
    assert abs(big.mean() - 0.5772156649) < 0.03
