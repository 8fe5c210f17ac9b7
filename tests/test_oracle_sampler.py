"""Pins for the oracle's token choice: Philox4x32-10 and Gumbel-max."""

import numpy as np
from scipy import stats

from oracle import sampler


def test_philox_known_answer_vectors():
    # Known-answer vectors published with the Random123 library for
    # philox4x32 with 10 rounds (counter, key) -> output.
    kat = [
        ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
        ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
        ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
         (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
    ]
    for ctr, key, want in kat:
        assert sampler.philox4x32_10(ctr, key) == want


def test_uniforms_chi_square():
    u = np.concatenate([sampler.uniforms(1234, s, 4096) for s in range(8)])
    assert np.all((u > 0) & (u < 1))
    counts, _ = np.histogram(u, bins=64, range=(0, 1))
    _, pval = stats.chisquare(counts)
    assert pval > 1e-4


def test_argmax_lowest_index():
    rng = np.random.default_rng(5)
    for _ in range(200):
        x = rng.integers(-3, 4, size=17).astype(np.float32)
        m = x.max()
        brute = min(i for i in range(len(x)) if x[i] == m)
        assert sampler.argmax_lowest(x) == brute


def test_gumbel_max_matches_softmax_frequencies():
    logits = np.array([1.0, 0.0, -0.5, 2.0], dtype=np.float32)
    T = 0.8
    n = 20000
    counts = np.zeros(4)
    for step in range(n):
        counts[sampler.sample(logits, T, seed=99, step=step)] += 1
    p = np.exp(logits / T) / np.exp(logits / T).sum()
    sd = np.sqrt(n * p * (1 - p))
    assert np.all(np.abs(counts - n * p) < 5 * sd), (counts, n * p)


def test_temperature_zero_is_greedy():
    x = np.array([0.5, 3.0, 3.0, -1.0])
    assert sampler.sample(x, 0.0, seed=1, step=0) == 1
