"""Token choice for the oracle (test infrastructure).

* Greedy: argmax over the vocabulary, the lowest index among equal maxima.
* Seeded sampling: Gumbel-max, ``argmax_i(l_i / T + G_i)`` with
  ``G_i = -log(-log(u_i))``, the uniforms drawn from the counter-based
  Philox4x32-10 generator of Salmon, Moraes, Dror and Shaw, "Parallel Random
  Numbers: As Easy as 1, 2, 3" (SC'11), written here from that definition.

The per-request sampler state is (seed, counter): the counter is the index
of the output token and advances once per emitted token.  That state is the
"initial sampler state" of 深入解析 Vosti §二 Definition 2.1 (sampler_0).

Stream layout (shared contract with the CUDA sampler, stated, not shared
code): for vocabulary index i, key = (seed & 0xffffffff, seed >> 32),
counter = (i // 4, step & 0xffffffff, step >> 32, 0x5644), and the uniform
is word i % 4 of the block, mapped to u = ((word >> 8) + 0.5) / 2**24, a
24-bit uniform that float32 holds exactly and that is never 0 or 1.

Pinned by tests/test_oracle_sampler.py: Philox known-answer vectors from
the Random123 distribution, a chi-square uniformity check, argmax against
brute force, and Gumbel-max frequencies against the softmax distribution.
"""

import numpy as np

_M0 = 0xD2511F53
_M1 = 0xCD9E8D57
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """One Philox4x32 block with 10 rounds; ctr: 4 words, key: 2 words."""
    c0, c1, c2, c3 = (int(v) & _MASK for v in ctr)
    k0, k1 = (int(v) & _MASK for v in key)
    for r in range(10):
        if r:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> 32, p0 & _MASK
        hi1, lo1 = p1 >> 32, p1 & _MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return (c0, c1, c2, c3)


def philox_words(seed: int, step: int, n: int) -> np.ndarray:
    """The n 32-bit words used for vocabulary indices 0..n-1 at one step."""
    key = (seed & _MASK, (seed >> 32) & _MASK)
    out = np.empty(n, dtype=np.uint64)
    for b in range((n + 3) // 4):
        w = philox4x32_10((b, step & _MASK, (step >> 32) & _MASK, 0x5644), key)
        for j in range(4):
            i = 4 * b + j
            if i < n:
                out[i] = w[j]
    return out


def uniforms(seed: int, step: int, n: int) -> np.ndarray:
    return ((philox_words(seed, step, n) >> np.uint64(8)).astype(np.float64) + 0.5) / 2.0 ** 24


def argmax_lowest(logits) -> int:
    """Index of the maximum; the lowest index wins ties."""
    x = np.asarray(logits)
    m = x.max()
    return int(np.flatnonzero(x == m)[0])


def gumbel_scores(logits, temperature: float, seed: int, step: int) -> np.ndarray:
    u = uniforms(seed, step, len(logits))
    g = -np.log(-np.log(u))
    return np.asarray(logits, dtype=np.float64) / temperature + g


def sample(logits, temperature: float, seed: int, step: int) -> int:
    """Greedy for temperature <= 0, else seeded Gumbel-max."""
    if temperature <= 0:
        return argmax_lowest(logits)
    return argmax_lowest(gumbel_scores(logits, temperature, seed, step))
