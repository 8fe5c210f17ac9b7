"""Failure source 4 of 深入解析 Vosti §四 on the CPU: a tiled online softmax
that replaces the -inf maximum of a fully masked key tile by 0 gives
different bits depending on whether a row's partition visits that tile;
the masking rule of §六 6.2 (a tile without a visible key leaves the row's
running state unchanged) makes the bits independent of it.

The model is a float32 online softmax over 32-key tiles written here for the
demonstration (it is neither the oracle nor the GPU kernel); the kernel
follows the rule and `test_failure_sources_gpu.py` checks it bitwise.
"""

import numpy as np

TILE = 32


def _row(q, K, V, lo, hi, first_tile, zero_for_masked_max):
    """Attention of one query over keys [lo, hi], scanning key tiles from first_tile."""
    f = np.float32
    scale = f(1.0 / np.sqrt(q.shape[0]))
    m, l, o = f(-np.inf), f(0), np.zeros(V.shape[1], np.float32)
    for t0 in range(first_tile * TILE, hi + 1, TILE):
        idx = np.arange(t0, min(t0 + TILE, K.shape[0]))
        s = (K[idx] @ q).astype(np.float32) * scale
        s = np.where((idx >= lo) & (idx <= hi), s, f(-np.inf))
        tmax = s.max()
        if zero_for_masked_max and tmax == -np.inf:
            tmax = f(0)  # the failure: a fully masked tile contributes a maximum of 0
        m_new = max(m, tmax)
        if m_new == -np.inf:
            continue  # nothing visible yet: the state stays as it is
        alpha = np.exp(m - m_new, dtype=np.float32)
        p = np.exp(s - m_new, dtype=np.float32)
        l = l * alpha + p.sum(dtype=np.float32)
        o = o * alpha + (p @ V[idx]).astype(np.float32)
        m = m_new
    return o / l


def _rows(zero_for_masked_max, first_tile_of):
    rng = np.random.default_rng(5)
    n, hd, window = 400, 64, 100
    K = -np.abs(rng.standard_normal((n, hd))).astype(np.float32)  # scores mostly negative
    V = rng.standard_normal((n, hd)).astype(np.float32)
    out = []
    for p in range(150, n):
        q = np.abs(rng.standard_normal(hd)).astype(np.float32)
        lo = p - window + 1
        out.append(_row(q, K, V, lo, p, first_tile_of(lo), zero_for_masked_max))
    return np.array(out)


def test_visiting_fully_masked_tiles_moves_bits_only_under_the_faulty_rule():
    from_zero = lambda lo: 0               # a partition that scans every tile of the split
    from_visible = lambda lo: lo // TILE   # a partition that starts at the first visible tile
    good_a, good_b = _rows(False, from_zero), _rows(False, from_visible)
    bad_a, bad_b = _rows(True, from_zero), _rows(True, from_visible)
    assert np.array_equal(good_a.view(np.uint32), good_b.view(np.uint32))
    assert not np.array_equal(bad_a.view(np.uint32), bad_b.view(np.uint32))
    # both rules compute attention; only the rounding differs
    assert np.allclose(bad_a, good_a, rtol=1e-5, atol=1e-6)
    assert np.array_equal(bad_b.view(np.uint32), good_b.view(np.uint32))  # no masked tile visited: identical
