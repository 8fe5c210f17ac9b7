"""Unified paged attention: parity with the oracle and the causal contract.

K/V are seeded synthetic values written straight into caller-owned pool
memory ([layer][page][K/V][kv_head][16][hd]); q rows are seeded per
(request, position), so the same logical row can be recomputed under any
batch composition, chunking, page placement or split placement.
"""

import numpy as np
import pytest

from attn_scenario import SPECS, Scenario, check_parity as _check_parity
from gpu_util import bits, ready

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_decode_and_prefill_rows_vs_oracle(hd):
    ready()
    lens = [1, 17, 64, 65, 511, 512, 513, 1100]
    sc = Scenario(SPECS[hd], lens, num_pages=200, seed=hd)
    # decode rows (last position), a full prefill of one request, and a chunk
    res = sc.run([(r, n - 1, 1) for r, n in enumerate(lens)])
    _check_parity(sc, res)
    res = sc.run([(6, 0, 513), (7, 1000, 100), (2, 3, 61)])
    _check_parity(sc, res)


def test_sliding_window_vs_oracle():
    ready()
    spec = SPECS[128].with_(sliding_window=100, local_global_period=1000)
    lens = [50, 99, 100, 101, 700]
    sc = Scenario(spec, lens, num_pages=120, seed=3)
    res = sc.run([(r, n - 1, 1) for r, n in enumerate(lens)])
    _check_parity(sc, res, window=100)
    res = sc.run([(4, 0, 700)])
    _check_parity(sc, res, window=100)


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_causal_contract_bitwise_across_schedules(hd):
    # The same (request, position) row must be bit-identical whatever the
    # query length, row index, batch, chunking and split placement.
    ready()
    lens = [300, 1030, 77]
    sc = Scenario(SPECS[hd], lens, num_pages=120, seed=11 + hd)
    runs = [
        [(0, 0, 300), (1, 0, 1030), (2, 0, 77)],                  # one prefill each
        [(1, 0, 500), (0, 0, 150), (2, 0, 10)],                   # chunks ...
        [(1, 500, 530), (0, 150, 150), (2, 10, 67)],              # ... continued
        [(2, 76, 1), (0, 299, 1), (1, 1029, 1)],                  # decode rows
        [(0, 299, 1)], [(1, 511, 1)], [(1, 512, 1)],              # alone, at split edges
        [(1, 1000, 30), (0, 290, 10)],
        [(0, 63, 2), (1, 63, 2)],
        # decode-shaped CTAs of 9..16 rows (q_len 3 or 4 with a group of 4; 5..8 with a group of 2),
        # which keep the softmax of the warp's rows 8..15, next to CTAs of at most 8 rows, which skip
        # it, in one launch
        [(0, 100, 3), (1, 600, 1), (2, 20, 2)],
        [(1, 700, 4), (0, 200, 5), (2, 40, 8)],
    ]
    seen = {}
    for parts in runs:
        for key, row in sc.run(parts).items():
            b = bits(row)
            if key in seen:
                np.testing.assert_array_equal(b, seen[key], err_msg=f"row {key} differs in {parts}")
            else:
                seen[key] = b
    assert len(seen) > 1400


def test_page_placement_does_not_change_bits():
    ready()
    lens = [333, 700]
    sc = Scenario(SPECS[128], lens, num_pages=80, seed=5)
    a = sc.run([(0, 0, 333), (1, 650, 50)])
    sc.place(np.arange(80)[::-1].copy())  # a different physical layout of the same logical K/V
    b = sc.run([(0, 0, 333), (1, 650, 50)])
    for k in a:
        np.testing.assert_array_equal(bits(a[k]), bits(b[k]))
