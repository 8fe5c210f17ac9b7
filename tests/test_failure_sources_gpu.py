"""The four failure sources the pages list, as negative tests on the GPU.

深入解析 Vosti §四 names four ways production kernels lose batch invariance in
attention.  Each test below sets up the situation that breaks those kernels
and requires bitwise-equal attention rows here:

1. a batch-wide specialisation on the longest K length (or local window) --
   one row in batches whose longest context differs by 500x;
2. tiling that follows storage metadata -- the same keys behind page tables
   of different widths and under different physical placements;
3. different prefill and decode attention algorithms -- a position computed
   inside a long prefill chunk, as a decode row, in a short chunk and at the
   start of a chunk;
4. query partitions that visit fully masked tiles and replace their -inf
   maximum by 0 -- rows of one request split across chunk boundaries and
   query tiles under a sliding window, where early key tiles of a split are
   fully masked for some rows and not for others (that this change of rule
   does move bits is shown on the CPU by `test_failure_source_model.py`).

The host compacts every page table to the pages a request needs, so the
page-table width that reaches the kernel is the batch's widest request:
test 2 varies it through the co-scheduled requests as well as through the
caller's table width.

The first failure source's reduction-strategy half (split-K) is shown to be
detectable by `test_llm42_gpu.py::test_a_changed_reduction_strategy_is_visible_in_the_bits`.
"""

import numpy as np
import pytest

from attn_scenario import SPECS, Scenario
from gpu_util import bits, ready

pytestmark = pytest.mark.gpu


def _same_rows(results, key_filter=None):
    """results: list of {(r, pos): row}; every key seen twice must have equal bits."""
    seen, n = {}, 0
    for i, res in enumerate(results):
        for k, row in res.items():
            if key_filter is not None and not key_filter(k):
                continue
            b = bits(row)
            if k in seen:
                np.testing.assert_array_equal(b, seen[k][1], err_msg=f"row {k}: run {i} vs run {seen[k][0]}")
                n += 1
            else:
                seen[k] = (i, b)
    return n


@pytest.mark.parametrize("window", [0, 128])
def test_1_longest_context_in_the_batch_does_not_change_a_row(window):
    ready()
    spec = SPECS[128] if window == 0 else SPECS[128].with_(sliding_window=window, local_global_period=1000)
    lens = [300, 8000, 17] + [1000 + 37 * i for i in range(40)]
    sc = Scenario(spec, lens, num_pages=sum((n + 15) // 16 for n in lens) + 8, seed=21)
    probe = [(0, 299, 1), (0, 200, 3)]  # a decode row and a short chunk of request 0
    runs = [
        probe,                                                   # alone: longest K 300
        probe + [(2, 16, 1)],                                    # with a 17-key request
        probe + [(1, 7999, 1)],                                  # with an 8000-key request
        probe + [(1, 7999, 1)] + [(r, lens[r] - 1, 1) for r in range(3, 43)],  # 43 requests
        [(1, 7000, 64)] + probe + [(2, 0, 17)],                  # next to prefill chunks
    ]
    assert _same_rows([sc.run(p) for p in runs]) >= 4 * 4


def test_2_page_table_width_and_placement_do_not_change_a_row():
    ready()
    lens = [300, 1200, 40]
    sc = Scenario(SPECS[128], lens, num_pages=200, seed=22)
    t0 = sc.tables[0]  # 19 pages
    spare = np.arange(150, 200, dtype=np.int32)  # valid page ids past the request's keys
    padded = {0: np.concatenate([t0, spare[:21]])}
    wide = {0: np.concatenate([t0, spare, spare])}
    parts = [(0, 299, 1), (0, 250, 20)]
    runs = [sc.run(parts), sc.run(parts, tables=padded), sc.run(parts, tables=wide),
            sc.run(parts + [(1, 1199, 1)]),                        # batch page-table width set by request 1
            sc.run(parts + [(1, 1199, 1)], tables=wide)]
    sc.place(np.roll(np.arange(200), 77).astype(np.int32))          # new physical placement, same keys
    runs += [sc.run(parts), sc.run(parts + [(2, 39, 1)], tables={0: np.concatenate([sc.tables[0], spare[:5]])})]
    assert _same_rows(runs) >= 6 * 21


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_3_prefill_and_decode_compute_a_position_alike(hd):
    ready()
    lens = [1600, 900]
    sc = Scenario(SPECS[hd], lens, num_pages=200, seed=23 + hd)
    positions = [0, 15, 16, 31, 32, 511, 512, 513, 1023, 1024, 1500, 1599]
    runs = [sc.run([(0, 0, 1600)]),                                  # one prefill chunk (prefill-class CTAs)
            sc.run([(0, p, 1) for p in positions]),                  # decode rows (decode-class CTAs)
            sc.run([(0, 0, 700), (0, 700, 900)])]                    # two chunks of the same request in one step
    # (a step never writes one KV slot twice, so overlapping chunks go to separate steps)
    runs += [sc.run([(0, p, 3)]) for p in positions if p + 3 <= 1600]                 # short chunks
    runs += [sc.run([(0, p, 64), (1, 0, 900)]) for p in positions if p + 64 <= 1600]  # chunks starting at p
    assert _same_rows(runs, key_filter=lambda k: k[0] == 0 and k[1] in positions) >= 3 * len(positions)


@pytest.mark.parametrize("window", [37, 100, 512])
def test_4_fully_masked_key_tiles_leave_rows_unchanged(window):
    ready()
    spec = SPECS[128].with_(sliding_window=window, local_global_period=1000)
    lens = [1100]
    sc = Scenario(spec, lens, num_pages=80, seed=24)
    runs = [sc.run([(0, 0, 1100)]),
            sc.run([(0, 0, 37), (0, 37, 1063)]),                      # chunk boundary inside a key tile
            sc.run([(0, 0, 250), (0, 250, 1), (0, 251, 849)]),
            sc.run([(0, 5, 40), (0, 600, 21), (0, 1099, 1)]),         # chunks starting mid-tile
            sc.run([(0, p, 1) for p in range(600, 640)] + [(0, 100, 3), (0, 511, 2)]),
            sc.run([(0, 900, 200)])]
    assert _same_rows(runs) >= 1100
