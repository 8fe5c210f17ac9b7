"""The tcgen05 prefill attention kernel against the mma.sync one and the oracle.

Prefill-class rows (q_len * Hq/Hkv > 16) run on tcgen05 by default for head
dims 64, 128 and 256 (128 rows per CTA, accumulators in tensor memory) and on
mma.sync when asked (64 rows per CTA).  Both take the per-row steps of the
unified traversal (深入解析 Vosti §六 6.2) in the same order, and a tcgen05
K = 16 step computes what an mma.sync m16n8k16 step computes, so every row
must come out bit for bit the same under either kernel: full prefills,
chunks after cached context, short chunks just above the decode class,
row blocks with ragged tails, sliding windows, groups of 1, 4 and 8 query
heads per KV head, and rows crossing split boundaries.
"""

import numpy as np
import pytest

from attn_scenario import SPECS, Scenario, check_parity
from gpu_util import bits, ready
from invariant_vd_step_gb300 import synth, vd

pytestmark = pytest.mark.gpu


def _both(sc, parts):
    sc.model.set_attention_prefill(0)
    tc = sc.run(parts)
    sc.model.set_attention_prefill(1)
    ms = sc.run(parts)
    sc.model.set_attention_prefill(0)
    assert tc.keys() == ms.keys()
    for k in tc:
        np.testing.assert_array_equal(bits(tc[k]), bits(ms[k]), err_msg=f"row {k} in {parts}")
    return tc


SCHEDULES = [
    [(0, 0, 1100)],                              # one long prefill: splits 0..2, a ragged last row block
    [(1, 0, 300), (2, 0, 77), (3, 0, 5)],        # several requests; 5 tokens x G rows: one short block
    [(0, 700, 400), (1, 290, 10)],               # chunks after cached context (not tile aligned)
    [(0, 500, 30), (2, 60, 17), (3, 1, 4)],      # chunks across the first split edge
    [(1, 31, 33), (0, 1023, 77)],                # starting one key before a tile / split edge
]


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_tc_equals_mma_sync_bitwise_and_matches_oracle(hd):
    ready()
    lens = [1100, 300, 77, 5]
    sc = Scenario(SPECS[hd], lens, num_pages=200, seed=31 + hd)
    for parts in SCHEDULES:
        res = _both(sc, parts)
        check_parity(sc, res)


@pytest.mark.parametrize("hd", [128, 256])
def test_tc_sliding_window(hd):
    ready()
    spec = SPECS[hd].with_(sliding_window=100, local_global_period=1000)
    lens = [700, 101, 40]
    sc = Scenario(spec, lens, num_pages=120, seed=41)
    for parts in ([(0, 0, 700)], [(0, 600, 100), (1, 0, 101), (2, 0, 40)], [(0, 150, 9)]):
        res = _both(sc, parts)
        check_parity(sc, res, window=100)


@pytest.mark.parametrize("heads", [(8, 8), (8, 1)], ids=["G1", "G8"])
def test_tc_query_group_sizes(heads):
    ready()
    hq, hkv = heads
    spec = synth.ModelSpec(f"att128g{hq // hkv}", 1, 256, hq, hkv, 128, 256, 256)
    lens = [600, 129, 33]
    sc = Scenario(spec, lens, num_pages=120, seed=43 + hq // hkv)
    for parts in ([(0, 0, 600), (1, 0, 129)], [(0, 500, 100), (2, 0, 33)], [(1, 100, 29), (2, 16, 17)]):
        res = _both(sc, parts)
        check_parity(sc, res)


def test_tc_rows_equal_decode_rows():
    # the causal contract across kernels: rows of a tcgen05 prefill equal the
    # same rows computed one at a time by the mma.sync decode kernel
    ready()
    lens = [1030, 200]
    sc = Scenario(SPECS[128], lens, num_pages=120, seed=47)
    full = sc.run([(0, 0, 1030), (1, 0, 200)])
    for r, p in [(0, 0), (0, 31), (0, 32), (0, 511), (0, 512), (0, 1029), (1, 127), (1, 128), (1, 199)]:
        one = sc.run([(r, p, 1)])
        np.testing.assert_array_equal(bits(one[(r, p)]), bits(full[(r, p)]), err_msg=f"row {(r, p)}")


def test_prefill_kernel_choice_is_validated():
    ready()
    sc = Scenario(SPECS[128], [40], num_pages=8, seed=49)
    for bad in (-1, 2, 7):
        with pytest.raises(vd.VDError):
            sc.model.set_attention_prefill(bad)
    sc.model.set_attention_prefill(1)
    sc.model.set_attention_prefill(0)
