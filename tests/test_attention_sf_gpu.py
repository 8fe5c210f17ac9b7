"""The scores-first decode CTA against the tile-at-a-time decode CTA.

A decode launch of at most one CTA per SM (a few requests) runs the
scores-first CTA at head dims 64 and 128: its warps score a split's tiles
first, then fold P V in rounds.  A launch with more CTAs than SMs runs the
2-warp tile-at-a-time CTA.  Both take every row through the same per-tile
steps of the unified traversal (深入解析 Vosti §六 6.2), so each request's
rows computed alone must equal, bit for bit, the same rows computed inside
a batch large enough to take the other kernel: blocks of 4, 8, 12 and 16
rows, splits with all 16 key tiles and ragged last or (under a window)
first splits, GQA groups of 4 and 8 query heads per KV head.
"""

import numpy as np
import pytest
import torch

from attn_scenario import Scenario, check_parity
from gpu_util import bits, ready
from invariant_vd_step_gb300 import synth

pytestmark = pytest.mark.gpu

SPLIT = 512


def _items(parts, hkv, group):
    """CTAs of one decode-class launch: (KV splits of the row block) x KV heads, one row block each."""
    n = 0
    for _, cached, ql in parts:
        assert ql * group <= 16
        n += ((cached + ql - 1) // SPLIT + 1) * hkv
    return n


def _alone_equals_batched(sc, parts, window=0):
    spec = sc.spec
    hkv, group = spec.n_kv_heads, spec.n_heads // spec.n_kv_heads
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert _items(parts, hkv, group) > sms, "the batched launch must have more CTAs than SMs"
    batched = sc.run(parts)
    for part in parts:
        assert _items([part], hkv, group) <= sms
        alone = sc.run([part])
        for k, row in alone.items():
            np.testing.assert_array_equal(bits(row), bits(batched[k]), err_msg=f"row {k}")
    check_parity(sc, batched, window=window)


def _parts(lens, qlens):
    # the last q_len positions of each request (a decode step, or a short chunk after cached context)
    return [(r, n - ql, ql) for r, (n, ql) in enumerate(zip(lens, qlens))]


@pytest.mark.parametrize("hd", [64, 128])
def test_sf_rows_equal_tile_at_a_time_rows(hd):
    ready()
    spec = synth.ModelSpec(f"sf{hd}", 1, 256, 32, 8, hd, 256, 256)  # G = 4
    # contexts ending inside a split (ragged last split) and on a split edge (all splits full)
    lens = [2048, 1900, 1537, 1536, 1100, 1024, 700, 513]
    qlens = [1, 3, 4, 1, 2, 4, 1, 3]  # 4, 12, 16, 4, 8, 16, 4, 12 rows per CTA
    sc = Scenario(spec, lens, num_pages=sum((n + 15) // 16 for n in lens) + 8, seed=61 + hd)
    _alone_equals_batched(sc, _parts(lens, qlens))


def test_sf_group_of_8():
    ready()
    spec = synth.ModelSpec("sf128g8", 1, 256, 64, 8, 128, 256, 256)  # G = 8
    lens = [2000, 1600, 1030, 900, 515, 1800, 1200]
    qlens = [1, 2, 1, 2, 1, 1, 2]  # 8 or 16 rows per CTA
    sc = Scenario(spec, lens, num_pages=sum((n + 15) // 16 for n in lens) + 8, seed=67)
    _alone_equals_batched(sc, _parts(lens, qlens))


def test_sf_sliding_window():
    ready()
    # a window of 700 keys: the first split a row sees starts inside it
    spec = synth.ModelSpec("sf128w", 1, 256, 32, 8, 128, 256, 256).with_(sliding_window=700,
                                                                         local_global_period=1000)
    lens = [2100, 1800, 1300, 1250, 900, 2050]
    qlens = [1, 4, 3, 1, 2, 1]
    sc = Scenario(spec, lens, num_pages=sum((n + 15) // 16 for n in lens) + 8, seed=71)
    _alone_equals_batched(sc, _parts(lens, qlens), window=700)
