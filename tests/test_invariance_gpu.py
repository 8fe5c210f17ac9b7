"""The execution-variation matrix on the GPU: 3,200 bitwise row comparisons."""

import pytest

from gpu_util import ready
from invariant_vd_step_gb300 import invariance

pytestmark = pytest.mark.gpu


def test_matrix_is_all_bitwise_equal():
    ready()
    r = invariance.run_matrix()
    assert r.pairs == 3200, r
    assert r.runs == 25
    assert r.prefix_hit_pages > 0 and (r.evicted > 0 or r.preempted > 0), r
    assert r.equal == r.pairs, r.categories
