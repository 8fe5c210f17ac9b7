"""The no-allocation attention entry point (vd_op_attention_static).

Some hosts cannot let a library allocate device memory during a call: the
host may own all device memory through its own pool, or cannot tolerate the
device-wide synchronisation cudaMalloc/cudaFree can cause.  For them the
attention op has a variant whose split scratch is a fixed array inside
libvd.so.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes alone.
"""

import numpy as np
import pytest
import torch

from gpu_util import bits, ready
from invariant_vd_step_gb300 import synth, vd

pytestmark = pytest.mark.gpu


def _setup():
    spec = synth.ModelSpec("noalloc128", 1, 256, 8, 2, 128, 256, 256)
    W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=1).items()}
    model = vd.Model(spec, W, max_tokens=2048, max_seqs=16, max_logit_rows=8, max_context=4096)
    pool = vd.KVPool(model, 300, memory=torch.zeros(model.pool_bytes(300), dtype=torch.uint8, device="cuda"))
    view = pool.view()
    view.copy_(synth.make_normal_bf16(tuple(view.shape), seed=2).cuda())  # seeded K/V in every slot
    return spec, model, pool


def _batch(spec, lens, qlens, tables):
    seqs = [(np.zeros(q, np.int32), n - q, t) for n, q, t in zip(lens, qlens, tables)]
    T = sum(qlens)
    q = synth.make_normal_bf16((T, spec.n_heads, spec.head_dim), seed=sum(lens)).cuda()
    return vd.StepBatch(seqs), q


def test_static_scratch_attention_matches_workspace_attention_twice_in_a_row():
    ready()
    spec, model, pool = _setup()
    perm = synth.page_permutation(300, seed=3)
    calls = [  # two different calls in a row: decode rows, then prefill chunks over longer contexts
        ([700, 1500, 33, 2048], [1, 1, 1, 1]),
        ([1030, 600, 90], [300, 17, 90]),
    ]
    for lens, qlens in calls:
        tables, k = [], 0
        for n in lens:
            npg = (n + 15) // 16
            tables.append(perm[k:k + npg])
            k += npg
        b, q = _batch(spec, lens, qlens, tables)
        ref = torch.full_like(q, float("nan"))
        got = torch.full_like(q, float("nan"))
        model.attention(pool, 0, b, q, ref)               # workspace scratch
        model.attention_static(pool, 0, b, q, got)        # static scratch
        torch.cuda.synchronize()
        # GPU-vs-GPU comparisons of the same rows use a tolerance of 0 ulp
        np.testing.assert_array_equal(bits(got), bits(ref))
        assert not torch.isnan(got.float()).any()
    assert model.device_status() == 0


def test_static_scratch_rejects_calls_larger_than_the_array():
    ready()
    spec, model, pool = _setup()
    # 2048 prefill rows over 4 splits: 2048 * 8 * 4 * 130 * 4 bytes > 16 MiB
    lens, qlens = [2048], [2048]
    b, q = _batch(spec, lens, qlens, [np.arange(128, dtype=np.int32)])
    out = torch.empty_like(q)
    with pytest.raises(vd.VDError) as e:
        model.attention_static(pool, 0, b, q, out)
    assert e.value.code == 4 and "static buffer" in str(e.value)
