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


def _setup(spec=None):
    spec = spec or synth.ModelSpec("noalloc128", 1, 256, 8, 2, 128, 256, 256)
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


def _tables(lens, seed):
    perm = synth.page_permutation(300, seed=seed)
    tables, k = [], 0
    for n in lens:
        npg = (n + 15) // 16
        tables.append(perm[k:k + npg])
        k += npg
    return tables


# hd 64 / 128 / 256; a layer with a 64-key window (layer 0 of a 1:1 local /
# global model) next to a global one; decode calls in fold mode (one CTA
# folds every split of its rows) as well as split mode
WINDOWED = synth.ModelSpec("noalloc-window", 2, 256, 4, 2, 256, 256, 256, sliding_window=64,
                           local_global_period=2, rope_theta_local=1e4)
HD64 = synth.ModelSpec("noalloc64", 1, 256, 4, 2, 64, 256, 256)


@pytest.mark.parametrize("spec", [HD64, WINDOWED], ids=lambda s: s.name)
@pytest.mark.parametrize("fold", [0, 1])
def test_static_scratch_matches_workspace_windows_fold_and_head_dims(spec, fold):
    ready()
    spec, model, pool = _setup(spec)
    model.set_attention_fold(fold)
    calls = [([1500, 700, 2048, 65], [1, 1, 1, 1]), ([1100, 300], [40, 300])]
    for layer in range(spec.n_layers):
        for ci, (lens, qlens) in enumerate(calls):
            b, q = _batch(spec, lens, qlens, _tables(lens, 10 + ci))
            ref = torch.full_like(q, float("nan"))
            got = torch.full_like(q, float("nan"))
            model.attention(pool, layer, b, q, ref)
            model.attention_static(pool, layer, b, q, got)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(bits(got), bits(ref), err_msg=f"layer {layer} call {ci}")
            assert not torch.isnan(got.float()).any()
    assert model.device_status() == 0


def test_static_scratch_calls_allocate_no_device_memory():
    ready()
    spec, model, pool = _setup()
    lens, qlens = [900, 1700, 40], [1, 1, 1]
    b, q = _batch(spec, lens, qlens, _tables(lens, 20))
    out = torch.empty_like(q)
    model.attention_static(pool, 0, b, q, out)  # first call on the device: module and symbol lookup
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(5):
        model.attention_static(pool, 0, b, q, out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_static_and_workspace_entries_reject_bad_batches_alike():
    ready()
    spec, model, pool = _setup()
    q = torch.zeros((4, spec.n_heads, spec.head_dim), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    bad = [
        vd.StepBatch([(np.zeros(1, np.int32), 5000, np.arange(300, dtype=np.int32))]),  # past max_context
        vd.StepBatch([(np.zeros(2, np.int32), 10, np.array([400], np.int32))]),        # page id out of range
        vd.StepBatch([(np.zeros(2, np.int32), 40, np.array([1], np.int32))]),          # page table too narrow
        vd.StepBatch([(np.zeros(1, np.int32), 0, np.array([1], np.int32)),
                      (np.zeros(1, np.int32), 0, np.array([1], np.int32))]),          # two writers of one slot
    ]
    for i, b in enumerate(bad):
        codes = []
        for call in (model.attention, model.attention_static):
            with pytest.raises(vd.VDError) as e:
                call(pool, 0, b, q, out)
            codes.append(e.value.code)
        assert codes[0] == codes[1], (i, codes)
    torch.cuda.synchronize()
    assert model.device_status() == 0
