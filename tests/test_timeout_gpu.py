"""Failure detection on the device, without a fault: a bounded wait that
nothing completes gives up, reports VD_ERR_TIMEOUT through the model's
status word, the step kernels skip their work while it is set, and after
the host reads (and so clears) it the next step is correct again.

The wait is vd_op_wait_probe's: an mbarrier that no thread arrives at,
waited on with the same bounded-wait routines the pipelined GEMM and
attention kernels use (the waiting call, whose first timeout stops the
other waiter through the CTA's abort flag, and the teardown wait).  Nothing
is in flight, so nothing can fault, trap or hang.
"""

import numpy as np
import pytest
import torch

from gpu_util import bits, ready
from invariant_vd_step_gb300 import synth, vd

pytestmark = pytest.mark.gpu


def _model():
    spec = synth.TINY
    W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=3, gain_std=0.1).items()}
    model = vd.Model(spec, W, max_tokens=64, max_seqs=4, max_logit_rows=8, max_context=256)
    pool = vd.KVPool(model, 16)
    toks = synth.make_tokens(24, spec.vocab, seed=5)
    batch = vd.StepBatch([(toks, 0, np.array([3, 9], np.int32))], logit_rows=[23])
    return spec, W, model, pool, batch


def test_a_wait_that_runs_out_reports_a_timeout_and_the_model_recovers():
    ready()
    spec, W, model, pool, batch = _model()
    ref = torch.empty((1, spec.vocab), device="cuda")
    model.step(pool, batch, ref)
    torch.cuda.synchronize()
    assert model.device_status() == 0

    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    model.wait_probe(50_000, out)  # 50 ms limit
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    # the first waiter gives up after the limit, the second through the abort
    # flag (or its own limit), then the teardown wait after the limit again
    assert out[:3].tolist() == [1, 1, 1]
    assert 90.0 <= ms < 2000.0, ms

    # while the timeout is recorded, a step's kernels skip their work
    skipped = torch.full((1, spec.vocab), float("nan"), device="cuda")
    model.step(pool, batch, skipped)
    torch.cuda.synchronize()
    assert torch.isnan(skipped).all()

    assert model.device_status() == vd.VD_ERR_TIMEOUT  # read ...
    assert model.device_status() == 0                  # ... and cleared

    again = torch.empty_like(ref)
    model.step(pool, batch, again)  # the same step, rewriting its own K/V slots
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(again), bits(ref))
    assert model.device_status() == 0


def test_wait_probe_rejects_bad_limits():
    ready()
    _, _, model, _, _ = _model()
    for bad in (0, -5, 2_000_001):
        with pytest.raises(vd.VDError) as e:
            model.wait_probe(bad)
        assert e.value.code == vd.VD_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert model.device_status() == 0
