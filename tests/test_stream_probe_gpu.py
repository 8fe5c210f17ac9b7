"""The measurement ops.  The weight-stream op (vd_op_tma_stream) runs every
copy shape the GEMM plans use, with and without activation copies and K
parts, leaves the device status clean, and rejects shapes the GEMM cannot
take.  The MMA-issue op (vd_op_mma_issue_probe) completes every MMA it
issues, reports plausible cycle counts, and rejects shapes it cannot take."""

import pytest
import torch

from gpu_util import ready
from invariant_vd_step_gb300 import synth, vd

pytestmark = pytest.mark.gpu


def test_stream_runs_every_plan_copy_shape():
    ready()
    W = synth.make_normal_bf16((512, 1024), seed=1).cuda()
    X = synth.make_normal_bf16((256, 1024), seed=2).cuda()
    for bm, kpo in ((64, 1), (64, 4), (128, 2), (128, 4), (256, 1)):
        for xr in (0, 1, 16, 256):
            if 2 * kpo * (bm * 128 + (xr * 128 + 1023) // 1024 * 1024) > 200 * 1024:
                continue  # the GEMM halves kpo for such a plan; the op streams the copies it is given
            for kp in (1, 2):
                vd.tma_stream(W, bm, kpo, X if xr else None, xr, k_parts=kp)
    torch.cuda.synchronize()
    # the ops' status word is checked through a GEMM that must still run in full
    C = torch.full((3, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    vd.gemm(X[:3].contiguous(), W[:128].contiguous(), C)
    torch.cuda.synchronize()
    assert not torch.isnan(C.float()).any()


def test_stream_rejects_shapes_no_plan_has():
    ready()
    W = synth.make_normal_bf16((192, 1024), seed=1).cuda()
    for bm, kpo, kp in ((128, 2, 1), (96, 1, 1), (64, 3, 1), (256, 2, 1), (64, 4, 5)):
        with pytest.raises(vd.VDError) as e:
            vd.tma_stream(W, bm, kpo, k_parts=kp)
        assert e.value.code == vd.VD_ERR_INVALID_ARG


def test_mma_issue_probe_runs_and_reports_cycles():
    ready()
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    for M in (64, 128):
        for N in (16, 64, 256):
            for wait in (0, 1, 2, 3):
                out.fill_(0)
                vd.mma_issue_probe(M, N, 160, wait, out)
                torch.cuda.synchronize()
                issue, done = out.cpu().tolist()
                # every MMA completed (no timeout); at least a few cycles each, far below a microsecond
                assert 0 < issue <= done < 160 * 5000, (M, N, wait, issue, done)


def test_mma_issue_probe_rejects_shapes_it_cannot_take():
    ready()
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    for bad in [(32, 16, 16, 0), (128, 8, 16, 0), (128, 272, 16, 0), (128, 16, 15, 0), (128, 16, 0, 0),
                (128, 16, 16, 4)]:
        with pytest.raises(vd.VDError):
            vd.mma_issue_probe(*bad, out)
