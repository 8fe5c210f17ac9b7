"""GEMM launch shapes change speed, never bits.

The tile of a GEMM launch -- weight rows per tile (64 or 128, the MMA's M,
or 256 as two M = 128 instructions sharing each activation block),
tokens per tile (16 .. 256, the MMA's N) and 64-wide K blocks per weight copy
(1, 2, 4) -- is chosen per launch.  Every output element stays one chain of
K = 16 MMA steps in ascending K order into a zeroed accumulator, so the
matmul contract of 深入解析 Vosti §六 6.1 (row x of a batched run equals the
singleton run bit for bit) holds whatever shape a launch takes, provided the
tensor cores compute an element the same way at every M and N.  These tests
force every shape and require identical bits: single GEMMs with every
epilogue, token counts inside one token tile, across several and with ragged
tails, and whole decoder steps (Llama- and Gemma-style blocks) whose logits
must not move by a bit under any forced shape.
"""

import numpy as np
import pytest
import torch

from gpu_util import bits, ready
from invariant_vd_step_gb300 import synth, vd

pytestmark = pytest.mark.gpu

PLANS = [(bm, bn, kpo) for bm in (128, 64, 256) for bn in (16, 32, 64, 128, 256) for kpo in (1, 2, 4)]


@pytest.fixture(autouse=True)
def _default_plan_after():
    yield
    vd.set_gemm_plan(0, 0, 0)


def _run(A, W, N, epi, residual=None):
    dt = torch.float32 if epi == vd.EPI_F32 else torch.bfloat16
    C = torch.full((A.shape[0], N), float("nan"), dtype=dt, device="cuda")
    vd.gemm(A, W, C, epi, residual)
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("epi", [vd.EPI_BF16, vd.EPI_F32, vd.EPI_RESIDUAL, vd.EPI_SWIGLU, vd.EPI_GEGLU])
def test_every_plan_gives_the_same_bits(epi):
    ready()
    K = 512  # 8 K blocks: every kpo divides them
    glu = epi in (vd.EPI_SWIGLU, vd.EPI_GEGLU)
    N = 128 if glu else 256  # GLU: F = 128 features, 256 weight rows
    W = synth.make_normal_bf16((2 * N if glu else N, K), seed=51, std=0.05).cuda()
    for T in (1, 7, 16, 33, 100, 300):
        A = synth.make_normal_bf16((T, K), seed=50 + T).cuda()
        R = synth.make_normal_bf16((T, N), seed=52).cuda() if epi == vd.EPI_RESIDUAL else None
        vd.set_gemm_plan(0, 0, 0)
        ref = bits(_run(A, W, N, epi, R))
        for plan in PLANS:
            vd.set_gemm_plan(*plan)
            np.testing.assert_array_equal(bits(_run(A, W, N, epi, R)), ref, err_msg=f"T={T} plan={plan}")


def test_row_equals_singleton_under_small_token_tiles():
    # The relational contract with 16-token tiles and 64-row weight tiles:
    # a row's position inside a tile and the tile's shape move no bit.
    ready()
    K, N = 1024, 384
    A = synth.make_normal_bf16((300, K), seed=60).cuda()
    W = synth.make_normal_bf16((N, K), seed=61, std=0.05).cuda()
    vd.set_gemm_plan(0, 0, 0)
    single = {x: bits(_run(A[x:x + 1].contiguous(), W, N, vd.EPI_BF16))[0] for x in (0, 15, 16, 150, 299)}
    for plan in [(64, 16, 4), (128, 16, 2), (64, 64, 1), (128, 256, 4), (256, 256, 1), (256, 32, 1)]:
        vd.set_gemm_plan(*plan)
        C = bits(_run(A, W, N, vd.EPI_BF16))
        for x, row in single.items():
            np.testing.assert_array_equal(C[x], row, err_msg=f"plan={plan} x={x}")


def test_plan_validation():
    ready()
    for bad in [(32, 0, 0), (0, 48, 0), (0, 512, 0), (0, 0, 3), (-1, 0, 0)]:
        with pytest.raises(vd.VDError):
            vd.set_gemm_plan(*bad)


GEMMA_TINY = synth.ModelSpec("gemma-tiny", 3, 256, 2, 1, 256, 512, 512, act="geglu", qk_norm=True,
                             rope_theta=1e6, rope_theta_local=1e4, sliding_window=24, local_global_period=2,
                             rms_eps=1e-6, embed_scale=True, norm_offset=True, sandwich_norm=True)


@pytest.mark.parametrize("spec", [synth.TINY, GEMMA_TINY], ids=lambda s: s.name)
@pytest.mark.parametrize("sample", [False, True])
def test_step_logits_do_not_move_under_any_forced_plan(spec, sample):
    """A mixed step (one prefill chunk, decode rows, a short chunk) and a
    pure decode step, with and without the fused token choice in the LM head
    (which takes no 64-row weight tiles), under forced shapes."""
    ready()
    W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=4, gain_std=0.1).items()}
    m = vd.Model(spec, W, max_tokens=320, max_seqs=16, max_logit_rows=64, max_context=512)
    pool = vd.KVPool(m, 128)
    hist = [synth.make_tokens(90, spec.vocab, seed=70 + r) for r in range(6)]
    pages = {r: np.arange(16 * r, 16 * r + 16, dtype=np.int32) for r in range(6)}

    def steps():
        out = []
        # prefill 60 tokens of requests 0..4 first (cached context for decode rows)
        b0 = vd.StepBatch([(hist[r][:60], 0, pages[r]) for r in range(5)], logit_rows=[59, 119, 179, 239, 299])
        mixed = vd.StepBatch([(hist[r][60:61], 60, pages[r]) for r in range(4)] +
                             [(hist[4][60:67], 60, pages[4]), (hist[5][:48], 0, pages[5])],
                             logit_rows=[0, 1, 2, 3, 4, 7, 10, 57])
        decode = vd.StepBatch([(hist[r][61:62], 61, pages[r]) for r in range(4)], logit_rows=[0, 1, 2, 3])
        for b in (b0, mixed, decode):
            R = len(b.logit_rows)
            lg = torch.full((R, spec.vocab), float("nan"), device="cuda")
            if sample:
                tok = torch.empty(R, dtype=torch.int32, device="cuda")
                m.step_sample(pool, b, [(3, i, 0.7 if i % 2 else 0.0) for i in range(R)], lg, tok)
                torch.cuda.synchronize()
                out.append((bits(lg), tok.cpu().numpy()))
            else:
                m.step(pool, b, lg)
                torch.cuda.synchronize()
                out.append((bits(lg), None))
        return out

    vd.set_gemm_plan(0, 0, 0)
    ref = steps()
    for plan in [(64, 16, 4), (128, 16, 1), (64, 32, 2), (128, 64, 4), (64, 128, 1), (128, 256, 2),
                 (256, 256, 1), (256, 64, 1)]:
        vd.set_gemm_plan(*plan)
        got = steps()
        for i, ((lb, tb), (rb, rt)) in enumerate(zip(got, ref)):
            np.testing.assert_array_equal(lb, rb, err_msg=f"plan={plan} step={i}")
            if sample:
                np.testing.assert_array_equal(tb, rt, err_msg=f"plan={plan} step={i} tokens")
    assert m.device_status() == 0


def test_model_creation_checks_the_tile_shapes():
    """vd_create_model compares every GEMM tile shape bit for bit on seeded
    operands once per device; on this GPU they agree, so shapes stay chosen
    per launch (the check would otherwise pin one fixed shape)."""
    ready()
    spec = synth.TINY
    W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=1).items()}
    model = vd.Model(spec, W, max_tokens=32, max_seqs=2, max_logit_rows=2, max_context=64)
    assert vd.gemm_shape_check() == 1
    assert vd.gemm_plan(1, 4096, 4096) != vd.gemm_plan(256, 4096, 4096)  # still chosen per launch
    model.close()
