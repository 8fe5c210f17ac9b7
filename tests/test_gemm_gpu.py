"""tcgen05 GEMM: parity with the oracle and the matmul relational contract."""

import numpy as np
import pytest
import torch

from gpu_util import bf16_ulp_dist, bits, f64, ready
from invariant_vd_step_gb300 import synth, vd
from oracle.bf16 import round_bf16
from oracle.decoder import gelu_tanh, silu

pytestmark = pytest.mark.gpu


def _run(A, W, N, epi=vd.EPI_BF16, residual=None):
    dt = torch.float32 if epi == vd.EPI_F32 else torch.bfloat16
    C = torch.full((A.shape[0], N), float("nan"), dtype=dt, device="cuda")
    vd.gemm(A, W, C, epi, residual)
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("T,N,K", [(1, 128, 64), (5, 256, 512), (130, 384, 256), (257, 128, 1024), (64, 640, 4096)])
def test_bf16_and_f32_epilogues_vs_oracle(T, N, K):
    ready()
    A = synth.make_normal_bf16((T, K), seed=10 + T).cuda()
    W = synth.make_normal_bf16((N, K), seed=11 + N, std=0.05).cuda()
    exact = f64(A) @ f64(W).T
    # fp32 accumulation error bound (K terms, <= 2 ulp per addition), then one bf16 rounding
    acc_bound = K * 2.0 ** -23 * (np.abs(f64(A)) @ np.abs(f64(W)).T)
    c16 = f64(_run(A, W, N))
    assert np.all(np.abs(c16 - exact) <= 2.0 ** -8 * np.abs(exact) + acc_bound)
    assert np.mean(bf16_ulp_dist(c16, round_bf16(exact)) <= 1) >= 0.99
    c32 = f64(_run(A, W, N, vd.EPI_F32))
    assert np.all(np.abs(c32 - exact) <= acc_bound)


def test_small_integers_are_exact():
    ready()
    T, N, K = 37, 256, 1024
    A = synth.make_small_int_bf16((T, K), seed=3).cuda()
    W = synth.make_small_int_bf16((N, K), seed=4).cuda()
    exact = (f64(A) @ f64(W).T)
    np.testing.assert_array_equal(f64(_run(A, W, N, vd.EPI_F32)), exact)


def test_matmul_contract_row_equals_singleton_bitwise():
    # Row x of a batched run == the singleton run of that row, for many M
    # and row positions inside and across 128-token tiles.
    ready()
    K, N = 512, 256
    A = synth.make_normal_bf16((1000, K), seed=20).cuda()
    W = synth.make_normal_bf16((N, K), seed=21, std=0.05).cuda()
    single = {}
    for M in (1, 2, 3, 7, 64, 127, 128, 129, 256, 1000):
        C = _run(A[:M].contiguous(), W, N)
        for x in sorted({0, M // 2, M - 1, min(M - 1, 63), min(M - 1, 127), min(M - 1, 128)}):
            if x not in single:
                single[x] = bits(_run(A[x:x + 1].contiguous(), W, N))[0]
            np.testing.assert_array_equal(bits(C)[x], single[x], err_msg=f"M={M} x={x}")
    # the same row placed at another position of another batch
    perm = torch.randperm(300, generator=torch.Generator().manual_seed(5))
    Ap = A[:300][perm].contiguous()
    Cp = bits(_run(Ap, W, N))
    Cr = bits(_run(A[:300].contiguous(), W, N))
    np.testing.assert_array_equal(Cp, Cr[perm.numpy()])


def test_residual_epilogue_vs_oracle_and_in_place():
    ready()
    T, N, K = 70, 256, 512
    A = synth.make_normal_bf16((T, K), seed=30).cuda()
    W = synth.make_normal_bf16((N, K), seed=31, std=0.05).cuda()
    R = synth.make_normal_bf16((T, N), seed=32).cuda()
    acc = f64(A) @ f64(W).T
    ref = round_bf16(round_bf16(acc) + f64(R))
    out = f64(_run(A, W, N, vd.EPI_RESIDUAL, R))
    # one bf16 ulp of acc on either side, plus one ulp of the sum
    assert np.all(np.abs(out - ref) <= 2.0 ** -6 * (np.abs(acc) + np.abs(f64(R))) + 1e-30)
    X = R.clone()
    vd.gemm(A, W, X, vd.EPI_RESIDUAL, X)  # residual aliases the output
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(X), bits(_run(A, W, N, vd.EPI_RESIDUAL, R)))


@pytest.mark.parametrize("plan", [(0, 0, 0), (64, 16, 4), (64, 32, 4), (128, 64, 2), (128, 128, 2), (256, 64, 1)])
def test_bf16_and_residual_epilogues_round_the_f32_accumulator(plan):
    # The bf16 epilogues take the same fp32 accumulator as the f32 one: C = bf16(acc) and
    # C = bf16(bf16(acc) + R), each element rounded once to nearest even.  Pinned bit for bit
    # against the f32 epilogue's output rounded here, for token counts inside one 32-token chunk,
    # across several and with ragged tails, at 64-, 128- and 256-row tiles.
    ready()
    N, K = 512, 256
    W = synth.make_normal_bf16((N, K), seed=61, std=0.05).cuda()
    vd.set_gemm_plan(*plan)
    try:
        for T in (1, 3, 8, 31, 33, 64, 100, 257):
            A = synth.make_normal_bf16((T, K), seed=60 + T).cuda()
            R = synth.make_normal_bf16((T, N), seed=62 + T).cuda()
            acc = _run(A, W, N, vd.EPI_F32).cpu()
            want_bf16 = acc.to(torch.bfloat16)
            want_res = (want_bf16.float() + R.cpu().float()).to(torch.bfloat16)
            np.testing.assert_array_equal(bits(_run(A, W, N, vd.EPI_BF16)), bits(want_bf16), err_msg=f"bf16 T={T}")
            np.testing.assert_array_equal(bits(_run(A, W, N, vd.EPI_RESIDUAL, R)), bits(want_res),
                                          err_msg=f"residual T={T}")
            X = R.clone()
            vd.gemm(A, W, X, vd.EPI_RESIDUAL, X)  # in place
            torch.cuda.synchronize()
            np.testing.assert_array_equal(bits(X), bits(want_res), err_msg=f"in place T={T}")
    finally:
        vd.set_gemm_plan(0, 0, 0)


@pytest.mark.parametrize("epi", [vd.EPI_SWIGLU, vd.EPI_GEGLU])
def test_glu_epilogue_vs_oracle(epi):
    ready()
    T, F, K = 45, 192, 256
    A = synth.make_normal_bf16((T, K), seed=40).cuda()
    W = synth.make_normal_bf16((2 * F, K), seed=41, std=0.1).cuda()
    acc = f64(A) @ f64(W).T
    g, u = round_bf16(acc[:, :F]), round_bf16(acc[:, F:])
    act = silu(g) if epi == vd.EPI_SWIGLU else gelu_tanh(g)
    ref = round_bf16(act * u)
    out = f64(_run(A, W, F, epi))
    # g and u may each differ by one bf16 ulp (|act'| <= 1.2), plus the final rounding
    bound = 2.0 ** -7 * np.abs(u) * (1.2 * np.abs(g) + np.abs(act)) + 2.0 ** -7 * np.abs(ref) + 1e-30
    assert np.all(np.abs(out - ref) <= bound)


def test_rmsnorm_vs_oracle_and_row_invariance():
    ready()
    from oracle.decoder import rmsnorm
    for d in (256, 2560, 4096):
        x = synth.make_normal_bf16((33, d), seed=d).cuda()
        w = synth.make_normal_bf16((d,), seed=d + 1, std=0.1).cuda() + 1
        w = w.to(torch.bfloat16)
        y = torch.empty_like(x)
        vd.rmsnorm(x, w, y, 1e-5)
        torch.cuda.synchronize()
        ref = rmsnorm(f64(x), f64(w), 1e-5)
        assert np.all(bf16_ulp_dist(f64(y), ref) <= 1)
        y1 = torch.empty_like(x[:1])
        vd.rmsnorm(x[17:18].contiguous(), w, y1, 1e-5)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits(y1)[0], bits(y)[17])
