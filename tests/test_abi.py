"""The C-ABI library builds, loads and exports every declared symbol (CPU)."""

import ctypes

import pytest

from invariant_vd_step_gb300 import build, vd


@pytest.fixture(scope="module")
def L():
    build.build()
    return vd.lib()


def test_exports_every_header_symbol(L):
    names = vd.header_symbols()
    assert {"vd_create_model", "vd_kv_pool_alloc", "vd_step", "vd_sample"} <= names
    raw = ctypes.CDLL(build.LIB)
    missing = [n for n in sorted(names) if not hasattr(raw, n)]
    assert not missing, missing
    assert names == set(vd._SIGS), names ^ set(vd._SIGS)
    assert L.vd_version().decode().startswith("vd ")


def test_create_model_rejects_unsupported_shapes_before_any_cuda_call(L):
    from invariant_vd_step_gb300 import synth
    lw = (vd.LayerWeights * 2)()
    for i in range(2):
        lw[i] = vd.LayerWeights(*([16] * 8))
    w = vd.WeightPtrs(16, lw, 16, 16)
    h = ctypes.c_void_p()
    bad = [
        (synth.TINY.with_(head_dim=96), vd.ERRORS and 2),       # head_dim
        (synth.TINY.with_(page_size=32), 2),                     # page size
        (synth.TINY.with_(d_model=200), 2),                      # no GEMM tiling
        (synth.TINY.with_(n_kv_heads=3), 1),                     # Hq % Hkv
        (synth.TINY.with_(sandwich_norm=True), 1),               # post-sub-layer norms missing
    ]
    for spec, code in bad:
        cfg = vd.config_of(spec, 64, 4, 8, 256)
        assert L.vd_create_model(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == code
        assert L.vd_last_error()
    assert L.vd_create_model(None, None, None) == 1


def test_ops_validate_arguments(L):
    assert L.vd_op_gemm(None, None, None, 1, 128, 64, 0, None, None) == 1
    assert L.vd_op_gemm(16, 16, 16, 1, 100, 64, 0, None, None) == 2      # N not a tile multiple
    assert L.vd_op_gemm(16, 16, 16, 1, 128, 64, 1, None, None) == 1      # residual missing
    assert L.vd_op_gemm(16, 16, 16, 1, 128, 64, 1, 18, None) == 1        # residual not 16-byte aligned
    assert L.vd_op_gemm(16, 16, 16, 1, 128, 64, 9, None, None) == 1      # unknown epilogue
    assert L.vd_op_rmsnorm(16, 16, 16, 4, 12, 1e-5, None) == 1           # d % 8
    assert L.vd_op_philox(1, 2, -1, None, None) == 1
    assert L.vd_sample(None, None, 1, None, None, None) == 1
    assert L.vd_step(None, None, None, None, None) == 1


def test_step_batch_from_arrays_matches_per_request_builder():
    import numpy as np
    seqs = [(np.array([5, 6, 7]), 10, np.array([3, 4])), (np.array([9]), 0, np.array([8]))]
    a = vd.StepBatch(seqs, logit_rows=[2, 3])
    b = vd.StepBatch.from_arrays(np.array([5, 6, 7, 9]), np.array([0, 3, 4]), np.array([10, 0]),
                                 np.array([[3, 4], [8, 0]]), [2, 3])
    for f in ("tokens", "positions", "cu_q", "cached", "page_table", "logit_rows"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    assert (a.c.num_tokens, a.c.num_seqs, a.c.num_logit_rows, a.c.page_table_stride) == \
        (b.c.num_tokens, b.c.num_seqs, b.c.num_logit_rows, b.c.page_table_stride)


def test_gemm_plan_query_and_override_host_logic(L):
    """The per-launch GEMM shape is host logic: it comes from the documented
    sets, never splits a K block between copies, keeps 64-row tiles away from
    the fused token choice, and a forced shape applies where a launch can take
    it (no GPU work; the SM count falls back to a default without a GPU)."""
    shapes = [(6144, 4096, vd.EPI_BF16), (4096, 14336, vd.EPI_RESIDUAL), (14336, 4096, vd.EPI_SWIGLU),
              (128256, 4096, 5), (512, 256, vd.EPI_BF16), (768, 256, vd.EPI_GEGLU)]
    try:
        for N, K, epi in shapes:
            for T in (1, 5, 16, 64, 100, 256, 300, 2048, 8192):
                bm, bn, kpo = vd.gemm_plan(T, N, K, epi)
                assert bm in (64, 128, 256) and bn in (16, 32, 64, 128, 256) and kpo in (1, 2, 4), (N, K, T)
                assert (K // 64) % kpo == 0
                assert bn <= max(16, 1 << (T - 1).bit_length())
                if epi == 5:
                    assert bm != 64          # the token choice scores 32-row groups per warp
                if bm == 256:
                    assert kpo == 1 and N * (2 if epi in (vd.EPI_SWIGLU, vd.EPI_GEGLU) else 1) % 256 == 0
        vd.set_gemm_plan(64, 32, 4)
        assert vd.gemm_plan(7, 4096, 4096, vd.EPI_BF16) == (64, 32, 4)
        bm, bn, _ = vd.gemm_plan(7, 128256, 4096, 5)              # bm 64 is not taken by the token choice
        assert bm != 64 and bn == 32
        assert vd.gemm_plan(7, 512, 192, vd.EPI_BF16)[2] == 1      # 3 K blocks: kpo 4 does not divide them
        vd.set_gemm_plan(0, 256, 0)
        assert vd.gemm_plan(7, 4096, 4096, vd.EPI_BF16)[1] == 256
    finally:
        vd.set_gemm_plan(0, 0, 0)
    for bad in [(32, 0, 0), (0, 48, 0), (0, 0, 3)]:
        with pytest.raises(vd.VDError):
            vd.set_gemm_plan(*bad)
    with pytest.raises(vd.VDError):
        vd.gemm_plan(0, 4096, 4096)
    with pytest.raises(vd.VDError):
        vd.gemm_plan(1, 4096, 100)   # K not a multiple of 64
