"""Pins for the float32 C++ oracle (oracle/fp32_decoder.cpp).

Each check ties the oracle to something other than itself: the bf16 format
(hand-worked ties, and the float64 oracle's rounding, itself pinned against
PyTorch), closed forms, brute force in 40-digit arithmetic, exact small-
integer products, torch float64 reductions of one- and two-token forwards
written from the definition, and the float64 numpy oracle as an
independent cross-check within the stated tolerance.  Where float32
rounding makes a closed form inexact, the check uses the unrounded output
and a bound derived from float32's unit roundoff (2^-24).
"""

import math
import os

import mpmath
import numpy as np
import pytest
import torch

from invariant_vd_step_gb300 import synth
from oracle import decoder as od
from oracle import fp32 as oc
from oracle.bf16 import round_bf16 as round64

U = 2.0 ** -24  # float32 unit roundoff


def bits16(x):
    return oc.to_bits(oc.round_bf16(x))


# ---------------------------------------------------------------- bf16 rounding
def test_bf16_rounding_hand_worked_and_against_the_float64_oracle():
    one = 1.0
    cases = {
        one + 2 ** -8: one,                      # tie, 1.0 is even
        one + 3 * 2 ** -8: one + 2 ** -6,        # tie, rounds to the even neighbour above
        one + 2 ** -8 + 2 ** -20: one + 2 ** -7,  # just above the tie
        -(one + 2 ** -8): -one,
        2.0 ** -130: 2.0 ** -130,               # subnormal kept
        3.4e38: math.inf,                        # past the largest bf16
        3.39e38: 3.3895313892515355e38,          # to the largest finite bf16
    }
    got = oc.round_bf16(np.array(list(cases), dtype=np.float32))
    np.testing.assert_array_equal(got, np.array(list(cases.values()), dtype=np.float32))
    assert np.isnan(oc.round_bf16(np.array([np.nan], np.float32))[0])
    rng = np.random.default_rng(0)
    with np.errstate(over="ignore"):  # some draws overflow float32 to infinity on purpose
        x = (rng.standard_normal(200000) * np.exp(rng.uniform(-90, 90, 200000))).astype(np.float32)
    np.testing.assert_array_equal(oc.round_bf16(x), round64(x.astype(np.float64)).astype(np.float32))


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_closed_forms():
    for c in (0.5, -3.0, 7.25, 1e-3):
        x = np.full((1, 64), c, np.float32)
        c32 = np.float32(c)
        # float32 evaluation of c / sqrt(c^2 + eps): one float32 op at a time
        ss = np.float32(0)
        for _ in range(64):
            ss = np.float32(ss + c32 * c32)
        inv = np.float32(1) / np.sqrt(np.float32(ss / np.float32(64)) + np.float32(1e-5))
        want = oc.round_bf16(np.array([c32 * inv]))[0]
        np.testing.assert_array_equal(oc.rmsnorm(x, np.ones(64), 1e-5), np.full((1, 64), want))
        # and the exact value, to within float32 error before the bf16 rounding
        unr = oc.rmsnorm(x, np.ones(64), 1e-5, round=False)[0, 0]
        assert abs(unr - c / math.sqrt(c * c + 1e-5)) <= 8 * U
    # offset gains: g = 1 + w, w = -1 gives exactly 0
    x = np.full((2, 32), 2.0, np.float32)
    np.testing.assert_array_equal(oc.rmsnorm(x, -np.ones(32), 1e-6, offset=True), np.zeros((2, 32)))
    a = 2.0
    r = a / math.sqrt(a * a + 1e-6)
    w = np.arange(1, 17) / 4.0
    got = oc.rmsnorm(np.array([[a, -a] * 8]), w - 1.0, 1e-6, offset=True, round=False)[0]
    np.testing.assert_allclose(got, np.array([r, -r] * 8) * w, rtol=4 * U, atol=0)


def test_qk_norm_per_head_closed_form():
    # each head of hd elements normalised on its own (the model calls the
    # norm with rows of hd elements); a constant head c_h gives c_h/sqrt(c_h^2+eps)*g
    c = np.array([0.5, -3.0, 40.0])
    x = np.repeat(c[None, :, None], 16, axis=2).astype(np.float32)
    g = np.linspace(0.5, 1.5, 16)
    got = oc.rmsnorm(x, g, 1e-6, round=False)
    want = (c / np.sqrt(c * c + 1e-6))[None, :, None] * g[None, None, :]
    np.testing.assert_allclose(got, want, rtol=4 * U, atol=0)


# ---------------------------------------------------------------- RoPE
def test_rope_identity_rotations_and_norm():
    rng = np.random.default_rng(1)
    x = oc.round_bf16(rng.standard_normal((1, 3, 64)))
    np.testing.assert_array_equal(oc.rope(x, [0], 1e4), x)
    for p in (1, 2, 5, 100):  # hd = 2: (1, 0) -> (cos p, sin p)
        got = oc.rope(np.array([[[1.0, 0.0]]]), [p], 1e4, round=False)[0, 0]
        np.testing.assert_array_equal(got, np.array([math.cos(p), math.sin(p)], np.float32))
    # hd = 4, theta = 16: pairs (0,2) at frequency 1, (1,3) at 1/4; second-half elements rotate the other way
    e = np.eye(4)[:, None, :]
    got = oc.rope(e, [3] * 4, 16.0, round=False)[:, 0]
    c3, s3, c1, s1 = math.cos(3), math.sin(3), math.cos(0.75), math.sin(0.75)
    want = np.array([[c3, 0, s3, 0], [0, c1, 0, s1], [-s3, 0, c3, 0], [0, -s1, 0, c1]], np.float32)
    np.testing.assert_array_equal(got, want)
    # a rotation keeps each pair's norm (before rounding), to float32 precision
    x = oc.round_bf16(rng.standard_normal((5, 2, 64)))
    y = oc.rope(x, [0, 7, 300, 4097, 8191], 5e5, round=False).astype(np.float64)
    n0 = x[..., :32].astype(np.float64) ** 2 + x[..., 32:].astype(np.float64) ** 2
    n1 = y[..., :32] ** 2 + y[..., 32:] ** 2
    assert np.all(np.abs(n1 - n0) <= 2.0 ** -21 * n0 + 1e-30)


def test_rope_relative_position_property():
    rng = np.random.default_rng(2)
    q = oc.round_bf16(rng.standard_normal((1, 1, 64)))
    k = oc.round_bf16(rng.standard_normal((1, 1, 64)))
    dot = lambda m, n: float(oc.rope(q, [m], 1e4, round=False)[0, 0].astype(np.float64) @
                             oc.rope(k, [n], 1e4, round=False)[0, 0].astype(np.float64))
    ref = dot(7, 3)
    for shift in (1, 10, 500):
        assert abs(dot(7 + shift, 3 + shift) - ref) < 1e-4 * (abs(ref) + 1)
    assert abs(dot(7, 3) - dot(9, 3)) > 1e-2


# ---------------------------------------------------------------- attention
def _kv(rng, P, Hkv, hd, scale=1.0):
    return bits16(rng.standard_normal((P, Hkv, hd)) * scale), bits16(rng.standard_normal((P, Hkv, hd)))


def test_attention_single_key_equal_keys_and_gqa():
    rng = np.random.default_rng(3)
    K, V = _kv(rng, 1, 1, 8)
    q = oc.round_bf16(rng.standard_normal((1, 1, 8)))
    np.testing.assert_array_equal(oc.attention(q, K, V, [0])[0, 0], oc.from_bits(V[0, 0]))
    # equal keys: every weight is exp(0) = 1, so the output is the mean; with
    # 4 keys and small-integer values every float32 step is exact
    K = np.tile(bits16(rng.standard_normal(8)), (4, 1, 1))
    Vv = rng.integers(-20, 21, (4, 1, 8)).astype(np.float32)
    got = oc.attention(q, K, oc.to_bits(Vv), [3])[0, 0]
    np.testing.assert_array_equal(got, round64(Vv[:, 0].astype(np.float64).mean(0)))
    # 4 query heads over 2 kv heads: heads 0,1 read kv 0; heads 2,3 read kv 1
    K = oc.to_bits(np.ones((4, 2, 8), np.float32))
    Vv = np.zeros((4, 2, 8), np.float32)
    Vv[:, 0] = 1.5
    Vv[:, 1] = -2.5
    out = oc.attention(oc.round_bf16(rng.standard_normal((1, 4, 8))), K, oc.to_bits(Vv), [3])[0]
    np.testing.assert_array_equal(out[:, 0], [1.5, 1.5, -2.5, -2.5])


def test_attention_two_key_closed_form_checks_scale():
    hd, a = 16, 3.0
    q = np.zeros((1, 1, hd), np.float32)
    q[0, 0, 0] = a
    Kv = np.zeros((2, 1, hd), np.float32)
    Kv[0, 0, 0] = 1.0
    Vv = np.zeros((2, 1, hd), np.float32)
    Vv[0] = 1.0
    Vv[1] = -1.0
    w0 = 1.0 / (1.0 + math.exp(-a / math.sqrt(hd)))
    got = oc.attention(q, oc.to_bits(Kv), oc.to_bits(Vv), [1], round=False)[0, 0]
    np.testing.assert_allclose(got, 2 * w0 - 1, rtol=0, atol=8 * U)


def test_attention_brute_force_high_precision():
    rng = np.random.default_rng(4)
    mpmath.mp.dps = 40
    for trial in range(8):
        n, hd = 8, 8
        K, V = _kv(rng, n, 1, hd, scale=2.0)
        Kf, Vf = oc.from_bits(K), oc.from_bits(V)
        q = oc.round_bf16(rng.standard_normal((1, 1, hd)) * 2)
        p = int(rng.integers(0, n))
        s = [mpmath.fsum(mpmath.mpf(float(q[0, 0, d])) * mpmath.mpf(float(Kf[j, 0, d])) for d in range(hd))
             / mpmath.sqrt(hd) for j in range(p + 1)]
        e = [mpmath.exp(v) for v in s]
        Z = mpmath.fsum(e)
        want = np.array([float(mpmath.fsum(e[j] * mpmath.mpf(float(Vf[j, 0, d])) for j in range(p + 1)) / Z)
                         for d in range(hd)])
        mag = np.array([float(mpmath.fsum(e[j] * abs(mpmath.mpf(float(Vf[j, 0, d]))) for j in range(p + 1)) / Z)
                        for d in range(hd)])
        got = oc.attention(q, K, V, [p], round=False)[0, 0]
        assert np.all(np.abs(got - want) <= 1e-6 * mag), (trial, np.abs(got - want).max())
        np.testing.assert_array_equal(oc.attention(q, K, V, [p])[0, 0], oc.round_bf16(got))


def test_softmax_weights_sum_to_one():
    rng = np.random.default_rng(5)
    P, Hq, Hkv, hd = 64, 4, 2, 16
    K, V = _kv(rng, P, Hkv, hd, scale=3.0)
    q = oc.round_bf16(rng.standard_normal((6, Hq, hd)) * 3)
    pos = np.array([0, 1, 9, 30, 50, 63])
    for window in (0, 7):
        _, w = oc.attention(q, K, V, pos, window, probs=True)
        sums = w.astype(np.float64).sum(-1)
        assert np.all(np.abs(sums - 1.0) <= P * 2 * U), np.abs(sums - 1).max()
        assert np.all(w >= 0)
        for t, p in enumerate(pos):
            lo = max(0, p - window + 1) if window else 0
            assert np.all(w[t, :, :lo] == 0) and np.all(w[t, :, p + 1:] == 0)
            assert np.all(w[t, :, lo:p + 1] > 0)


def test_attention_causal_window_and_permutation():
    rng = np.random.default_rng(6)
    P, hd = 12, 8
    K, V = _kv(rng, P, 1, hd)
    q = oc.round_bf16(rng.standard_normal((1, 1, hd)))
    base = oc.attention(q, K, V, [6])
    K2, V2 = K.copy(), V.copy()
    K2[7:] = bits16(np.full(hd, 99.0))
    V2[7:] = bits16(np.full(hd, -99.0))
    np.testing.assert_array_equal(oc.attention(q, K2, V2, [6]), base)  # future keys are not read
    w = oc.attention(q, K, V, [6], window=3)  # keys 4..6 only
    K3 = K.copy()
    K3[:4] = bits16(np.full(hd, 50.0))
    np.testing.assert_array_equal(oc.attention(q, K3, V, [6], window=3), w)
    np.testing.assert_array_equal(w, oc.attention(q, K[4:7], V[4:7], [2]))
    np.testing.assert_array_equal(oc.attention(q, K, V, [6], window=7), base)
    # attention is a function of the set of (k, v) pairs: a permutation changes
    # only the order of the float32 sums
    perm = np.array([3, 0, 6, 1, 5, 2, 4])
    a = oc.attention(q, K[:7][perm], V[:7][perm], [6], round=False)
    b = oc.attention(q, K, V, [6], round=False)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-6)


# ---------------------------------------------------------------- projections and GLU
def test_linear_small_integers_exact_and_error_bound():
    rng = np.random.default_rng(7)
    W = rng.integers(-8, 9, size=(512, 256))
    x = rng.integers(-8, 9, size=(5, 256)).astype(np.float32)
    got = oc.linear(x, synth.bf16_to_u16(torch.from_numpy(W).to(torch.bfloat16)))
    np.testing.assert_array_equal(got, (x.astype(np.float64) @ W.T))
    # random bf16 operands: within the float32 accumulation bound of the exact product
    Wb = synth.bf16_to_u16(synth.make_normal_bf16((300, 4096), seed=8, std=0.02))
    xb = oc.round_bf16(rng.standard_normal((3, 4096)))
    Wf = oc.from_bits(Wb).astype(np.float64)
    exact = xb.astype(np.float64) @ Wf.T
    bound = 4096 * U * (np.abs(xb.astype(np.float64)) @ np.abs(Wf).T)
    got = oc.linear(xb, Wb)
    assert np.all(np.abs(got - exact) <= bound)
    assert np.any(got != exact.astype(np.float32))  # float32 rounding is really there


def test_glu_matches_torch_activations():
    g = np.linspace(-6, 6, 241).astype(np.float32)
    u = oc.round_bf16(np.cos(np.arange(241)) * 2)
    for act, fn in (("swiglu", lambda t: torch.nn.functional.silu(t)),
                    ("geglu", lambda t: torch.nn.functional.gelu(t, approximate="tanh"))):
        want = fn(torch.from_numpy(g.astype(np.float64))).numpy() * u
        got = oc.glu(g, u, act).astype(np.float64)
        # one bf16 rounding of a value within float32 error of want
        assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-6), act


def test_layer_rule_is_five_local_to_one_global():
    pattern = [oc.layer_is_local(i, 1024, 6) for i in range(34)]
    assert pattern == ([True] * 5 + [False]) * 5 + [True] * 4
    assert not any(oc.layer_is_local(i, 0, 6) for i in range(12))
    assert not any(oc.layer_is_local(i, 1024, 0) for i in range(12))
    assert all(oc.layer_is_local(i, 1024, 6) == od.layer_is_local(i, 1024, 6) for i in range(60))


# ---------------------------------------------------------------- model
def _tiny(seed=0, gain_std=0.0, threads=None, **kw):
    spec = synth.TINY.with_(**kw)
    W = synth.make_weights(spec, seed=seed, gain_std=gain_std)
    return spec, W, oc.Fp32Decoder(spec, synth.weights_to_numpy(W), threads=threads)


def test_zero_model_golden_outputs():
    path = os.path.join(os.path.dirname(__file__), "golden", "zero_model_outputs.txt")
    with open(path) as f:
        kv = dict(line.split() for line in f if line.strip() and not line.startswith("#"))
    for extra in ({}, dict(embed_scale=True, norm_offset=True, sandwich_norm=True, qk_norm=True, act="geglu")):
        spec = synth.TINY.with_(**extra)
        dec = oc.Fp32Decoder(spec, synth.weights_to_numpy(synth.make_weights(spec, zero=True)))
        lg = dec.forward_all(synth.make_tokens(9, spec.vocab)).astype(np.float32)
        assert np.all(lg.view(np.uint32) == int(kv["logit_float32_bits"], 16))


def _torch_forward_one_token(spec, W, tok):
    """A single token attends to itself only, so attention returns v; the
    rest written from the block's definition with torch float64 ops."""
    T = {k: v.to(torch.float64) for k, v in W.items()}
    bf = lambda t: t.to(torch.bfloat16).to(torch.float64)
    off = 1.0 if spec.norm_offset else 0.0
    rms = lambda x, w: bf(x * torch.rsqrt((x * x).mean() + spec.rms_eps) * (w + off))
    x = T["embed"][tok]
    if spec.embed_scale:
        x = bf(x * bf(torch.tensor(math.sqrt(spec.d_model), dtype=torch.float64)))
    Hq, Hkv, hd, F = spec.n_heads, spec.n_kv_heads, spec.head_dim, spec.ffn_dim
    for i in range(spec.n_layers):
        p = f"layers.{i}."
        a = rms(x, T[p + "attn_norm"])
        v = bf(T[p + "wqkv"][(Hq + Hkv) * hd:] @ a).reshape(Hkv, hd)
        h = bf(T[p + "wo"] @ v.repeat_interleave(Hq // Hkv, dim=0).reshape(-1))
        x = bf(x + (rms(h, T[p + "post_attn_norm"]) if spec.sandwich_norm else h))
        a = rms(x, T[p + "ffn_norm"])
        g = bf(T[p + "w_gate_up"][:F] @ a)
        u = bf(T[p + "w_gate_up"][F:] @ a)
        act = torch.nn.functional.gelu(g, approximate="tanh") if spec.act == "geglu" else torch.nn.functional.silu(g)
        h = bf(T[p + "w_down"] @ bf(act * u))
        x = bf(x + (rms(h, T[p + "post_ffn_norm"]) if spec.sandwich_norm else h))
    return (T["lm_head"] @ rms(x, T["final_norm"])).numpy()


GEMMA_BLOCK = dict(act="geglu", qk_norm=True, embed_scale=True, norm_offset=True, sandwich_norm=True, rms_eps=1e-6)


@pytest.mark.parametrize("extra", [{}, GEMMA_BLOCK], ids=["llama", "gemma"])
def test_one_token_forward_reduces_to_library_ops(extra):
    spec, W, dec = _tiny(seed=3, gain_std=0.1, **extra)
    want = _torch_forward_one_token(spec, W, 29)
    got = dec.forward(np.array([29]))
    # float32 sums against float64 ones: the bf16 roundings may flip a few
    # values, which moves a logit by ~1e-3 at most at this size; a wiring
    # mistake (a wrong slice, a missing norm or gain) moves them by > 0.05
    assert np.abs(got - want).max() < 5e-3, np.abs(got - want).max()
    wrong = dict(extra)
    wrong["norm_offset"] = not extra.get("norm_offset", False)
    spec_w = spec.with_(**wrong)
    assert np.abs(_torch_forward_one_token(spec_w, W, 29) - want).max() > 0.05


def test_qk_norm_two_token_wiring():
    import test_oracle_decoder as t64
    spec, W, dec = _tiny(seed=9, gain_std=0.5, n_layers=1, qk_norm=True)
    toks = np.array([11, 1500])
    want = t64._qk_reference(spec, W, toks)
    assert np.abs(dec.forward(toks) - want).max() < 5e-3
    for wrong in ("after_rope", "no_gain", "whole_row"):
        assert np.abs(t64._qk_reference(spec, W, toks, wrong) - want).max() > 0.05, wrong


def test_local_layer_uses_its_own_rope_theta():
    import test_oracle_decoder as t64
    spec, W, dec = _tiny(seed=10, gain_std=0.5, **t64.LOCAL_THETA)
    toks = np.array([7, 1999])
    want = t64._qk_reference(spec, W, toks, theta=spec.rope_theta_local)
    assert np.abs(dec.forward(toks) - want).max() < 5e-3
    assert np.abs(t64._qk_reference(spec, W, toks, theta=spec.rope_theta) - want).max() > 0.05


def test_fkv_lemma_and_incremental_equals_cold_bitwise():
    spec, W, dec = _tiny(seed=2, gain_std=0.1, **GEMMA_BLOCK, sliding_window=5, local_global_period=2)
    h = synth.make_tokens(30, spec.vocab, seed=12)
    cold, cache = dec.step(h, dec.empty_cache(), logit_rows=range(30))
    for p in (0, 5, 16, 29):
        for layer, (k, v) in enumerate(dec.fkv(h, p)):
            np.testing.assert_array_equal(oc.from_bits(cache.K[layer, p]), k)
            np.testing.assert_array_equal(oc.from_bits(cache.V[layer, p]), v)
    c, parts = dec.empty_cache(), []
    for a, b in ((0, 7), (7, 8), (8, 16), (16, 30)):
        lg, c = dec.step(h[a:b], c, logit_rows=range(b - a))
        parts.append(lg)
    np.testing.assert_array_equal(np.concatenate(parts), cold)
    h2 = h.copy()
    h2[15:] = (h2[15:] + 1) % spec.vocab
    np.testing.assert_array_equal(dec.forward_all(h2)[:15], cold[:15])


def test_sliding_window_layer_ignores_tokens_before_the_window():
    spec, W, dec = _tiny(seed=4, n_layers=1, sliding_window=4, local_global_period=1000)
    h = synth.make_tokens(12, spec.vocab, seed=13)
    h2 = h.copy()
    h2[:8] = (h2[:8] + 5) % spec.vocab
    np.testing.assert_array_equal(dec.forward(h2), dec.forward(h))
    g = spec.with_(local_global_period=1)  # every layer global: now the early tokens matter
    d2 = oc.Fp32Decoder(g, synth.weights_to_numpy(W))
    assert np.any(d2.forward(h2) != d2.forward(h))


def test_thread_count_does_not_change_a_bit():
    spec, W, _ = _tiny(seed=5, gain_std=0.1, **GEMMA_BLOCK)
    h = synth.make_tokens(20, spec.vocab, seed=14)
    one = oc.Fp32Decoder(spec, synth.weights_to_numpy(W), threads=1).forward_all(h)
    many = oc.Fp32Decoder(spec, synth.weights_to_numpy(W), threads=7).forward_all(h)
    np.testing.assert_array_equal(one, many)


GEMMA_TINY = synth.ModelSpec("gemma-tiny", 3, 256, 2, 1, 256, 512, 512, act="geglu", qk_norm=True,
                             rope_theta=1e6, rope_theta_local=1e4, sliding_window=24, local_global_period=2,
                             rms_eps=1e-6, embed_scale=True, norm_offset=True, sandwich_norm=True)
LLAMA_TINY128 = synth.ModelSpec("llama-tiny-128", 2, 512, 8, 2, 128, 1024, 1024, rope_theta=5e5,
                                rope_theta_local=5e5)


@pytest.mark.parametrize("spec", [synth.TINY, GEMMA_TINY, LLAMA_TINY128], ids=lambda s: s.name)
def test_agrees_with_the_float64_oracle(spec):
    W = synth.weights_to_numpy(synth.make_weights(spec, seed=1, gain_std=0.1))
    h = synth.make_tokens(60, spec.vocab, seed=2)
    a = oc.Fp32Decoder(spec, W).forward_all(h)
    b = od.OracleDecoder(spec, W).forward_all(h)
    assert np.all(np.abs(a - b) <= 2e-2 + 1e-2 * np.abs(b)), np.abs(a - b).max()
