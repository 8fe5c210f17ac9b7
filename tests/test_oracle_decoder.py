"""Pins for the oracle decoder: closed forms, special cases and invariants."""

import math

import mpmath
import numpy as np
import torch

from invariant_vd_step_gb300 import synth
from oracle import decoder as od
from oracle.bf16 import bits_to_f64, round_bf16


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_constant_row_closed_form():
    for c in (0.5, -3.0, 1e-3, 7.25):
        x = np.full((1, 64), c)
        w = np.ones(64)
        want = round_bf16(np.array(c / math.sqrt(c * c + 1e-5)))
        np.testing.assert_array_equal(od.rmsnorm(x, w, 1e-5), np.full((1, 64), want))


def test_rmsnorm_gain_and_two_value_row():
    # row (a, -a, a, -a ...) has mean square a^2; output = sign * a/sqrt(a^2+eps) * w
    a = 2.0
    x = np.array([[a, -a] * 8])
    w = np.arange(1, 17) / 4.0
    r = a / math.sqrt(a * a + 1e-6)
    want = round_bf16(np.array([r, -r] * 8) * w)
    np.testing.assert_array_equal(od.rmsnorm(x, w, 1e-6)[0], want)


# ---------------------------------------------------------------- RoPE
def test_rope_identity_at_position_zero():
    rng = np.random.default_rng(0)
    x = round_bf16(rng.standard_normal((1, 3, 64)))
    np.testing.assert_array_equal(od.rope(x, [0], 1e4), x)


def test_rope_hd2_is_plane_rotation():
    # hd = 2: inv_freq = 1, (1, 0) at position p -> (cos p, sin p)
    for p in (1, 2, 5, 100):
        got = od.rope(np.array([[[1.0, 0.0]]]), [p], 1e4)[0, 0]
        np.testing.assert_array_equal(got, round_bf16(np.array([math.cos(p), math.sin(p)])))


def test_rope_hd4_pairs_rotate_half():
    # hd = 4, theta = 16: pairs (0,2) at frequency 1, (1,3) at 16^(-1/2) = 1/4
    p = 3
    e0 = od.rope(np.array([[[1.0, 0, 0, 0]]]), [p], 16.0)[0, 0]
    e1 = od.rope(np.array([[[0, 1.0, 0, 0]]]), [p], 16.0)[0, 0]
    np.testing.assert_array_equal(e0, round_bf16(np.array([math.cos(3), 0, math.sin(3), 0])))
    np.testing.assert_array_equal(e1, round_bf16(np.array([0, math.cos(0.75), 0, math.sin(0.75)])))
    # rotating the second half element goes the other way: (0,0,1,0) -> (-sin, 0, cos, 0)
    e2 = od.rope(np.array([[[0, 0, 1.0, 0]]]), [p], 16.0)[0, 0]
    np.testing.assert_array_equal(e2, round_bf16(np.array([-math.sin(3), 0, math.cos(3), 0])))


def test_rope_relative_position_property():
    # <rope(q, m), rope(k, n)> depends only on m - n (checked before rounding
    # by using values that survive bf16 rounding exactly: compare with loose tol)
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    def dot(m, n):
        a = od.rope(q, [m], 1e4)[0, 0]
        b = od.rope(k, [n], 1e4)[0, 0]
        return a @ b
    ref = dot(7, 3)
    for shift in (1, 10, 500):
        assert abs(dot(7 + shift, 3 + shift) - ref) < 0.05 * (abs(ref) + 1)
    # a non-rotation (sign error) breaks this by far more: sanity of the tolerance
    assert abs(dot(7, 3) - dot(9, 3)) > 1e-3


# ---------------------------------------------------------------- attention
def _attn(q, K, V, pos, window=0):
    return od.attention(np.asarray(q, float), np.asarray(K, float), np.asarray(V, float), pos, window)


def test_attention_single_visible_key_returns_v0():
    rng = np.random.default_rng(2)
    K = round_bf16(rng.standard_normal((1, 1, 8)))
    V = round_bf16(rng.standard_normal((1, 1, 8)))
    q = round_bf16(rng.standard_normal((1, 1, 8)))
    np.testing.assert_array_equal(_attn(q, K, V, [0])[0, 0], V[0, 0])


def test_attention_equal_keys_gives_mean_of_values():
    rng = np.random.default_rng(3)
    k = rng.standard_normal(8)
    K = np.tile(k, (5, 1, 1))
    V = rng.standard_normal((5, 1, 8))
    q = rng.standard_normal((1, 1, 8))
    got = _attn(q, K, V, [4])[0, 0]
    np.testing.assert_array_equal(got, round_bf16(V[:, 0].mean(0)))


def test_attention_two_key_closed_form_checks_scale():
    # q = a e0, k0 = e0, k1 = 0: weights sigmoid(a/sqrt(hd)), 1 - that
    hd = 16
    a = 3.0
    q = np.zeros((1, 1, hd)); q[0, 0, 0] = a
    K = np.zeros((2, 1, hd)); K[0, 0, 0] = 1.0
    V = np.zeros((2, 1, hd)); V[0, 0, :] = 1.0; V[1, 0, :] = -1.0
    w0 = 1.0 / (1.0 + math.exp(-a / math.sqrt(hd)))
    got = _attn(q, K, V, [1])[0, 0]
    np.testing.assert_array_equal(got, round_bf16(np.full(hd, w0 - (1 - w0))))


def test_attention_brute_force_high_precision():
    rng = np.random.default_rng(4)
    mpmath.mp.dps = 40
    for trial in range(5):
        n, hd = 6, 8
        K = rng.standard_normal((n, 1, hd)); V = rng.standard_normal((n, 1, hd))
        q = rng.standard_normal((1, 1, hd))
        p = int(rng.integers(0, n))
        s = [mpmath.fsum(mpmath.mpf(float(q[0, 0, d])) * mpmath.mpf(float(K[j, 0, d])) for d in range(hd))
             / mpmath.sqrt(hd) for j in range(p + 1)]
        e = [mpmath.exp(v) for v in s]
        Z = mpmath.fsum(e)
        want = np.array([float(mpmath.fsum(e[j] * mpmath.mpf(float(V[j, 0, d])) for j in range(p + 1)) / Z)
                         for d in range(hd)])
        np.testing.assert_array_equal(_attn(q, K, V, [p])[0, 0], round_bf16(want))


def test_attention_causal_and_window_and_permutation():
    rng = np.random.default_rng(5)
    P, hd = 12, 8
    K = rng.standard_normal((P, 1, hd)); V = rng.standard_normal((P, 1, hd))
    q = rng.standard_normal((1, 1, hd))
    base = _attn(q, K, V, [6])
    K2 = K.copy(); V2 = V.copy(); K2[7:] = 99.0; V2[7:] = -99.0  # future keys
    np.testing.assert_array_equal(_attn(q, K2, V2, [6]), base)
    # window 3 at p=6 sees keys 4..6 only
    w = _attn(q, K, V, [6], window=3)
    K3 = K.copy(); K3[:4] = 50.0
    np.testing.assert_array_equal(_attn(q, K3, V, [6], window=3), w)
    np.testing.assert_array_equal(w, _attn(q, K[4:7], V[4:7], [2]))
    # a window covering everything equals global attention
    np.testing.assert_array_equal(_attn(q, K, V, [6], window=7), base)
    # attention is a function of the set of (k, v) pairs
    perm = np.array([3, 0, 6, 1, 5, 2, 4])
    np.testing.assert_array_equal(_attn(q, K[perm], V[perm], [6]), base)


def test_attention_gqa_mapping():
    # 4 query heads over 2 kv heads: heads 0,1 -> kv 0; heads 2,3 -> kv 1
    hd, P = 8, 4
    K = np.ones((P, 2, hd))
    V = np.zeros((P, 2, hd)); V[:, 0, :] = 1.5; V[:, 1, :] = -2.5
    q = np.random.default_rng(6).standard_normal((1, 4, hd))
    out = _attn(q, K, V, [3])[0]
    np.testing.assert_array_equal(out[:, 0], [1.5, 1.5, -2.5, -2.5])


# ---------------------------------------------------------------- projections
def test_linear_small_integers_exact():
    spec = synth.TINY
    rng = np.random.default_rng(7)
    W = rng.integers(-8, 9, size=(512, 256))
    x = rng.integers(-8, 9, size=(5, 256))
    Wt = torch.from_numpy(W).to(torch.bfloat16)
    dec = od.OracleDecoder(spec, {"w": synth.bf16_to_u16(Wt)})
    got = dec.linear("w", x.astype(float))
    np.testing.assert_array_equal(got, (x @ W.T).astype(float))


# ---------------------------------------------------------------- model
def _tiny(seed=0, gain_std=0.0, **kw):
    spec = synth.TINY.with_(**kw)
    W = synth.make_weights(spec, seed=seed, gain_std=gain_std)
    return spec, W, od.OracleDecoder(spec, synth.weights_to_numpy(W))


def test_zero_model_gives_zero_logits():
    spec = synth.TINY
    W = synth.make_weights(spec, zero=True)
    dec = od.OracleDecoder(spec, synth.weights_to_numpy(W))
    logits = dec.forward(synth.make_tokens(9, spec.vocab))
    assert np.all(logits == 0)


def test_one_token_forward_reduces_to_library_ops():
    # A single token attends only to itself, so attention returns v exactly;
    # the rest is torch float64 ops on the documented weight layout.
    spec, W, dec = _tiny(seed=3, gain_std=0.1)
    tok = 17
    T = {k: v.to(torch.float64) for k, v in W.items()}
    bf = lambda t: t.to(torch.bfloat16).to(torch.float64)
    def rms(x, w):
        return bf(x * torch.rsqrt((x * x).mean() + spec.rms_eps) * w)
    x = T["embed"][tok]
    Hq, Hkv, hd, F = spec.n_heads, spec.n_kv_heads, spec.head_dim, spec.ffn_dim
    for i in range(spec.n_layers):
        p = f"layers.{i}."
        a = rms(x, T[p + "attn_norm"])
        v = bf(T[p + "wqkv"][(Hq + Hkv) * hd:] @ a).reshape(Hkv, hd)
        o = v.repeat_interleave(Hq // Hkv, dim=0).reshape(-1)
        x = bf(x + bf(T[p + "wo"] @ o))
        a = rms(x, T[p + "ffn_norm"])
        g = bf(T[p + "w_gate_up"][:F] @ a)
        u = bf(T[p + "w_gate_up"][F:] @ a)
        z = bf(torch.nn.functional.silu(g) * u)
        x = bf(x + bf(T[p + "w_down"] @ z))
    want = T["lm_head"] @ rms(x, T["final_norm"])
    got = dec.forward(np.array([tok]))
    np.testing.assert_allclose(got, want.numpy(), rtol=0, atol=1e-12)


def test_geglu_activation_matches_torch():
    g = np.linspace(-6, 6, 101)
    want = torch.nn.functional.gelu(torch.from_numpy(g), approximate="tanh").numpy()
    np.testing.assert_allclose(od.gelu_tanh(g), want, rtol=1e-14, atol=1e-15)
    want = torch.nn.functional.silu(torch.from_numpy(g)).numpy()
    np.testing.assert_allclose(od.silu(g), want, rtol=1e-14, atol=1e-15)


def test_fkv_lemma_bitwise():
    spec, W, dec = _tiny(seed=1)
    h = synth.make_tokens(24, spec.vocab, seed=11)
    _, cache = dec.step(h, dec.empty_cache())
    for p in (0, 5, 15, 23):
        kv = dec.fkv(h, p)
        for layer, (k, v) in enumerate(kv):
            np.testing.assert_array_equal(cache[layer][0][p], k)
            np.testing.assert_array_equal(cache[layer][1][p], v)


def test_incremental_equals_cold_forward_bitwise():
    # Definition 2.1 / Theorem 4.1 for the oracle itself: logits depend on the
    # history only, not on how it was split into steps.
    spec, W, dec = _tiny(seed=2, gain_std=0.1)
    h = synth.make_tokens(21, spec.vocab, seed=12)
    cold = dec.forward_all(h)
    cache = dec.empty_cache()
    rows = []
    for a, b in ((0, 7), (7, 8), (8, 16), (16, 21)):
        lg, cache = dec.step(h[a:b], cache, logit_rows=range(b - a))
        rows.append(lg)
    np.testing.assert_array_equal(np.concatenate(rows), cold)
    # causality: logits at p do not depend on later tokens
    h2 = h.copy(); h2[15:] = (h2[15:] + 1) % spec.vocab
    np.testing.assert_array_equal(dec.forward_all(h2)[:15], cold[:15])


def test_sliding_window_one_layer_ignores_tokens_before_window():
    spec, W, dec = _tiny(seed=4, n_layers=1, sliding_window=4, local_global_period=1000)
    assert od.layer_is_local(0, spec.sliding_window, spec.local_global_period)
    h = synth.make_tokens(12, spec.vocab, seed=13)
    h2 = h.copy(); h2[:8] = (h2[:8] + 5) % spec.vocab   # row 11 sees 8..11
    np.testing.assert_array_equal(dec.forward(h2), dec.forward(h))


def test_qk_norm_geglu_model_runs_and_is_causal():
    spec, W, dec = _tiny(seed=5, qk_norm=True, act="geglu", sliding_window=5,
                         local_global_period=2)
    h = synth.make_tokens(14, spec.vocab, seed=14)
    cold = dec.forward_all(h)
    assert np.all(np.isfinite(cold))
    lg, cache = dec.step(h[:9], dec.empty_cache(), logit_rows=range(9))
    lg2, _ = dec.step(h[9:], cache, logit_rows=range(5))
    np.testing.assert_array_equal(np.concatenate([lg, lg2]), cold)


def test_two_token_one_layer_attention_wiring():
    # Row 1 attends to keys 0 and 1: a 2-way softmax written with torch ops.
    # Pins the q / k / v slices of the fused QKV rows and the GQA head map.
    spec, W, dec = _tiny(seed=6, n_layers=1)
    toks = np.array([5, 901])
    T = {k: v.to(torch.float64) for k, v in W.items()}
    bf = lambda t: t.to(torch.bfloat16).to(torch.float64)
    Hq, Hkv, hd = spec.n_heads, spec.n_kv_heads, spec.head_dim
    x = T["embed"][torch.from_numpy(toks)]
    a = bf(x * torch.rsqrt((x * x).mean(-1, keepdim=True) + spec.rms_eps))
    qkv = bf(a @ T["layers.0.wqkv"].T)
    q = qkv[:, :Hq * hd].reshape(2, Hq, hd).numpy()
    k = qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(2, Hkv, hd).numpy()
    v = qkv[:, (Hq + Hkv) * hd:].reshape(2, Hkv, hd)
    q1 = torch.from_numpy(od.rope(q[1:], [1], spec.rope_theta)[0])
    kr = torch.from_numpy(np.concatenate([od.rope(k[:1], [0], spec.rope_theta),
                                          od.rope(k[1:], [1], spec.rope_theta)]))
    o = []
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = kr[:, g, :] @ q1[h] / math.sqrt(hd)
        o.append(torch.softmax(s, 0) @ v[:, g, :])
    o = bf(torch.cat(o))
    x1 = bf(x[1] + bf(T["layers.0.wo"] @ o))
    a = bf(x1 * torch.rsqrt((x1 * x1).mean() + spec.rms_eps))
    F = spec.ffn_dim
    g = bf(T["layers.0.w_gate_up"][:F] @ a)
    u = bf(T["layers.0.w_gate_up"][F:] @ a)
    x2 = bf(x1 + bf(T["layers.0.w_down"] @ bf(torch.nn.functional.silu(g) * u)))
    want = T["lm_head"] @ bf(x2 * torch.rsqrt((x2 * x2).mean() + spec.rms_eps))
    np.testing.assert_allclose(dec.forward(toks), want.numpy(), rtol=0, atol=1e-9)


# ---------------------------------------------------------------- Gemma-3 block
GEMMA_BLOCK = dict(act="geglu", qk_norm=True, embed_scale=True, norm_offset=True, sandwich_norm=True,
                   rms_eps=1e-6)


def test_rmsnorm_offset_gain_closed_form():
    # Gemma-style gains: g = 1 + w.  A constant row c with w = 0 gives c/sqrt(c^2+eps);
    # with w = -1 the gain is exactly 0.
    for c in (0.5, -3.0, 7.25):
        x = np.full((1, 32), c)
        want = round_bf16(np.array(c / math.sqrt(c * c + 1e-6)))
        np.testing.assert_array_equal(od.rmsnorm(x, np.zeros(32), 1e-6, offset=1.0), np.full((1, 32), want))
        np.testing.assert_array_equal(od.rmsnorm(x, -np.ones(32), 1e-6, offset=1.0), np.zeros((1, 32)))


def test_gemma_block_zero_model_gives_zero_logits():
    spec = synth.TINY.with_(**GEMMA_BLOCK)
    W = synth.make_weights(spec, zero=True)
    dec = od.OracleDecoder(spec, synth.weights_to_numpy(W))
    assert np.all(dec.forward(synth.make_tokens(9, spec.vocab)) == 0)


def test_gemma_block_one_token_forward_reduces_to_library_ops():
    # One token attends to itself only, so attention returns v; the rest is
    # torch float64 ops written from the block's definition: embeddings times
    # bf16(sqrt(d)), (1 + w) gains, a norm on each sub-layer output before the
    # residual add, GeGLU with the tanh GELU.
    spec, W, dec = _tiny(seed=4, gain_std=0.1, **GEMMA_BLOCK)
    assert "layers.0.post_attn_norm" in W and "layers.1.post_ffn_norm" in W
    tok = 29
    T = {k: v.to(torch.float64) for k, v in W.items()}
    bf = lambda t: t.to(torch.bfloat16).to(torch.float64)
    def rms(x, w):
        return bf(x * torch.rsqrt((x * x).mean() + spec.rms_eps) * (1.0 + w))
    x = bf(T["embed"][tok] * bf(torch.tensor(math.sqrt(spec.d_model), dtype=torch.float64)))
    Hq, Hkv, hd, F = spec.n_heads, spec.n_kv_heads, spec.head_dim, spec.ffn_dim
    for i in range(spec.n_layers):
        p = f"layers.{i}."
        a = rms(x, T[p + "attn_norm"])
        v = bf(T[p + "wqkv"][(Hq + Hkv) * hd:] @ a).reshape(Hkv, hd)
        o = v.repeat_interleave(Hq // Hkv, dim=0).reshape(-1)
        x = bf(x + rms(bf(T[p + "wo"] @ o), T[p + "post_attn_norm"]))
        a = rms(x, T[p + "ffn_norm"])
        g = bf(T[p + "w_gate_up"][:F] @ a)
        u = bf(T[p + "w_gate_up"][F:] @ a)
        z = bf(torch.nn.functional.gelu(g, approximate="tanh") * u)
        x = bf(x + rms(bf(T[p + "w_down"] @ z), T[p + "post_ffn_norm"]))
    want = T["lm_head"] @ rms(x, T["final_norm"])
    got = dec.forward(np.array([tok]))
    np.testing.assert_allclose(got, want.numpy(), rtol=0, atol=1e-12)


def test_gemma_block_incremental_equals_cold_forward_bitwise():
    spec, W, dec = _tiny(seed=6, gain_std=0.1, **GEMMA_BLOCK)
    h = synth.make_tokens(30, spec.vocab, seed=12)
    cold = dec.forward_all(h)
    cache, parts = dec.empty_cache(), []
    for a, b in ((0, 11), (11, 12), (12, 30)):
        lg, cache = dec.step(h[a:b], cache, logit_rows=range(b - a))
        parts.append(lg)
    np.testing.assert_array_equal(np.concatenate(parts), cold)


# ---------------------------------------------------------------- pins added for the layer rule,
# the softmax weights and QK-norm
def test_layer_rule_is_five_local_to_one_global():
    # Config C4 (Gemma-3-4B shape): a 5:1 interleave of window-1024 local layers and
    # global layers over 34 layers; the oracle's own rule, not the product's.
    pattern = [od.layer_is_local(i, 1024, 6) for i in range(34)]
    assert pattern == ([True] * 5 + [False]) * 5 + [True] * 4
    assert [i for i, loc in enumerate(pattern) if not loc] == [5, 11, 17, 23, 29]
    # no window or no period: every layer global
    assert not any(od.layer_is_local(i, 0, 6) for i in range(12))
    assert not any(od.layer_is_local(i, 1024, 0) for i in range(12))


def test_softmax_weights_sum_to_one_and_match_attention():
    rng = np.random.default_rng(21)
    P, Hq, Hkv, hd = 40, 4, 2, 16
    K = round_bf16(rng.standard_normal((P, Hkv, hd)) * 3)
    V = round_bf16(rng.standard_normal((P, Hkv, hd)))
    q = round_bf16(rng.standard_normal((5, Hq, hd)) * 3)
    pos = np.array([0, 7, 20, 33, 39])
    for window in (0, 6):
        w = od.attention_weights(q, K, pos, window)
        np.testing.assert_allclose(w.sum(-1), 1.0, rtol=0, atol=1e-12)
        assert np.all(w >= 0)
        for t, p in enumerate(pos):
            lo = max(0, p - window + 1) if window else 0
            assert np.all(w[t, :, :lo] == 0) and np.all(w[t, :, p + 1:] == 0)
        rep = Hq // Hkv
        want = np.stack([np.stack([w[t, h] @ V[:, h // rep] for h in range(Hq)]) for t in range(5)])
        np.testing.assert_array_equal(od.attention(q, K, V, pos, window), round_bf16(want))


def test_qk_norm_constant_head_closed_form():
    # QK-norm normalises each head over its own hd elements: a head holding
    # the constant c_h maps to c_h / sqrt(c_h^2 + eps) * gain, whatever the
    # other heads hold (a norm over the wrong axis mixes them).
    c = np.array([0.5, -3.0, 40.0])
    x = np.repeat(c[None, :, None], 16, axis=2)  # [1 token, 3 heads, hd 16]
    gain = np.linspace(0.5, 1.5, 16)
    got = od.rmsnorm(x, gain, 1e-6)
    want = round_bf16((c / np.sqrt(c * c + 1e-6))[None, :, None] * gain[None, None, :])
    np.testing.assert_array_equal(got, want)


def _qk_reference(spec, W, toks, variant="right", theta=None):
    """Two-token, one-layer forward with QK-norm written from the definition
    with torch float64 ops: per-head RMSNorm of q and k with their gains,
    then RoPE, then a 2-way softmax for row 1.  ``variant`` plants the
    plausible mistakes the pin must tell apart."""
    T = {k: v.to(torch.float64) for k, v in W.items()}
    bf = lambda t: t.to(torch.bfloat16).to(torch.float64)
    Hq, Hkv, hd, F, eps = spec.n_heads, spec.n_kv_heads, spec.head_dim, spec.ffn_dim, spec.rms_eps
    off = 1.0 if spec.norm_offset else 0.0
    def rms(x, w):
        return bf(x * torch.rsqrt((x * x).mean(-1, keepdim=True) + eps) * (w + off))
    def rope(x, p):  # x [H, hd] at position p, rotate-half
        half = hd // 2
        inv = (theta or spec.rope_theta) ** (-(2.0 * torch.arange(half, dtype=torch.float64)) / hd)
        c, s = torch.cos(p * inv), torch.sin(p * inv)
        return bf(torch.cat([x[:, :half] * c - x[:, half:] * s, x[:, half:] * c + x[:, :half] * s], -1))
    x = T["embed"][torch.from_numpy(np.asarray(toks))]
    a = rms(x, T["layers.0.attn_norm"])
    qkv = bf(a @ T["layers.0.wqkv"].T)
    q = qkv[:, :Hq * hd].reshape(2, Hq, hd)
    k = qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(2, Hkv, hd)
    v = qkv[:, (Hq + Hkv) * hd:].reshape(2, Hkv, hd)
    qn, kn = (T["layers.0.q_norm"], T["layers.0.k_norm"]) if spec.qk_norm else (None, None)
    if not spec.qk_norm:
        q1 = rope(q[1], 1)
        kr = torch.stack([rope(k[0], 0), rope(k[1], 1)])
    elif variant == "right":
        q1 = rope(rms(q[1], qn), 1)
        kr = torch.stack([rope(rms(k[0], kn), 0), rope(rms(k[1], kn), 1)])
    elif variant == "after_rope":
        q1 = rms(rope(q[1], 1), qn)
        kr = torch.stack([rms(rope(k[0], 0), kn), rms(rope(k[1], 1), kn)])
    elif variant == "no_gain":
        one = torch.ones(hd, dtype=torch.float64) - off
        q1 = rope(rms(q[1], one), 1)
        kr = torch.stack([rope(rms(k[0], one), 0), rope(rms(k[1], one), 1)])
    elif variant == "whole_row":  # one norm over all heads of the row
        q1 = rope(rms(q[1].reshape(-1), qn.repeat(Hq)).reshape(Hq, hd), 1)
        kr = torch.stack([rope(rms(k[j].reshape(-1), kn.repeat(Hkv)).reshape(Hkv, hd), j) for j in (0, 1)])
    o = []
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = kr[:, g, :] @ q1[h] / math.sqrt(hd)
        o.append(torch.softmax(s, 0) @ v[:, g, :])
    o = bf(torch.cat(o))
    x1 = bf(x[1] + bf(T["layers.0.wo"] @ o))
    a = rms(x1, T["layers.0.ffn_norm"])
    g = bf(T["layers.0.w_gate_up"][:F] @ a)
    u = bf(T["layers.0.w_gate_up"][F:] @ a)
    act = torch.nn.functional.gelu(g, approximate="tanh") if spec.act == "geglu" else torch.nn.functional.silu(g)
    x2 = bf(x1 + bf(T["layers.0.w_down"] @ bf(act * u)))
    return (T["lm_head"] @ rms(x2, T["final_norm"])).numpy()


QK_SPEC = dict(n_layers=1, qk_norm=True)


def test_qk_norm_two_token_wiring():
    # Row 1 attends to keys 0 and 1, so its logits depend on q and k: the
    # norm must come before RoPE, over each head, with the q_norm / k_norm gains.
    spec, W, dec = _tiny(seed=9, gain_std=0.5, **QK_SPEC)
    toks = np.array([11, 1500])
    want = _qk_reference(spec, W, toks)
    np.testing.assert_allclose(dec.forward(toks), want, rtol=0, atol=1e-9)
    for wrong in ("after_rope", "no_gain", "whole_row"):
        assert np.abs(_qk_reference(spec, W, toks, wrong) - want).max() > 0.05, wrong


LOCAL_THETA = dict(n_layers=1, qk_norm=True, sliding_window=4, local_global_period=1000, rope_theta=1e6, rope_theta_local=50.0)


def test_local_layer_uses_its_own_rope_theta():
    # Layer 0 of a model with a window and period 1000 is local: RoPE there
    # uses rope_theta_local.  Two tokens sit inside the window of 4 keys.
    spec, W, dec = _tiny(seed=10, gain_std=0.5, **LOCAL_THETA)
    toks = np.array([7, 1999])
    want = _qk_reference(spec, W, toks, theta=spec.rope_theta_local)
    np.testing.assert_allclose(dec.forward(toks), want, rtol=0, atol=1e-9)
    assert np.abs(_qk_reference(spec, W, toks, theta=spec.rope_theta) - want).max() > 0.05
