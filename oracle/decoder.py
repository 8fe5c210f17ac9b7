"""The plain float64 decoder forward (test infrastructure).

Follows the definitions cited in ``oracle/__init__.py``:

* ``forward(h)``      -- Forward(W, h) of Theorem 4.1 (深入解析 Vosti §二):
                         last-position logits of a cold causal forward.
* ``fkv(h, p)``       -- fKV(W, h, p) (深入解析 Vosti §五 5.1): the K/V
                         every layer produces at position p.
* ``step(...)``       -- the same forward continued from a given K/V prefix;
                         a cold forward is ``step`` from an empty prefix.
                         With a prefix from ``fkv`` this is the "reuse"
                         path of §五 5.2; with a synthetic prefix it is the
                         decode step over an arbitrary cache.

Per decoder layer (Llama block; Gemma deltas QK-RMSNorm, GeGLU and local
sliding-window layers as named by the model configuration):

    a = rms(x) ; q,k,v = bf16(a Wqkv^T) ; [q,k = bf16(rms_head(q,k))]
    q,k = bf16(rope(q,k)) ; o = bf16(attention) ; h = bf16(o Wo^T)
    [h = rms_post_attn(h)] ; x = bf16(x + h)
    a = rms(x) ; g,u = bf16(a Wgu^T) ; z = bf16(act(g) u) ; h = bf16(z Wd^T)
    [h = rms_post_ffn(h)] ; x = bf16(x + h)
    logits = rms(x_last) W_lm^T           (float64, not rounded)

``rms(x) = bf16(x / sqrt(mean(x^2) + eps) * g)`` with gain g = w, or
g = 1 + w for the Gemma-3 block, which also scales the embeddings by
bf16(sqrt(d)) and adds the bracketed sandwich norms.  The pages name the
Gemma3-4B model but not its block; these three deltas are the published
Gemma 3 architecture, taken as a reading.  RoPE rotates the pairs
(i, i + hd/2) ("rotate half") by angle ``p * theta**(-2i/hd)``; attention
of a row at position p sees keys ``[lo, p]`` with ``lo = 0`` for global
layers and ``max(0, p - w + 1)`` for a window of w keys (深入解析 Vosti
§六 6.2, sliding-window traversal), scale ``1/sqrt(hd)``; query head h
reads KV head ``h // (Hq / Hkv)``.

Pins (tests/test_oracle_decoder.py): RMSNorm of a constant row (closed
form); RoPE identity at p = 0, explicit hd = 2 / hd = 4 rotations and the
relative-position property; attention single-key, equal-key, causal,
window, permutation and GQA-mapping cases plus a two-key closed form;
small-integer projections exact; one-token forward reduced to library
ops; the all-zero model gives zero logits; fKV from a cold forward equals
the K/V inside a longer forward bitwise; incremental == cold logits.
End-to-end logits of a random model beyond those: parity unpinned.
"""

from __future__ import annotations

import math

import numpy as np

from .bf16 import bits_to_f64, round_bf16


def rmsnorm(x, w, eps, offset=0.0):
    """bf16(x / sqrt(mean(x^2) + eps) * (w + offset)) over the last axis, float64 inside."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return round_bf16(x * (1.0 / np.sqrt(ms + eps)) * (w + offset))


def rope(x, positions, theta):
    """Rotate-half RoPE; x: [n, H, hd], positions: [n]; rounded to bf16."""
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = theta ** (-(2.0 * np.arange(half)) / hd)  # [half]
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return round_bf16(np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1))


def layer_is_local(layer: int, window: int, period: int) -> bool:
    """Layer ``layer`` is a local (sliding-window) layer unless the model has
    no window, or no local:global period, or (layer + 1) % period == 0.

    With period 6 this is the 5:1 interleave of the Gemma-3-4B configuration:
    five local layers, then one global layer.
    """
    return window > 0 and period > 0 and (layer + 1) % period != 0


def _visible(p: int, window: int) -> int:
    """First key a row at position p sees (深入解析 Vosti §六 6.2 traversal range)."""
    return max(0, p - window + 1) if window > 0 else 0


def _softmax_row(q_h, Kg, lo, p, hd):
    s = (Kg[lo:p + 1] @ q_h) * (1.0 / math.sqrt(hd))
    e = np.exp(s - s.max())
    return e / e.sum()


def attention_weights(q, K, positions, window):
    """The softmax weights [n, Hq, P] of ``attention`` (0 off the visible range)."""
    n, Hq, hd = q.shape
    rep = Hq // K.shape[1]
    w = np.zeros((n, Hq, K.shape[0]))
    for t in range(n):
        p = int(positions[t])
        lo = _visible(p, window)
        for h in range(Hq):
            w[t, h, lo:p + 1] = _softmax_row(q[t, h], K[:, h // rep, :], lo, p, hd)
    return w


def attention(q, K, V, positions, window, perturb=None):
    """Causal (optionally windowed) GQA softmax attention, rounded to bf16.

    q: [n, Hq, hd] rows at absolute ``positions``; K, V: [P, Hkv, hd] for
    absolute positions 0..P-1 (P > max(positions)).  ``perturb`` (a test
    hook for measuring the noise floor, off by default): a function applied
    to the exact output before its rounding.
    """
    n, Hq, hd = q.shape
    Hkv = K.shape[1]
    rep = Hq // Hkv
    out = np.empty((n, Hq, hd), dtype=np.float64)
    for t in range(n):
        p = int(positions[t])
        lo = _visible(p, window)
        for h in range(Hq):
            g = h // rep
            out[t, h] = _softmax_row(q[t, h], K[:, g, :], lo, p, hd) @ V[lo:p + 1, g, :]
    return round_bf16(out if perturb is None else perturb(out))


def silu(g):
    return g / (1.0 + np.exp(-g))


def gelu_tanh(g):
    return 0.5 * g * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (g + 0.044715 * g ** 3)))


class OracleDecoder:
    """float64 decoder over bf16 weights given as raw uint16 bit arrays.

    ``spec`` is any object with the plain shape fields of a model
    (n_layers, d_model, heads, head_dim, ffn_dim, vocab, rms_eps, act,
    qk_norm, rope_theta, rope_theta_local, sliding_window,
    local_global_period and the Gemma-3 block flags); which layers are
    local is this module's own ``layer_is_local``, not a method of spec.
    """

    def __init__(self, spec, weights_u16: dict, chunk_rows: int = 8192, attention_perturbation=None):
        """``attention_perturbation`` = (rel, seed) is a test hook, off by
        default: every attention output is multiplied by 1 + rel * N(0, 1)
        (a seeded stream) before its bf16 rounding.  With rel = 1e-6 it
        stands for one evaluation of the same definition whose float
        operations round differently at that single site; the spread of the
        logits it causes is the noise floor of a model shape."""
        self.spec = spec
        self._perturb = None
        if attention_perturbation is not None:
            rel, seed = attention_perturbation
            rng = np.random.default_rng(seed)
            self._perturb = lambda o: o * (1.0 + rel * rng.standard_normal(o.shape))
        self.w = weights_u16
        self.chunk_rows = chunk_rows
        self._vec = {}
        self.offset = 1.0 if getattr(spec, "norm_offset", False) else 0.0
        self.embed_scale = bool(getattr(spec, "embed_scale", False))
        self.sandwich = bool(getattr(spec, "sandwich_norm", False))

    def rms(self, x, name):
        return rmsnorm(x, self.vec(name), self.spec.rms_eps, self.offset)

    # -- weights ---------------------------------------------------------
    def vec(self, name):
        if name not in self._vec:
            self._vec[name] = bits_to_f64(self.w[name])
        return self._vec[name]

    def linear(self, name, x):
        """x [n, in] @ W[name]^T in float64 (not rounded); W is [out, in]."""
        W = self.w[name]
        x = np.asarray(x, dtype=np.float64)
        out = np.empty((x.shape[0], W.shape[0]), dtype=np.float64)
        for r0 in range(0, W.shape[0], self.chunk_rows):
            r1 = min(W.shape[0], r0 + self.chunk_rows)
            out[:, r0:r1] = x @ bits_to_f64(W[r0:r1]).T
        return out

    # -- model -----------------------------------------------------------
    def empty_cache(self):
        s = self.spec
        z = np.zeros((0, s.n_kv_heads, s.head_dim))
        return [(z, z) for _ in range(s.n_layers)]

    def step(self, tokens, cache, logit_rows=None):
        """Process ``tokens`` at positions len(cache)..; returns (logits, cache).

        ``cache`` is a per-layer list of (K, V) float64 arrays [c, Hkv, hd]
        holding bf16 values for positions 0..c-1.  ``logit_rows`` selects the
        rows (indices into ``tokens``) whose logits are returned; default
        the last one.  Logits are float64 [len(logit_rows), V].
        """
        s = self.spec
        tokens = np.asarray(tokens, dtype=np.int64)
        n = len(tokens)
        start = cache[0][0].shape[0]
        positions = start + np.arange(n)
        Hq, Hkv, hd, F = s.n_heads, s.n_kv_heads, s.head_dim, s.ffn_dim
        x = bits_to_f64(self.w["embed"][tokens])
        if self.embed_scale:
            x = round_bf16(x * round_bf16(math.sqrt(s.d_model)))
        new_cache = []
        for i in range(s.n_layers):
            p = f"layers.{i}."
            a = self.rms(x, p + "attn_norm")
            qkv = round_bf16(self.linear(p + "wqkv", a))
            q = qkv[:, :Hq * hd].reshape(n, Hq, hd)
            k = qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(n, Hkv, hd)
            v = qkv[:, (Hq + Hkv) * hd:].reshape(n, Hkv, hd)
            if s.qk_norm:
                q = self.rms(q, p + "q_norm")
                k = self.rms(k, p + "k_norm")
            local = layer_is_local(i, getattr(s, "sliding_window", 0), getattr(s, "local_global_period", 0))
            theta = s.rope_theta_local if local else s.rope_theta
            window = s.sliding_window if local else 0
            q = rope(q, positions, theta)
            k = rope(k, positions, theta)
            K = np.concatenate([cache[i][0], k], axis=0)
            V = np.concatenate([cache[i][1], v], axis=0)
            new_cache.append((K, V))
            o = attention(q, K, V, positions, window, self._perturb).reshape(n, Hq * hd)
            h = round_bf16(self.linear(p + "wo", o))
            if self.sandwich:
                h = self.rms(h, p + "post_attn_norm")
            x = round_bf16(x + h)
            a = self.rms(x, p + "ffn_norm")
            gu = round_bf16(self.linear(p + "w_gate_up", a))
            g, u = gu[:, :F], gu[:, F:]
            act = gelu_tanh(g) if s.act == "geglu" else silu(g)
            z = round_bf16(act * u)
            h = round_bf16(self.linear(p + "w_down", z))
            if self.sandwich:
                h = self.rms(h, p + "post_ffn_norm")
            x = round_bf16(x + h)
        rows = [n - 1] if logit_rows is None else list(logit_rows)
        h = self.rms(x[rows], "final_norm")
        return self.linear("lm_head", h), new_cache

    def forward(self, history):
        """Forward(W, h): last-position logits of a cold causal forward."""
        logits, _ = self.step(history, self.empty_cache())
        return logits[0]

    def forward_all(self, history):
        """Logits at every position of one cold forward over ``history``."""
        logits, _ = self.step(history, self.empty_cache(), logit_rows=range(len(history)))
        return logits

    def fkv(self, history, p):
        """fKV(W, h, p): per-layer (k, v) [Hkv, hd] at position p, cold forward over h[:p+1]."""
        _, cache = self.step(np.asarray(history)[:p + 1], self.empty_cache())
        return [(K[p].copy(), V[p].copy()) for K, V in cache]
