"""ctypes binding of the float32 C++ oracle (test infrastructure only).

``Fp32Decoder`` has the interface of ``oracle.decoder.OracleDecoder`` (the
float64 numpy oracle, kept as an independent cross-check): ``step``,
``forward``, ``forward_all``, ``fkv``.  Its cache is a ``KVCache`` of bf16
bit patterns; ``KVCache.from_values`` / ``from_bits`` take the numpy
oracle's per-layer (K, V) list or raw bits.  The arithmetic is all in
``fp32_decoder.cpp``; this module only marshals arrays.  The layer rule
(local windowed layers versus global ones) is the C++ oracle's own, taken
from the model's window and local:global period, not from any helper of
the product package.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

_F = ctypes.POINTER(ctypes.c_float)
_U16 = ctypes.POINTER(ctypes.c_uint16)
_I32 = ctypes.POINTER(ctypes.c_int32)
_I64 = ctypes.c_int64


class OcSpec(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim", "ffn_dim", "vocab",
        "act", "qk_norm", "embed_scale", "norm_offset", "sandwich_norm",
        "sliding_window", "local_global_period")] + [
        ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_double), ("rope_theta_local", ctypes.c_double)]


def lib():
    global _LIB
    if _LIB is None:
        _LIB = ctypes.CDLL(_build.build())
        L = _LIB
        L.oc_layer_is_local.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.oc_round_bf16.argtypes = [_F, _F, _I64]
        L.oc_rmsnorm.argtypes = [_F, _I64, ctypes.c_int, _F, ctypes.c_float, ctypes.c_int, ctypes.c_int, _F]
        L.oc_linear.argtypes = [_F, _I64, ctypes.c_int, _U16, ctypes.c_int, _F, ctypes.c_int]
        L.oc_rope.argtypes = [_F, _I64, ctypes.c_int, ctypes.c_int, _I32, ctypes.c_double, ctypes.c_int, _F]
        L.oc_attention.argtypes = [_F, _I64, ctypes.c_int, ctypes.c_int, _U16, _U16, _I64, ctypes.c_int, _I32,
                                   ctypes.c_int, ctypes.c_int, _F, _F, ctypes.c_int]
        L.oc_glu.argtypes = [_F, _F, _I64, ctypes.c_int, _F]
        L.oc_step.argtypes = [ctypes.POINTER(OcSpec), ctypes.POINTER(_U16), _I32, _I64, _I64, _U16, _U16, _I64,
                              _I32, _I64, _F, ctypes.c_int]
        L.oc_step.restype = ctypes.c_int
    return _LIB


def default_threads() -> int:
    return int(os.environ.get("ORACLE_THREADS", os.cpu_count() or 1))


def _f32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _p(a, t):
    return a.ctypes.data_as(t)


def to_bits(values) -> np.ndarray:
    """bf16-valued floats -> uint16 bit patterns (values must already be bf16)."""
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float32))
    u = v.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "values are not bf16"
    return (u >> 16).astype(np.uint16)


def from_bits(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------ modules
def layer_is_local(layer: int, window: int, period: int) -> bool:
    return bool(lib().oc_layer_is_local(layer, window, period))


def round_bf16(x) -> np.ndarray:
    x = _f32(x)
    y = np.empty_like(x)
    lib().oc_round_bf16(_p(x, _F), _p(y, _F), x.size)
    return y


def rmsnorm(x, w, eps, offset=False, round=True) -> np.ndarray:
    """Over the last axis; float32 in and out."""
    x = _f32(x)
    w = _f32(w)
    d = x.shape[-1]
    y = np.empty_like(x)
    lib().oc_rmsnorm(_p(x, _F), x.size // d, d, _p(w, _F), eps, int(offset), int(round), _p(y, _F))
    return y


def linear(x, W_bits, threads=None) -> np.ndarray:
    """x [n, K] (float32, bf16 values) times W^T, W bf16 bits [N, K]; float32 [n, N], not rounded."""
    x = _f32(x)
    W = np.ascontiguousarray(W_bits, dtype=np.uint16)
    n, K = x.shape
    N = W.shape[0]
    assert W.shape[1] == K
    y = np.empty((n, N), dtype=np.float32)
    lib().oc_linear(_p(x, _F), n, K, _p(W, _U16), N, _p(y, _F), threads or default_threads())
    return y


def rope(x, positions, theta, round=True) -> np.ndarray:
    """x [n, H, hd] float32."""
    x = _f32(x)
    n, H, hd = x.shape
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    y = np.empty_like(x)
    lib().oc_rope(_p(x, _F), n, H, hd, _p(pos, _I32), float(theta), int(round), _p(y, _F))
    return y


def attention(q, K_bits, V_bits, positions, window=0, round=True, probs=False, threads=None):
    """q [n, Hq, hd] float32; K/V bf16 bits [P, Hkv, hd].  Returns out (and the softmax weights [n, Hq, P])."""
    q = _f32(q)
    K = np.ascontiguousarray(K_bits, dtype=np.uint16)
    V = np.ascontiguousarray(V_bits, dtype=np.uint16)
    n, Hq, hd = q.shape
    P, Hkv, _ = K.shape
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    assert pos.size == n and (n == 0 or pos.max() < P)
    out = np.empty_like(q)
    pr = np.empty((n, Hq, P), dtype=np.float32) if probs else None
    lib().oc_attention(_p(q, _F), n, Hq, hd, _p(K, _U16), _p(V, _U16), P, Hkv, _p(pos, _I32), int(window),
                       int(round), _p(out, _F), _p(pr, _F) if probs else None, threads or default_threads())
    return (out, pr) if probs else out


def glu(g, u, act) -> np.ndarray:
    g, u = _f32(g), _f32(u)
    z = np.empty_like(g)
    lib().oc_glu(_p(g, _F), _p(u, _F), g.size, 1 if act == "geglu" else 0, _p(z, _F))
    return z


# ------------------------------------------------------------ model
class KVCache:
    """bf16 K and V bit patterns [n_layers][length][Hkv][hd]."""

    def __init__(self, K: np.ndarray, V: np.ndarray):
        self.K, self.V = K, V

    @property
    def length(self) -> int:
        return self.K.shape[1]

    @classmethod
    def empty(cls, n_layers, n_kv_heads, head_dim):
        z = np.zeros((n_layers, 0, n_kv_heads, head_dim), dtype=np.uint16)
        return cls(z, z.copy())

    @classmethod
    def from_bits(cls, kv_bits):
        """[(K bits [c, Hkv, hd], V bits)] per layer."""
        return cls(np.stack([np.asarray(k, np.uint16) for k, _ in kv_bits]),
                   np.stack([np.asarray(v, np.uint16) for _, v in kv_bits]))

    @classmethod
    def from_values(cls, kv):
        """The float64 oracle's cache: [(K [c, Hkv, hd], V)] of bf16 values."""
        return cls.from_bits([(to_bits(k), to_bits(v)) for k, v in kv])

    def values(self):
        """Per-layer (K, V) float64 arrays, the float64 oracle's cache form."""
        return [(from_bits(self.K[l]).astype(np.float64), from_bits(self.V[l]).astype(np.float64))
                for l in range(self.K.shape[0])]


class Fp32Decoder:
    """The float32 C++ decoder over bf16 weights given as raw uint16 bit arrays.

    ``spec`` is any object with the attributes of a model shape
    (n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab,
    rms_eps, act, qk_norm, rope_theta, rope_theta_local, sliding_window,
    local_global_period, embed_scale, norm_offset, sandwich_norm); only
    plain fields are read.
    """

    def __init__(self, spec, weights_u16: dict, threads=None):
        self.spec = spec
        self.threads = threads or default_threads()
        g = lambda k, dflt=False: getattr(spec, k, dflt)
        self.cspec = OcSpec(spec.n_layers, spec.d_model, spec.n_heads, spec.n_kv_heads, spec.head_dim,
                            spec.ffn_dim, spec.vocab, 1 if spec.act == "geglu" else 0, int(g("qk_norm")),
                            int(g("embed_scale")), int(g("norm_offset")), int(g("sandwich_norm")),
                            int(g("sliding_window", 0)), int(g("local_global_period", 0)), float(spec.rms_eps),
                            float(spec.rope_theta), float(g("rope_theta_local", spec.rope_theta)))
        names = ["embed", "final_norm", "lm_head"]
        for i in range(spec.n_layers):
            p = f"layers.{i}."
            names += [p + s for s in ("attn_norm", "wqkv", "q_norm", "k_norm", "wo", "post_attn_norm",
                                      "ffn_norm", "w_gate_up", "w_down", "post_ffn_norm")]
        self._keep = []
        table = (_U16 * len(names))()
        for i, n in enumerate(names):
            if n in weights_u16:
                a = np.ascontiguousarray(weights_u16[n], dtype=np.uint16)
                self._keep.append(a)
                table[i] = _p(a, _U16)
            else:
                table[i] = None
        self.table = table
        for req in ("embed", "final_norm", "lm_head"):
            assert req in weights_u16, req

    def empty_cache(self) -> KVCache:
        s = self.spec
        return KVCache.empty(s.n_layers, s.n_kv_heads, s.head_dim)

    def step(self, tokens, cache, logit_rows=None):
        """Process ``tokens`` at positions cache.length ..; returns (logits float64 [R, V], new cache).

        ``cache`` is a ``KVCache`` or the float64 oracle's per-layer (K, V)
        list; the returned cache is a new ``KVCache`` (the input is unchanged).
        """
        if not isinstance(cache, KVCache):
            cache = KVCache.from_values(cache)
        s = self.spec
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        n = toks.size
        start = cache.length
        cap = start + n
        shape = (s.n_layers, cap, s.n_kv_heads, s.head_dim)
        K = np.zeros(shape, dtype=np.uint16)
        V = np.zeros(shape, dtype=np.uint16)
        K[:, :start] = cache.K
        V[:, :start] = cache.V
        rows = np.ascontiguousarray([n - 1] if logit_rows is None else list(logit_rows), dtype=np.int32)
        out = np.empty((rows.size, s.vocab), dtype=np.float32)
        rc = lib().oc_step(ctypes.byref(self.cspec), self.table, _p(toks, _I32), n, start, _p(K, _U16),
                           _p(V, _U16), cap, _p(rows, _I32), rows.size, _p(out, _F), self.threads)
        if rc != 0:
            raise ValueError("oracle step: bad arguments")
        return out.astype(np.float64), KVCache(K, V)

    def forward(self, history):
        """Forward(W, h): the last position's logits of a cold causal forward."""
        return self.step(history, self.empty_cache())[0][0]

    def forward_all(self, history):
        """Logits at every position of one cold forward over ``history``."""
        return self.step(history, self.empty_cache(), logit_rows=range(len(history)))[0]

    def fkv(self, history, p):
        """fKV(W, h, p): per-layer (k, v) bf16 values [Hkv, hd] at position p of a cold forward over h[:p+1]."""
        _, cache = self.step(np.asarray(history)[:p + 1], self.empty_cache(), logit_rows=[])
        return [(from_bits(cache.K[l, p]).astype(np.float64), from_bits(cache.V[l, p]).astype(np.float64))
                for l in range(self.spec.n_layers)]
