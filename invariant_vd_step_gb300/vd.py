"""ctypes binding of libvd.so (include/vd.h, include/vd_ops.h).

Argument marshalling only: every step of the decoder runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams.  There is no
fallback: if libvd.so is missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import torch

from . import build as _build

VD_OK = 0
ERRORS = {1: "VD_ERR_INVALID_ARG", 2: "VD_ERR_UNSUPPORTED", 3: "VD_ERR_OUT_OF_RANGE",
          4: "VD_ERR_CAPACITY", 5: "VD_ERR_CUDA", 6: "VD_ERR_TIMEOUT"}
(VD_ERR_INVALID_ARG, VD_ERR_UNSUPPORTED, VD_ERR_OUT_OF_RANGE, VD_ERR_CAPACITY, VD_ERR_CUDA,
 VD_ERR_TIMEOUT) = range(1, 7)
EPI_BF16, EPI_RESIDUAL, EPI_F32, EPI_SWIGLU, EPI_GEGLU = range(5)


class VDError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class ModelConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("act", ctypes.c_int32),
                ("qk_norm", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("rope_theta_local", ctypes.c_float), ("sliding_window", ctypes.c_int32),
                ("local_global_period", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("max_seqs", ctypes.c_int32),
                ("max_logit_rows", ctypes.c_int32), ("max_context", ctypes.c_int32),
                ("embed_scale", ctypes.c_int32), ("norm_offset", ctypes.c_int32), ("sandwich_norm", ctypes.c_int32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("attn_norm", "wqkv", "q_norm", "k_norm", "wo", "ffn_norm", "w_gate_up", "w_down",
                 "post_attn_norm", "post_ffn_norm")]


class WeightPtrs(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("layers", ctypes.POINTER(LayerWeights)),
                ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p)]


_I32P = ctypes.POINTER(ctypes.c_int32)


class Batch(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
                ("num_logit_rows", ctypes.c_int32), ("page_table_stride", ctypes.c_int32),
                ("token_ids", _I32P), ("positions", _I32P), ("cu_q", _I32P), ("cached_len", _I32P),
                ("page_table", _I32P), ("logit_rows", _I32P)]


class Sampler(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_uint64), ("step", ctypes.c_uint64), ("temperature", ctypes.c_float),
                ("pad_", ctypes.c_float)]


class KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int32), ("kernels", ctypes.c_int32),
                ("total_ms", ctypes.c_double)]


class EngineConfig(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("max_batch", ctypes.c_int32), ("token_budget", ctypes.c_int32),
                ("prefix_reuse", ctypes.c_int32), ("placement_seed", ctypes.c_int64),
                ("hash_mode", ctypes.c_int32), ("pad_", ctypes.c_int32)]


class EngineStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("steps", "prefix_hit_pages", "registered", "evicted", "preempted", "hash_candidates_rejected")]


class PlanOut(ctypes.Structure):
    _fields_ = [("batch", Batch), ("rids", ctypes.POINTER(ctypes.c_int64)),
                ("samplers", ctypes.POINTER(Sampler))]


_VP = ctypes.c_void_p
_I64P = ctypes.POINTER(ctypes.c_int64)
_SIGS = {
    "vd_create_model": (ctypes.c_int, [ctypes.POINTER(ModelConfig), ctypes.POINTER(WeightPtrs), ctypes.POINTER(_VP)]),
    "vd_destroy_model": (None, [_VP]),
    "vd_kv_pool_bytes": (ctypes.c_size_t, [_VP, ctypes.c_int32]),
    "vd_kv_pool_alloc": (ctypes.c_int, [_VP, ctypes.c_int32, _VP, ctypes.c_size_t, ctypes.POINTER(_VP)]),
    "vd_destroy_kv_pool": (None, [_VP]),
    "vd_kv_pool_data": (_VP, [_VP]),
    "vd_step": (ctypes.c_int, [_VP, _VP, ctypes.POINTER(Batch), _VP, _VP]),
    "vd_sample": (ctypes.c_int, [_VP, _VP, ctypes.c_int32, ctypes.POINTER(Sampler), _VP, _VP]),
    "vd_step_sample": (ctypes.c_int, [_VP, _VP, ctypes.POINTER(Batch), ctypes.POINTER(Sampler), _VP, _VP, _VP]),
    "vd_step_sample_fed": (ctypes.c_int, [_VP, _VP, ctypes.POINTER(Batch), _I32P, _VP, ctypes.POINTER(Sampler), _VP,
                                          _VP, _VP]),
    "vd_copy_kv": (ctypes.c_int, [_VP, _VP, ctypes.c_int32, _I32P, ctypes.c_int32, _VP, _VP, _VP]),
    "vd_device_status": (ctypes.c_int, [_VP]),
    "vd_set_graph_mode": (ctypes.c_int, [_VP, ctypes.c_int32]),
    "vd_set_attention_fold": (ctypes.c_int, [_VP, ctypes.c_int32]),
    "vd_set_attention_prefill": (ctypes.c_int, [_VP, ctypes.c_int32]),
    "vd_set_reduction_mode": (ctypes.c_int, [_VP, ctypes.c_int32]),
    "vd_graph_stats": (ctypes.c_int, [_VP, _I64P]),
    "vd_profile_enable": (ctypes.c_int, [_VP, ctypes.c_int32]),
    "vd_profile_collect": (ctypes.c_int, [_VP, ctypes.POINTER(KernelStat), ctypes.c_int32]),
    "vd_last_error": (ctypes.c_char_p, []),
    "vd_version": (ctypes.c_char_p, []),
    "vd_op_gemm": (ctypes.c_int, [_VP, _VP, _VP, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                  _VP, _VP]),
    "vd_set_gemm_plan": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    "vd_gemm_shape_check": (ctypes.c_int, []),
    "vd_gemm_plan_query": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.POINTER(ctypes.c_int32)]),
    "vd_op_rmsnorm": (ctypes.c_int, [_VP, _VP, _VP, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, _VP]),
    "vd_op_attention": (ctypes.c_int, [_VP, _VP, ctypes.c_int32, ctypes.POINTER(Batch), _VP, _VP, _VP]),
    "vd_op_rope_kv": (ctypes.c_int, [_VP, _VP, ctypes.c_int32, ctypes.POINTER(Batch), _VP, _VP, _VP]),
    "vd_op_attention_static": (ctypes.c_int, [_VP, _VP, ctypes.c_int32, ctypes.POINTER(Batch), _VP, _VP, _VP]),
    "vd_op_philox": (ctypes.c_int, [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int32, _VP, _VP]),
    "vd_op_wait_probe": (ctypes.c_int, [_VP, ctypes.c_int32, _VP, _VP]),
    "vd_op_tma_stream": (ctypes.c_int, [_VP, ctypes.c_int64, ctypes.c_int64, _VP, ctypes.c_int64, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _VP]),
    "vd_op_mma_issue_probe": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _VP, _VP]),
    "vd_engine_create": (ctypes.c_int, [ctypes.POINTER(EngineConfig), ctypes.POINTER(_VP)]),
    "vd_engine_destroy": (None, [_VP]),
    "vd_engine_add_request": (ctypes.c_int, [_VP, _I32P, ctypes.c_int32, ctypes.c_int32, ctypes.c_uint64,
                                             ctypes.c_float, _I64P]),
    "vd_engine_plan": (ctypes.c_int, [_VP, ctypes.POINTER(PlanOut)]),
    "vd_engine_commit": (ctypes.c_int, [_VP, _I32P]),
    "vd_engine_run_step": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _I64P, _I32P, _I32P, _VP]),
    "vd_engine_pending": (ctypes.c_int, [_VP]),
    "vd_engine_get_stats": (ctypes.c_int, [_VP, ctypes.POINTER(EngineStats)]),
    "vd_engine_check": (ctypes.c_int, [_VP]),
    "vd_engine_page_info": (ctypes.c_int, [_VP, ctypes.c_int32, _I32P, _I32P]),
    "vd_engine_history": (ctypes.c_int, [_VP, ctypes.c_int64, _I32P, ctypes.c_int32, _I32P, _I32P]),
}

_LIB = None


def header_symbols() -> set:
    """Every function name declared in include/*.h."""
    names = set()
    inc = os.path.join(_build.ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            txt = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"\b(vd_[a-z0-9_]+)\s*\(", txt))
    return names


def lib():
    """The loaded libvd.so; raises if it is missing (no fallback path exists)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libvd.so not built ({_build.LIB}); run __graft_entry__.build()")
        L = ctypes.CDLL(_build.LIB)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def check(rc: int):
    if rc != VD_OK:
        raise VDError(rc, lib().vd_last_error().decode())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(_I32P)


def config_of(spec, max_tokens: int, max_seqs: int, max_logit_rows: int, max_context: int) -> ModelConfig:
    return ModelConfig(
        n_layers=spec.n_layers, d_model=spec.d_model, n_heads=spec.n_heads, n_kv_heads=spec.n_kv_heads,
        head_dim=spec.head_dim, ffn_dim=spec.ffn_dim, vocab=spec.vocab, rms_eps=spec.rms_eps,
        act=1 if spec.act == "geglu" else 0, qk_norm=int(spec.qk_norm), rope_theta=spec.rope_theta,
        rope_theta_local=spec.rope_theta_local, sliding_window=spec.sliding_window,
        local_global_period=spec.local_global_period, page_size=spec.page_size, max_tokens=max_tokens,
        max_seqs=max_seqs, max_logit_rows=max_logit_rows, max_context=max_context,
        embed_scale=int(getattr(spec, "embed_scale", False)), norm_offset=int(getattr(spec, "norm_offset", False)),
        sandwich_norm=int(getattr(spec, "sandwich_norm", False)))


class StepBatch:
    """Host descriptor of one engine step (vd_batch), built from numpy arrays.

    ``seqs`` is a list of (token_ids, cached_len, page_table) for the
    requests of the step; ``logit_rows`` are token indices into the
    concatenated token list.
    """

    def __init__(self, seqs, logit_rows=()):
        toks, pos, cu, cached = [], [], [0], []
        width = max((len(pt) for _, _, pt in seqs), default=1)
        pt_all = np.zeros((max(len(seqs), 1), max(width, 1)), dtype=np.int32)
        for i, (t, c, pt) in enumerate(seqs):
            t = np.asarray(t, dtype=np.int32)
            toks.append(t)
            pos.append(c + np.arange(len(t), dtype=np.int32))
            cu.append(cu[-1] + len(t))
            cached.append(c)
            pt_all[i, :len(pt)] = pt
        cat = lambda xs: np.concatenate(xs).astype(np.int32) if xs else np.zeros(0, np.int32)
        self.tokens, p_tok = _i32(cat(toks))
        self.positions, p_pos = _i32(cat(pos))
        self.cu_q, p_cu = _i32(cu)
        self.cached, p_c = _i32(cached)
        self.page_table, p_pt = _i32(pt_all)
        self.logit_rows, p_lr = _i32(np.asarray(logit_rows, dtype=np.int32))
        self.c = Batch(len(self.tokens), len(seqs), len(self.logit_rows), pt_all.shape[1],
                       p_tok, p_pos, p_cu, p_c, p_pt, p_lr)

    @classmethod
    def from_arrays(cls, token_ids, cu_q, cached_len, page_table, logit_rows=()):
        """Builds the descriptor from ready numpy arrays (no per-request loop).

        page_table is [B][stride]; positions are derived as cached_len + offset.
        """
        self = cls.__new__(cls)
        self.tokens, p_tok = _i32(token_ids)
        self.cu_q, p_cu = _i32(cu_q)
        self.cached, p_c = _i32(cached_len)
        qlen = np.diff(self.cu_q)
        seq = np.repeat(np.arange(len(qlen), dtype=np.int32), qlen)
        self.positions, p_pos = _i32(self.cached[seq] + (np.arange(len(self.tokens), dtype=np.int32)
                                                         - self.cu_q[:-1][seq]))
        pt = np.ascontiguousarray(page_table, dtype=np.int32)
        if pt.ndim == 1:
            pt = pt.reshape(len(qlen), -1)
        self.page_table, p_pt = _i32(pt)
        self.logit_rows, p_lr = _i32(np.asarray(logit_rows, dtype=np.int32))
        self.c = Batch(len(self.tokens), len(qlen), len(self.logit_rows), pt.shape[1],
                       p_tok, p_pos, p_cu, p_c, p_pt, p_lr)
        return self

    @property
    def num_tokens(self):
        return int(self.c.num_tokens)

    @property
    def num_logit_rows(self):
        return int(self.c.num_logit_rows)


class Model:
    """A model over borrowed torch bf16 CUDA weights (see synth.weight_shapes)."""

    def __init__(self, spec, weights: dict, max_tokens: int = 512, max_seqs: int = 64,
                 max_logit_rows: int = 256, max_context: int = 4096):
        L = lib()
        self.spec = spec
        self.weights = weights  # keep alive
        self.cfg = config_of(spec, max_tokens, max_seqs, max_logit_rows, max_context)
        layers = (LayerWeights * spec.n_layers)()
        for i in range(spec.n_layers):
            p = f"layers.{i}."
            g = lambda n: _ptr(weights.get(p + n))
            layers[i] = LayerWeights(g("attn_norm"), g("wqkv"), g("q_norm"), g("k_norm"), g("wo"), g("ffn_norm"),
                                     g("w_gate_up"), g("w_down"), g("post_attn_norm"), g("post_ffn_norm"))
        self._layers = layers
        w = WeightPtrs(_ptr(weights["embed"]), layers, _ptr(weights["final_norm"]), _ptr(weights["lm_head"]))
        h = ctypes.c_void_p()
        check(L.vd_create_model(ctypes.byref(self.cfg), ctypes.byref(w), ctypes.byref(h)))
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            lib().vd_destroy_model(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def pool_bytes(self, num_pages: int) -> int:
        return int(lib().vd_kv_pool_bytes(self.h, num_pages))

    def step(self, pool: "KVPool", batch: StepBatch, logits: torch.Tensor, stream=None):
        check(lib().vd_step(self.h, pool.h, ctypes.byref(batch.c), _ptr(logits), _stream(stream)))

    def sample(self, logits: torch.Tensor, samplers, tokens_out: torch.Tensor, stream=None):
        R = len(samplers)
        arr = (Sampler * max(R, 1))()
        for i, (seed, step, temp) in enumerate(samplers):
            arr[i] = Sampler(seed, step, temp, 0.0)
        check(lib().vd_sample(self.h, _ptr(logits), R, arr, _ptr(tokens_out), _stream(stream)))

    def step_sample(self, pool: "KVPool", batch: StepBatch, samplers, logits, tokens_out: torch.Tensor,
                    stream=None):
        """vd_step_sample: one step with the token choice fused into the LM head (logits may be None)."""
        R = len(samplers)
        arr = (Sampler * max(R, 1))()
        for i, (seed, step, temp) in enumerate(samplers):
            arr[i] = Sampler(seed, step, temp, 0.0)
        check(lib().vd_step_sample(self.h, pool.h, ctypes.byref(batch.c), arr, _ptr(logits), _ptr(tokens_out),
                                   _stream(stream)))

    def step_sample_fed(self, pool: "KVPool", batch: StepBatch, feed_index, feed_tokens: torch.Tensor, samplers,
                        logits, tokens_out: torch.Tensor, stream=None):
        """vd_step_sample_fed: tokens with feed_index[t] >= 0 come from feed_tokens on the device."""
        R = len(samplers)
        arr = (Sampler * max(R, 1))()
        for i, (seed, step, temp) in enumerate(samplers):
            arr[i] = Sampler(seed, step, temp, 0.0)
        fi, fip = _i32(feed_index)
        check(lib().vd_step_sample_fed(self.h, pool.h, ctypes.byref(batch.c), fip,
                                       _ptr(feed_tokens), arr, _ptr(logits), _ptr(tokens_out), _stream(stream)))

    def copy_kv(self, pool: "KVPool", layer: int, page_table, n_tokens: int, out_k, out_v, stream=None):
        pt, p = _i32(page_table)
        check(lib().vd_copy_kv(self.h, pool.h, layer, p, n_tokens, _ptr(out_k), _ptr(out_v), _stream(stream)))

    def attention(self, pool, layer, batch: StepBatch, q, out, stream=None):
        check(lib().vd_op_attention(self.h, pool.h, layer, ctypes.byref(batch.c), _ptr(q), _ptr(out),
                                    _stream(stream)))

    def attention_static(self, pool, layer, batch: StepBatch, q, out, stream=None):
        """vd_op_attention_static: attention whose scratch is a fixed array in libvd.so (no allocation)."""
        check(lib().vd_op_attention_static(self.h, pool.h, layer, ctypes.byref(batch.c), _ptr(q), _ptr(out),
                                           _stream(stream)))

    def rope_kv(self, pool, layer, batch: StepBatch, qkv, q_out, stream=None):
        check(lib().vd_op_rope_kv(self.h, pool.h, layer, ctypes.byref(batch.c), _ptr(qkv), _ptr(q_out),
                                  _stream(stream)))

    def wait_probe(self, limit_us: int, out=None, stream=None):
        """vd_op_wait_probe: one bounded wait that nothing completes (records VD_ERR_TIMEOUT)."""
        check(lib().vd_op_wait_probe(self.h, int(limit_us), _ptr(out), _stream(stream)))

    def device_status(self) -> int:
        return int(lib().vd_device_status(self.h))

    def profile(self, on: bool):
        check(lib().vd_profile_enable(self.h, int(on)))

    def set_reduction_mode(self, mode: int):
        """0: batch-invariant steps (default); 1: fast split-K steps (not invariant; verify them)."""
        check(lib().vd_set_reduction_mode(self.h, int(mode)))

    def set_attention_fold(self, mode: int):
        """Decode attention mapping: 0 default (one CTA per split), 1 fold all splits in one CTA, 2 split."""
        check(lib().vd_set_attention_fold(self.h, int(mode)))

    def set_attention_prefill(self, kernel: int):
        """Prefill-class attention kernel: 0 default (tcgen05), 1 mma.sync."""
        check(lib().vd_set_attention_prefill(self.h, int(kernel)))

    def set_graph_mode(self, max_graphs: int):
        """Replay steps as captured CUDA graphs (0 = eager launches)."""
        check(lib().vd_set_graph_mode(self.h, int(max_graphs)))

    def graph_stats(self) -> dict:
        out = (ctypes.c_int64 * 4)()
        check(lib().vd_graph_stats(self.h, out))
        return {"captures": int(out[0]), "replays": int(out[1]), "cached": int(out[2]), "eager": int(out[3])}

    def profile_collect(self) -> dict:
        arr = (KernelStat * 32)()
        n = lib().vd_profile_collect(self.h, arr, 32)
        if n < 0:
            check(n)
        return {arr[i].name.decode(): (int(arr[i].launches), int(arr[i].kernels), float(arr[i].total_ms))
                for i in range(n)}


class KVPool:
    def __init__(self, model: Model, num_pages: int, memory: torch.Tensor | None = None):
        self.model = model
        self.num_pages = num_pages
        nbytes = model.pool_bytes(num_pages)
        self.memory = memory  # keep alive when caller-owned
        h = ctypes.c_void_p()
        ptr = _ptr(memory) if memory is not None else None
        check(lib().vd_kv_pool_alloc(model.h, num_pages, ptr, nbytes if memory is not None else 0,
                                     ctypes.byref(h)))
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            lib().vd_destroy_kv_pool(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def data_ptr(self) -> int:
        return int(lib().vd_kv_pool_data(self.h) or 0)

    def view(self) -> torch.Tensor:
        """The pool as a bf16 tensor [layers][pages][2][Hkv][16][hd] (requires caller memory)."""
        s = self.model.spec
        if self.memory is None:
            raise RuntimeError("view() needs a pool created over caller memory")
        return self.memory.view(torch.bfloat16)[: s.n_layers * self.num_pages * 2 * s.n_kv_heads * 16 * s.head_dim] \
            .view(s.n_layers, self.num_pages, 2, s.n_kv_heads, 16, s.head_dim)


def gemm(A, W, C, epilogue=EPI_BF16, residual=None, stream=None):
    T, K = A.shape
    N = C.shape[1]
    check(lib().vd_op_gemm(_ptr(A), _ptr(W), _ptr(C), T, N, K, epilogue, _ptr(residual), _stream(stream)))


def gemm_shape_check() -> int:
    """vd_gemm_shape_check: 1 if every GEMM tile shape gave the same bits on this device, 0 if shapes are pinned."""
    return int(lib().vd_gemm_shape_check())


def set_gemm_plan(bm=0, bn=0, kpo=0):
    """Process-wide GEMM launch shape override (0: chosen per launch); changes speed only."""
    check(lib().vd_set_gemm_plan(bm, bn, kpo))


def gemm_plan(T, N, K, epilogue=EPI_BF16):
    """(bm, bn, kpo) that a GEMM launch over T tokens takes (epilogue 5: LM head with token choice)."""
    out = (ctypes.c_int32 * 3)()
    check(lib().vd_gemm_plan_query(T, N, K, epilogue, out))
    return tuple(out)


def tma_stream(w, box_rows, kpo, x=None, x_box_rows=0, k_parts=1, ctas=0, stream=None):
    """vd_op_tma_stream: stream the bf16 matrix w [rows][K] through shared memory with a GEMM plan's copies."""
    rows, K = w.shape
    x_rows = x.shape[0] if x is not None else 0
    check(lib().vd_op_tma_stream(_ptr(w), rows, K, _ptr(x), x_rows, box_rows, kpo, x_box_rows, k_parts, ctas,
                                 _stream(stream)))


def mma_issue_probe(M, N, n_mma, wait, out, stream=None):
    """vd_op_mma_issue_probe: out (dev int64 [2]) = cycles to the last MMA issue and to completion."""
    check(lib().vd_op_mma_issue_probe(M, N, n_mma, wait, _ptr(out), _stream(stream)))


def rmsnorm(x, w, y, eps, stream=None):
    rows, d = x.shape
    check(lib().vd_op_rmsnorm(_ptr(x), _ptr(w), _ptr(y), rows, d, eps, _stream(stream)))


def philox(seed: int, step: int, n: int, out, stream=None):
    check(lib().vd_op_philox(seed, step, n, _ptr(out), _stream(stream)))
