"""Host engine: Python face of libvd's native scheduler and block manager.

The scheduling logic lives in C++ (include/vd_engine.h): continuous
batching with chunked prefill, exact-match prefix caching (a rolling hash
only finds candidate pages; reuse needs equal tokens, depth and physical
parent page), prefix hits resolved before new pages are registered,
read-only registered pages, leaf-only eviction and preemption with
recomputation (深入解析 Vosti §三 3.2, §五 5.4).  This module only marshals
arguments and keeps the per-request views of Definition 2.1 (深入解析
Vosti §二): for each request, the list of (logits row, token) it emitted.

An *executor* runs each planned step: ``step(seqs, logit_rows) -> logits``
(seqs: list of (token_ids, cached_len, page_table)) and ``sample(logits,
samplers) -> tokens``.  ``GpuExecutor`` drives libvd.so; ``Engine.run_native``
runs whole steps inside the library instead.
"""

from __future__ import annotations

import collections
import ctypes

import numpy as np

from . import vd

PAGE = 16


EngineConfig, EngineStats, PlanOut = vd.EngineConfig, vd.EngineStats, vd.PlanOut
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)


class RequestInfo:
    def __init__(self, history, prompt_len):
        self.history = [int(t) for t in history]
        self.prompt = np.asarray(self.history[:prompt_len], dtype=np.int32)


class Engine:
    """Continuous batching with chunked prefill over a paged, prefix-sharing pool.

    ``hash_mode=1`` makes every page hash alike (forced collisions, tests).
    """

    def __init__(self, executor, num_pages: int, max_batch: int = 8, token_budget: int = 64,
                 prefix_reuse: bool = True, placement_seed: int | None = None, hash_mode: int = 0):
        self.L = vd.lib()
        self.ex = executor
        cfg = EngineConfig(num_pages, max_batch, token_budget, int(prefix_reuse),
                           -1 if placement_seed is None else placement_seed, hash_mode, 0)
        h = ctypes.c_void_p()
        vd.check(self.L.vd_engine_create(ctypes.byref(cfg), ctypes.byref(h)))
        self.h = h
        self.views: dict = collections.defaultdict(list)   # rid -> [(logits, token)]
        self.rids: list = []

    def close(self):
        if getattr(self, "h", None):
            self.L.vd_engine_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_request(self, prompt, max_new: int, seed: int = 0, temperature: float = 0.0) -> int:
        p = np.ascontiguousarray(prompt, dtype=np.int32)
        rid = ctypes.c_int64()
        vd.check(self.L.vd_engine_add_request(self.h, p.ctypes.data_as(_I32P), len(p), max_new, seed,
                                              temperature, ctypes.byref(rid)))
        self.rids.append(rid.value)
        return rid.value

    def pending(self) -> int:
        return int(self.L.vd_engine_pending(self.h))

    @property
    def stats(self) -> dict:
        st = EngineStats()
        vd.check(self.L.vd_engine_get_stats(self.h, ctypes.byref(st)))
        return {n: int(getattr(st, n)) for n, _ in EngineStats._fields_}

    @property
    def steps(self) -> int:
        return self.stats["steps"]

    def check(self):
        vd.check(self.L.vd_engine_check(self.h))

    def page_info(self, page: int):
        ref, reg = ctypes.c_int32(), ctypes.c_int32()
        vd.check(self.L.vd_engine_page_info(self.h, page, ctypes.byref(ref), ctypes.byref(reg)))
        return ref.value, bool(reg.value)

    def history(self, rid: int) -> RequestInfo:
        n, p = ctypes.c_int32(), ctypes.c_int32()
        vd.check(self.L.vd_engine_history(self.h, rid, None, 0, ctypes.byref(n), ctypes.byref(p)))
        buf = np.zeros(n.value, dtype=np.int32)
        vd.check(self.L.vd_engine_history(self.h, rid, buf.ctypes.data_as(_I32P), n.value, ctypes.byref(n),
                                          ctypes.byref(p)))
        return RequestInfo(buf, p.value)

    @property
    def requests(self) -> dict:
        return {rid: self.history(rid) for rid in self.rids}

    def step(self) -> dict:
        """One engine step through the executor; returns the output record {rid: (logits, token)}."""
        plan = PlanOut()
        vd.check(self.L.vd_engine_plan(self.h, ctypes.byref(plan)))
        b = plan.batch
        if b.num_tokens == 0:
            return {}
        cu = np.ctypeslib.as_array(b.cu_q, (b.num_seqs + 1,)).copy()
        cached = np.ctypeslib.as_array(b.cached_len, (b.num_seqs,)).copy()
        toks = np.ctypeslib.as_array(b.token_ids, (b.num_tokens,)).copy()
        pt = np.ctypeslib.as_array(b.page_table, (b.num_seqs * b.page_table_stride,)).copy()
        pt = pt.reshape(b.num_seqs, b.page_table_stride)
        R = b.num_logit_rows
        rows = np.ctypeslib.as_array(b.logit_rows, (R,)).copy() if R else np.zeros(0, np.int32)
        rids = np.ctypeslib.as_array(plan.rids, (R,)).copy() if R else np.zeros(0, np.int64)
        samplers = [(plan.samplers[i].seed, plan.samplers[i].step, plan.samplers[i].temperature) for i in range(R)]
        seqs = []
        for i in range(b.num_seqs):
            npg = (cached[i] + cu[i + 1] - cu[i] + PAGE - 1) // PAGE
            seqs.append((toks[cu[i]:cu[i + 1]], int(cached[i]), pt[i, :npg]))
        logits = self.ex.step(seqs, rows)
        tokens = np.ascontiguousarray(self.ex.sample(logits, samplers) if R else np.zeros(0), dtype=np.int32)
        vd.check(self.L.vd_engine_commit(self.h, tokens.ctypes.data_as(_I32P)))
        record = {}
        for i in range(R):
            record[int(rids[i])] = (logits[i], int(tokens[i]))
            self.views[int(rids[i])].append((logits[i], int(tokens[i])))
        return record

    def run(self, max_steps: int = 1000000):
        n = 0
        while self.pending() and n < max_steps:
            self.step()
            n += 1
        return self.views

    def run_native(self, model, pool, logits, tokens_dev, keep_logits: bool = False, stream=None,
                   max_steps: int = 1000000, on_step=None):
        """Runs to completion with whole steps inside libvd (plan, step, sample, commit).

        ``on_step(rids, logits_rows, tokens)`` is called after every step that
        emitted rows (logits_rows: the first n rows of ``logits``)."""
        cap = int(tokens_dev.shape[0])
        rids = np.zeros(cap, dtype=np.int64)
        toks = np.zeros(cap, dtype=np.int32)
        n = ctypes.c_int32()
        s = vd._stream(stream)
        steps = 0
        while self.pending() and steps < max_steps:
            vd.check(self.L.vd_engine_run_step(self.h, model.h, pool.h, vd._ptr(logits), vd._ptr(tokens_dev),
                                               rids.ctypes.data_as(_I64P), toks.ctypes.data_as(_I32P),
                                               ctypes.byref(n), s))
            for i in range(n.value):
                self.views[int(rids[i])].append((logits[i].clone() if keep_logits else None, int(toks[i])))
            if on_step is not None and n.value:
                on_step(rids[:n.value].copy(), logits[:n.value], toks[:n.value].copy())
            steps += 1
        return self.views


class GpuExecutor:
    """Executor over libvd.so: logits stay on the device; tokens come back to the host."""

    def __init__(self, model, pool, stream=None):
        import torch
        self.torch = torch
        self.model, self.pool, self.stream = model, pool, stream

    def step(self, seqs, rows):
        torch = self.torch
        V = self.model.spec.vocab
        logits = torch.empty((max(len(rows), 1), V), dtype=torch.float32, device="cuda")
        self.model.step(self.pool, vd.StepBatch(seqs, logit_rows=rows), logits, self.stream)
        return logits[:len(rows)]

    def sample(self, logits, samplers):
        torch = self.torch
        out = torch.empty(len(samplers), dtype=torch.int32, device="cuda")
        self.model.sample(logits, samplers, out, self.stream)
        return out.cpu().numpy()
