"""Multi-turn sessions served through the native engine.

A session is a conversation: turn k submits the whole history so far (the
previous turns' prompts and outputs plus the new turn's tokens) as one
request, and the engine reuses whatever prefix pages are still cached
(深入解析 Vosti §三 3.2, prefix caching with exact matching; §五 5.4,
recomputation after eviction).  Everything a turn appends or decodes is a
function of (session, turn) alone, so a session's outputs may not depend on
which other sessions run beside it, on the pool size or on the order turns
finish in: the property the agentic workload checks.

The loop is plan -> vd_step_sample (token choice fused into the LM head) ->
tokens to the host -> commit, with the descriptors and sampler states the
engine plans handed to the library as they are.
"""

from __future__ import annotations

import collections
import ctypes
import time
from dataclasses import dataclass, field

import numpy as np

from . import synth, vd


@dataclass
class SessionWorkload:
    """n_sessions sessions of `turns` turns.

    Turn 0 starts from ``prefix`` (shared by every session) or from
    ``prompts[sid]``; every turn then appends U[append_lo, append_hi] tokens
    (none if append_hi == 0) and decodes U[decode_lo, decode_hi] tokens.
    """

    vocab: int
    n_sessions: int
    turns: int
    append_lo: int = 0
    append_hi: int = 0
    decode_lo: int = 16
    decode_hi: int = 16
    prefix: np.ndarray | None = None
    prompts: list | None = None
    seed: int = 7
    temperature: float = 0.0

    def turn(self, sid: int, k: int) -> tuple[np.ndarray, int]:
        """(tokens appended by turn k of session sid, tokens it decodes)."""
        rng = np.random.default_rng([self.seed, sid, k])
        n_add = int(rng.integers(self.append_lo, self.append_hi + 1)) if self.append_hi else 0
        add = synth.make_tokens(n_add, self.vocab, seed=100000 + sid * 64 + k) if n_add else np.zeros(0, np.int32)
        return add, int(rng.integers(self.decode_lo, self.decode_hi + 1))

    def start_history(self, sid: int) -> np.ndarray:
        if self.prompts is not None:
            return np.asarray(self.prompts[sid], dtype=np.int32)
        if self.prefix is not None:
            return np.asarray(self.prefix, dtype=np.int32)
        return np.zeros(0, np.int32)

    def max_context(self) -> int:
        base = max((len(p) for p in self.prompts), default=0) if self.prompts is not None else \
            (len(self.prefix) if self.prefix is not None else 0)
        return base + self.turns * (self.append_hi + self.decode_hi) + 16


@dataclass
class StepInfo:
    seqs: list            # (cached_len, q_len) per request
    rows: int             # logit rows
    seconds: float        # host wall time of the step (it ends with a stream sync)


@dataclass
class SessionResult:
    outputs: dict = field(default_factory=dict)   # sid -> [[tokens of turn 0], [turn 1], ...]
    submitted: int = 0                            # prompt tokens submitted (cache hits included)
    steps: list = field(default_factory=list)     # StepInfo per engine step


def run_sessions(work: SessionWorkload, model, pool, eng, concurrency: int, logits, tokens_dev, stream=None,
                 on_rows=None, only=None) -> SessionResult:
    """Serves the sessions in `only` (default: all) with at most `concurrency`
    turns in flight.  ``on_rows(sids, turns, logits_rows, tokens)`` sees every
    step's emitted rows (logits_rows: the first R rows of `logits`)."""
    import torch

    lib = vd.lib()
    s = vd._stream(stream)
    sids = list(range(work.n_sessions)) if only is None else list(only)
    hist = {sid: work.start_history(sid) for sid in sids}
    turn = {sid: 0 for sid in sids}
    res = SessionResult(outputs={sid: [] for sid in sids})
    rid_of = {}                      # rid -> (sid, turn, max_new)
    got = collections.defaultdict(list)
    queue = collections.deque(sids)
    cap = int(tokens_dev.shape[0])
    host_tok = torch.empty(cap, dtype=torch.int32, pin_memory=True)

    def start(sid):
        add, max_new = work.turn(sid, turn[sid])
        h = np.concatenate([hist[sid], add]).astype(np.int32)
        hist[sid] = h
        rid = eng.add_request(h, max_new, seed=1000 + sid * 64 + turn[sid], temperature=work.temperature)
        rid_of[rid] = (sid, turn[sid], max_new)
        res.submitted += len(h)

    while queue and len(rid_of) < concurrency:
        start(queue.popleft())
    plan = vd.PlanOut()
    i32p = ctypes.POINTER(ctypes.c_int32)
    while eng.pending():
        t0 = time.perf_counter()
        vd.check(lib.vd_engine_plan(eng.h, ctypes.byref(plan)))
        b = plan.batch
        if b.num_tokens == 0:
            raise RuntimeError("engine has pending requests but planned an empty step")
        B, R = b.num_seqs, b.num_logit_rows
        cu = np.ctypeslib.as_array(b.cu_q, (B + 1,))
        cached = np.ctypeslib.as_array(b.cached_len, (B,))
        seqs = [(int(cached[i]), int(cu[i + 1] - cu[i])) for i in range(B)]
        rids = np.ctypeslib.as_array(plan.rids, (R,)).copy() if R else np.zeros(0, np.int64)
        vd.check(lib.vd_step_sample(model.h, pool.h, ctypes.byref(b), plan.samplers, vd._ptr(logits),
                                    vd._ptr(tokens_dev), s))
        if R:
            host_tok[:R].copy_(tokens_dev[:R], non_blocking=True)
        (stream or torch.cuda.current_stream()).synchronize()
        toks = host_tok[:R].numpy().copy()
        vd.check(lib.vd_engine_commit(eng.h, toks.ctypes.data_as(i32p)))
        res.steps.append(StepInfo(seqs, R, time.perf_counter() - t0))
        if on_rows is not None and R:
            info = [rid_of[int(r)] for r in rids]
            on_rows([x[0] for x in info], [x[1] for x in info], logits[:R], toks)
        for r, t in zip(rids, toks):
            r = int(r)
            got[r].append(int(t))
            sid, k, max_new = rid_of[r]
            if len(got[r]) == max_new:
                del rid_of[r]
                out = got.pop(r)
                res.outputs[sid].append(out)
                hist[sid] = np.concatenate([hist[sid], np.asarray(out, np.int32)])
                turn[sid] += 1
                if turn[sid] < work.turns:
                    queue.append(sid)
        while queue and len(rid_of) < concurrency:
            start(queue.popleft())
    return res
