"""Decode-verify-rollback over the fast and the invariant step ("LLM-42:
Enabling Determinism in LLM Inference with Verified Speculation", §4).

Candidates come from the fast path (reduction mode 1: split-K GEMMs, not
batch-invariant).  Every `window` candidates of a request are replayed by one
invariant step as a single chunk, the tokens [last verified, c1 .. c(W-1)] at
their positions with a logit row at each; the verified tokens t1 .. tW are
compared with the candidates.  Up to the first disagreement j the candidates
are accepted, t_j replaces c_j, and the rest is dropped; the verify chunk has
already written the invariant K/V of every accepted position, and the slots
past it are rewritten as decoding goes on.  Each verification emits at least
one token, so decoding always progresses.  Full windows of several requests
are verified in the same step.

Because the invariant step is also prefill-decode invariant (a position's
logits do not depend on whether it was computed in a chunk or in a decode
step, 深入解析 Vosti §二 Theorem 4.1), every released token and every verified
logit row equals what plain invariant decoding produces, bit for bit.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from . import vd


@dataclass
class _Req:
    rid: int
    ctx: int                      # positions with verified (invariant) K/V
    cur: int                      # token at position ctx, not yet processed
    pages: list
    max_new: int
    seed: int
    temperature: float
    out: list = field(default_factory=list)    # released (verified) tokens
    cand: list = field(default_factory=list)   # fast-path candidates since the last verification

    @property
    def done(self) -> bool:
        return len(self.out) >= self.max_new


@dataclass
class Stats:
    fast_steps: int = 0
    verify_steps: int = 0
    candidates: int = 0
    accepted: int = 0            # candidates confirmed by verification
    rolled_back: int = 0         # candidates dropped after a disagreement


class SelectiveDecoder:
    """Runs requests to completion with decode-verify-rollback.

    ``pages``: free physical page ids this decoder may hand out.  A request
    starts either from a prompt (`add_prompt`, prefilled on the invariant
    path) or from K/V already in the pool (`add_cached`)."""

    def __init__(self, model: vd.Model, pool: vd.KVPool, pages, window: int = 8, max_batch: int = 256,
                 stream=None, keep_logits: bool = False):
        self.m, self.pool, self.W = model, pool, int(window)
        self.free = list(pages)[::-1]
        self.reqs: list[_Req] = []
        self.stats = Stats()
        self.stream = stream
        self.keep_logits = keep_logits
        self.verified_logits: dict = {}      # (rid, output index) -> logits row (keep_logits)
        V = model.spec.vocab
        self.logits = torch.empty((max(max_batch * window, 1), V), dtype=torch.float32, device="cuda")
        self.tok = torch.empty(max(max_batch * window, 1), dtype=torch.int32, device="cuda")

    # -- requests ------------------------------------------------------------
    def _alloc(self, r: _Req, upto: int):
        while len(r.pages) * 16 < upto:
            if not self.free:
                raise RuntimeError("out of KV pages")
            r.pages.append(self.free.pop())

    def add_cached(self, ctx: int, cur: int, pages, max_new: int, seed: int = 0, temperature: float = 0.0) -> int:
        r = _Req(len(self.reqs), int(ctx), int(cur), list(pages), int(max_new), int(seed), float(temperature))
        self.reqs.append(r)
        return r.rid

    def add_prompt(self, prompt, max_new: int, seed: int = 0, temperature: float = 0.0) -> int:
        """Prefill on the invariant path; the first output token is verified by construction."""
        prompt = np.asarray(prompt, dtype=np.int32)
        r = _Req(len(self.reqs), 0, 0, [], int(max_new), int(seed), float(temperature))
        self._alloc(r, len(prompt))
        self.m.set_reduction_mode(0)
        b = vd.StepBatch([(prompt, 0, np.array(r.pages, np.int32))], logit_rows=[len(prompt) - 1])
        self.m.step_sample(self.pool, b, [(r.seed, 0, r.temperature)], self.logits[:1], self.tok[:1], self.stream)
        t = int(self.tok[0].item())
        if self.keep_logits:
            self.verified_logits[(r.rid, 0)] = self.logits[0].clone()
        r.ctx, r.cur, r.out = len(prompt), t, [t]
        self.reqs.append(r)
        return r.rid

    # -- steps ----------------------------------------------------------------
    def _fast_step(self, live):
        seqs, samp = [], []
        for r in live:
            p = r.ctx + len(r.cand)                     # position of the token to process
            self._alloc(r, p + 1)
            last = r.cand[-1] if r.cand else r.cur
            seqs.append((np.array([last], np.int32), p, np.array(r.pages, np.int32)))
            samp.append((r.seed, len(r.out) + len(r.cand), r.temperature))
        self.m.set_reduction_mode(1)
        b = vd.StepBatch(seqs, logit_rows=range(len(seqs)))
        self.m.step_sample(self.pool, b, samp, self.logits, self.tok, self.stream)
        toks = self.tok[:len(seqs)].cpu().numpy()
        for r, t in zip(live, toks):
            r.cand.append(int(t))
        self.stats.fast_steps += 1
        self.stats.candidates += len(live)

    def _verify_step(self, group):
        seqs, rows, samp, t = [], [], [], 0
        for r in group:
            n = len(r.cand)
            chunk = np.array([r.cur] + r.cand[:-1], np.int32)
            seqs.append((chunk, r.ctx, np.array(r.pages, np.int32)))
            rows += list(range(t, t + n))
            samp += [(r.seed, len(r.out) + i, r.temperature) for i in range(n)]
            t += n
        self.m.set_reduction_mode(0)
        b = vd.StepBatch(seqs, logit_rows=rows)
        self.m.step_sample(self.pool, b, samp, self.logits, self.tok, self.stream)
        ver = self.tok[:len(rows)].cpu().numpy()
        k = 0
        for r in group:
            n = len(r.cand)
            v = [int(x) for x in ver[k:k + n]]
            j = next((i for i in range(n) if v[i] != r.cand[i]), n)   # first disagreement
            take = v[:j + 1] if j < n else v                         # verifier's token at j included
            if self.keep_logits:
                for i in range(len(take)):
                    self.verified_logits[(r.rid, len(r.out) + i)] = self.logits[k + i].clone()
            self.stats.accepted += min(j, n)
            self.stats.rolled_back += n - min(j, n)
            r.ctx += len(take)
            r.cur = take[-1]
            r.out += take
            r.cand = []
            k += n
        self.stats.verify_steps += 1

    def run(self) -> dict:
        """Decodes every request to max_new released tokens; returns {rid: tokens}."""
        while True:
            live = [r for r in self.reqs if not r.done]
            if not live:
                break
            # a window is full once it holds W candidates or reaches the request's end
            full = [r for r in live if len(r.cand) >= min(self.W, r.max_new - len(r.out))]
            if len(full) == len(live):
                self._verify_step(full)
            else:
                self._fast_step([r for r in live if r not in full])
        return {r.rid: r.out[:r.max_new] for r in self.reqs}
