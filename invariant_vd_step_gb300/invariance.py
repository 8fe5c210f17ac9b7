"""Execution-variation matrix: bitwise comparison of per-request logit views.

Definition 2.1 (深入解析 Vosti §二): two executions sharing W, given the same
prompt and initial sampler state, must yield prefix-comparable per-request
views.  Here every execution is compared with a canonical one, row by row,
bit for bit, in the categories of the paper's evaluation (深入解析 Vosti
§七 7.1): batch composition, chunked prefill, prefill vs decode, prefix
reuse; plus eviction with recomputation (§五 5.2).

The tiny workload: 8 requests with uniform-random prompts of 17..64 tokens,
4 of them sharing a 32-token prefix, 16 greedy decode steps, pages of 16.
Executions: max batch {1, 3, 8} x chunk budget {16, 64} x prefix reuse
{off, on} x page placement {sequential, shuffled} = 24 runs, each compared
with (1, 64, off, sequential) on every emitted row (23 x 128 pairs); one
cold prefill per request of its final history compared with every emitted
decode row (128 pairs); one run with a 12-page pool that forces eviction
and recomputation (128 pairs).  3,200 pairs in all.
"""

from __future__ import annotations

import dataclasses
import itertools

import numpy as np
import torch

from . import engine, synth, vd


@dataclasses.dataclass
class MatrixResult:
    pairs: int
    equal: int
    categories: dict
    runs: int
    evicted: int
    preempted: int
    prefix_hit_pages: int

    @property
    def pass_pct(self) -> float:
        return 100.0 * self.equal / max(1, self.pairs)


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.int32)


def _row_bits(x) -> bytes:
    if isinstance(x, torch.Tensor):
        return x.detach().contiguous().view(torch.int32).cpu().numpy().tobytes()
    return np.ascontiguousarray(x, dtype=np.float32).view(np.int32).tobytes()


def prefix_comparable(view_a, view_b) -> bool:
    """Definition 2.1 (深入解析 Vosti §二): two views of one request are
    prefix-comparable iff the shorter is a prefix of the longer.  A view is a
    list of (logits, token) rows; logits compare by their float32 bits."""
    for (la, ta), (lb, tb) in zip(view_a, view_b):
        if int(ta) != int(tb) or _row_bits(la) != _row_bits(lb):
            return False
    return True


def tiny_workload(seed: int = 1):
    spec = synth.TINY
    prompts = synth.make_prompts(8, 17, 64, spec.vocab, seed=seed, shared_prefix=32, n_sharing=4)
    return spec, prompts, 16


def run_matrix(seed_weights: int = 0, seed_prompts: int = 1, device="cuda") -> MatrixResult:
    spec, prompts, max_new = tiny_workload(seed_prompts)
    W = synth.make_weights(spec, seed=seed_weights, device=device)
    max_ctx = max(len(p) for p in prompts) + max_new + 16
    model = vd.Model(spec, W, max_tokens=256, max_seqs=8, max_logit_rows=64, max_context=max_ctx)
    pool = vd.KVPool(model, 128)
    ex = engine.GpuExecutor(model, pool)

    def execute(max_batch, budget, reuse, shuffled, num_pages=128):
        eng = engine.Engine(ex, num_pages, max_batch=max_batch, token_budget=budget, prefix_reuse=reuse,
                            placement_seed=7 if shuffled else None)
        for i, p in enumerate(prompts):
            eng.add_request(p, max_new, seed=1000 + i)
        eng.run()
        return eng

    canon = execute(1, 64, False, False)
    ref = {rid: [_bits(l) for l, _ in v] for rid, v in canon.views.items()}
    cats = {"batch_chunk_prefix_pages": [0, 0], "prefill_decode": [0, 0], "evict_recompute": [0, 0]}
    stats = {"evicted": 0, "preempted": 0, "prefix_hit_pages": 0}
    runs = 1

    def compare(views, cat):
        for rid, rows in ref.items():
            got = views.get(rid, [])
            for j, r in enumerate(rows):
                cats[cat][0] += 1
                if j < len(got) and torch.equal(_bits(got[j][0]), r):
                    cats[cat][1] += 1

    for b, c, reuse, sh in itertools.product((1, 3, 8), (16, 64), (False, True), (False, True)):
        if (b, c, reuse, sh) == (1, 64, False, False):
            continue
        eng = execute(b, c, reuse, sh)
        runs += 1
        for k in stats:
            stats[k] += eng.stats[k]
        compare(eng.views, "batch_chunk_prefix_pages")

    # prefill vs decode: one cold prefill of each final history, all emitted rows
    pf = {}
    for rid, r in canon.requests.items():
        h = np.asarray(r.history[:-1], dtype=np.int32)
        n0 = len(r.prompt) - 1
        pt = np.arange((len(h) + 15) // 16, dtype=np.int32)
        logits = torch.empty((len(h) - n0, spec.vocab), dtype=torch.float32, device=device)
        model.step(pool, vd.StepBatch([(h, 0, pt)], logit_rows=range(n0, len(h))), logits)
        pf[rid] = [(logits[j], None) for j in range(len(h) - n0)]
    compare(pf, "prefill_decode")

    ev = execute(8, 64, True, True, num_pages=12)
    runs += 1
    for k in stats:
        stats[k] += ev.stats[k]
    compare(ev.views, "evict_recompute")
    torch.cuda.synchronize()
    pairs = sum(v[0] for v in cats.values())
    equal = sum(v[1] for v in cats.values())
    del ex, pool
    model.close()
    return MatrixResult(pairs, equal, {k: {"pairs": v[0], "equal": v[1]} for k, v in cats.items()}, runs,
                        stats["evicted"], stats["preempted"], stats["prefix_hit_pages"])
