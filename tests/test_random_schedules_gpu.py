"""Seeded random execution schedules: every request's per-row logits and
tokens are bitwise those of the canonical execution.

Definition 2.1 (深入解析 Vosti §二) asks that two executions sharing W, given
the same prompt and initial sampler state, yield prefix-comparable views;
Theorem 4.1 that a row's logits are Forward(W, history).  The fixed
3,200-pair matrix covers a grid of settings; this test draws the settings
at random per seed instead: request counts and prompt lengths (1..120
tokens, some sharing prefixes of any length), greedy and sampled requests,
the engine's batch cap, chunk budget, prefix reuse and page placement, a
pool small enough to force eviction, recomputation and preemption in some
runs, step-graph replay on or off, and a forced GEMM tile shape, for a
Llama-style and a Gemma-style block (sliding windows, QK-norm, GeGLU,
sandwich norms).  The canonical execution runs one request at a time with a
large budget, no reuse, sequential pages and a roomy pool.
"""

import numpy as np
import pytest
import torch

from gpu_util import ready
from invariant_vd_step_gb300 import engine, synth, vd

pytestmark = pytest.mark.gpu

PLANS = [(0, 0, 0), (64, 16, 4), (128, 32, 2), (128, 256, 1), (256, 64, 1), (64, 128, 1)]


def _workload(rng, vocab):
    n = int(rng.integers(4, 13))
    base = synth.make_tokens(120, vocab, seed=int(rng.integers(1 << 30)))
    reqs = []
    for i in range(n):
        length = int(rng.integers(1, 121))
        if i > 0 and rng.random() < 0.4:  # share a prefix (any length) with the common stream
            share = int(rng.integers(1, length + 1))
            own = synth.make_tokens(length - share, vocab, seed=int(rng.integers(1 << 30)))
            prompt = np.concatenate([base[:share], own]).astype(np.int32)
        else:
            prompt = synth.make_tokens(length, vocab, seed=int(rng.integers(1 << 30)))
        max_new = int(rng.integers(1, 25))
        temperature = 0.0 if rng.random() < 0.5 else float(rng.choice([0.5, 1.0]))
        reqs.append((prompt, max_new, 500 + i, temperature))
    return reqs


def _execute(model, pool, reqs, max_batch, budget, reuse, placement, num_pages):
    ex = engine.GpuExecutor(model, pool)
    eng = engine.Engine(ex, num_pages, max_batch=max_batch, token_budget=budget, prefix_reuse=reuse,
                        placement_seed=placement)
    for prompt, max_new, seed, temp in reqs:
        eng.add_request(prompt, max_new, seed=seed, temperature=temp)
    eng.run()
    eng.check()
    views = {rid: [(l.contiguous().view(torch.int32).clone(), int(t)) for l, t in rows]
             for rid, rows in eng.views.items()}
    stats = dict(eng.stats)
    eng.close()
    return views, stats


GEMMA_TINY = synth.ModelSpec("gemma-tiny", 3, 256, 2, 1, 256, 512, 512, act="geglu", qk_norm=True,
                             rope_theta=1e6, rope_theta_local=1e4, sliding_window=24, local_global_period=2,
                             rms_eps=1e-6, embed_scale=True, norm_offset=True, sandwich_norm=True)


def _one_seed(spec, seed, totals):
    rng = np.random.default_rng(1000 + seed)
    W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=seed, gain_std=0.1).items()}
    reqs = _workload(rng, spec.vocab)
    longest = max(len(p) + m for p, m, _, _ in reqs)
    need_one = (longest + 15) // 16 + 1
    roomy = sum((len(p) + m + 15) // 16 + 1 for p, m, _, _ in reqs) + 4
    model = vd.Model(spec, W, max_tokens=256, max_seqs=16, max_logit_rows=64, max_context=longest + 32)
    pool = vd.KVPool(model, roomy)
    try:
        canon, _ = _execute(model, pool, reqs, 1, 256, False, None, roomy)
        assert sum(len(v) for v in canon.values()) == sum(m for _, m, _, _ in reqs)
        for run in range(4):
            max_batch = int(rng.integers(1, 13))
            budget = int(rng.choice([8, 16, 33, 64, 200]))
            reuse = bool(rng.random() < 0.7)
            placement = int(rng.integers(1 << 20)) if rng.random() < 0.7 else None
            tight = rng.random() < 0.4
            num_pages = int(rng.integers(need_one, need_one + 8)) if tight else roomy
            model.set_graph_mode(int(rng.choice([0, 8])))
            vd.set_gemm_plan(*PLANS[int(rng.integers(len(PLANS)))])
            got, stats = _execute(model, pool, reqs, max_batch, budget, reuse, placement, num_pages)
            for k in ("evicted", "preempted", "prefix_hit_pages"):
                totals[k] += stats[k]
            totals["runs"] += 1
            cfg = (seed, max_batch, budget, reuse, placement, num_pages)
            assert got.keys() == canon.keys(), cfg
            for rid, rows in canon.items():
                assert len(got[rid]) == len(rows), (cfg, rid)
                for j, ((lc, tc), (lg, tg)) in enumerate(zip(rows, got[rid])):
                    assert tg == tc, (cfg, rid, j, "token")
                    assert torch.equal(lg, lc), (cfg, rid, j, "logits")
        assert model.device_status() == 0
    finally:
        vd.set_gemm_plan(0, 0, 0)
        pool.close()
        model.close()


@pytest.mark.parametrize("spec,seeds", [(synth.TINY, 24), (GEMMA_TINY, 8)], ids=["tiny-llama", "gemma-tiny"])
def test_random_schedules_match_the_canonical_execution(spec, seeds):
    ready()
    totals = {"evicted": 0, "preempted": 0, "prefix_hit_pages": 0, "runs": 0}
    for seed in range(seeds):
        _one_seed(spec, seed, totals)
    # the draws did reach the behaviours they are meant to exercise
    assert totals["runs"] == 4 * seeds and totals["evicted"] > 0 and totals["prefix_hit_pages"] > 0, totals
