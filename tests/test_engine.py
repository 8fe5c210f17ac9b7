"""Host scheduler and block manager on the CPU (oracle-backed paged executor)."""

import numpy as np
import pytest

from invariant_vd_step_gb300 import engine, invariance, synth
from oracle.decoder import OracleDecoder
from oracle_executor import OracleExecutor

SPEC = synth.TINY.with_(n_layers=1)


@pytest.fixture(scope="module")
def weights():
    return synth.weights_to_numpy(synth.make_weights(SPEC, seed=3, gain_std=0.1))


def _prompts(n=6, seed=1):
    return synth.make_prompts(n, 17, 50, SPEC.vocab, seed=seed, shared_prefix=32, n_sharing=4)


def _run(weights, prompts, max_new=6, num_pages=64, **kw):
    box = {}
    ex = OracleExecutor(SPEC, weights, num_pages,
                        write_guard=lambda pg: not box["eng"].page_info(pg)[1])
    eng = engine.Engine(ex, num_pages, **kw)
    box["eng"] = eng
    for i, p in enumerate(prompts):
        eng.add_request(p, max_new, seed=100 + i)
    n = 0
    while eng.pending():
        eng.step()
        eng.check()
        n += 1
        assert n < 10000
    return eng


def _cold_check(weights, eng):
    dec = OracleDecoder(SPEC, weights)
    for rid, r in eng.requests.items():
        h = np.asarray(r.history)
        cold = dec.forward_all(h[:-1])
        n0 = len(r.prompt) - 1
        for j, (lg, tok) in enumerate(eng.views[rid]):
            np.testing.assert_array_equal(lg, cold[n0 + j])  # Theorem 4.1, bitwise
            assert tok == h[n0 + j + 1]


def test_engine_views_equal_cold_forward_with_prefix_reuse(weights):
    eng = _run(weights, _prompts(), max_batch=3, token_budget=24, placement_seed=5)
    assert eng.stats["prefix_hit_pages"] > 0
    _cold_check(weights, eng)


def test_forced_hash_collisions_never_cause_reuse(weights):
    # Every page hashes to the same value: candidates must be rejected by the
    # exact token / depth / parent check (深入解析 Vosti §五 5.4).
    prompts = _prompts(seed=2)
    prompts.append(prompts[0][:20].copy())
    prompts[-1][17] = (prompts[-1][17] + 1) % SPEC.vocab  # same first page, different second
    eng = _run(weights, prompts, max_batch=2, token_budget=32, hash_mode=1)
    assert eng.stats["hash_candidates_rejected"] > 0
    _cold_check(weights, eng)


def test_pool_pressure_evicts_leaves_and_recomputes(weights):
    eng = _run(weights, _prompts(seed=3), max_new=8, num_pages=9, max_batch=4, token_budget=40)
    assert eng.stats["preempted"] > 0 or eng.stats["evicted"] > 0
    _cold_check(weights, eng)


def test_definition_2_1_prefix_comparable_across_executions(weights):
    prompts = _prompts(seed=4)
    base = _run(weights, prompts, max_batch=1, token_budget=64, prefix_reuse=False)
    variants = [
        dict(max_batch=6, token_budget=16, placement_seed=1),
        dict(max_batch=2, token_budget=7, prefix_reuse=True, placement_seed=2),
        dict(max_batch=3, token_budget=64, num_pages=10),
    ]
    for kw in variants:
        other = _run(weights, prompts, **kw)
        for rid in base.views:
            a, b = base.views[rid], other.views[rid]
            assert min(len(a), len(b)) > 0
            assert invariance.prefix_comparable(a, b), (kw, rid)


def test_finished_prefix_is_retained_then_evicted_leaf_first(weights):
    # A finished request's registered pages stay reusable (retain); under
    # pressure the unreferenced leaves go first, never a parent of a kept page.
    base = synth.make_tokens(40, SPEC.vocab, seed=21)
    first = _run(weights, [base], max_new=2, num_pages=8, max_batch=1)
    assert first.stats["registered"] >= 2
    ex = OracleExecutor(SPEC, weights, 8)
    eng = engine.Engine(ex, 8, max_batch=1, token_budget=64)
    eng.add_request(base, 2, seed=1)
    eng.run()
    eng.add_request(base[:36], 2, seed=2)         # same first two pages
    eng.run()
    st = eng.stats
    assert st["prefix_hit_pages"] == 2, st
    eng.add_request(synth.make_tokens(100, SPEC.vocab, seed=22), 2, seed=3)  # needs 7 of 8 pages
    eng.run()
    eng.check()
    assert eng.stats["evicted"] >= 1
    _cold_check(weights, eng)


class _NoCompute:
    """Executor stand-in for scheduling-only tests: token = (rid-independent) 7."""

    def step(self, seqs, rows):
        return np.zeros((len(rows), 1))

    def sample(self, logits, samplers):
        return np.full(len(samplers), 7, dtype=np.int32)


@pytest.mark.parametrize("num_pages", [40, 48, 64, 96])
def test_multi_turn_sessions_under_pressure_make_progress(num_pages):
    """Sessions with a shared prefix resubmitting their whole history every turn,
    under a pool far smaller than their working set: every plan makes progress
    (preemption never re-admits its victim in the same pass), the block
    manager stays consistent, and everything finishes."""
    rng = np.random.default_rng(num_pages)
    prefix = synth.make_tokens(96, SPEC.vocab, seed=5)
    eng = engine.Engine(_NoCompute(), num_pages, max_batch=8, token_budget=64, placement_seed=1)
    hist, live, emitted = {}, {}, {}

    def submit(s, k):
        base = prefix if k == 0 else hist[s]
        hist[s] = np.concatenate([base, synth.make_tokens(int(rng.integers(10, 60)), SPEC.vocab, seed=100 * s + k)])
        max_new = int(rng.integers(4, 20))
        rid = eng.add_request(hist[s], max_new, seed=s)
        live[rid] = (s, k, max_new)
        emitted[rid] = 0

    for s in range(10):
        submit(s, 0)
    steps = 0
    while eng.pending():
        rec = eng.step()
        eng.check()
        steps += 1
        assert steps < 5000, "scheduler stopped making progress"
        for rid in rec:
            emitted[rid] += 1
        for rid in [r for r in live if emitted[r] == live[r][2]]:
            s, k, _ = live.pop(rid)
            hist[s] = np.asarray(eng.history(rid).history, dtype=np.int32)
            if k + 1 < 3:
                submit(s, k + 1)
    assert not live
    assert eng.stats["evicted"] > 0 or num_pages >= 96


def test_decode_growth_preempts_newest_and_finishes():
    """Requests admitted when their prompts fit, then outgrowing the pool while
    decoding: the newest is preempted and recomputed, nothing livelocks, and
    every request emits all of its tokens."""
    eng = engine.Engine(_NoCompute(), 24, max_batch=8, token_budget=64, prefix_reuse=False)
    want = {}
    for i in range(8):
        want[eng.add_request(synth.make_tokens(20, SPEC.vocab, seed=i), 60, seed=i)] = 60
    got = {r: 0 for r in want}
    steps = 0
    while eng.pending():
        for rid in eng.step():
            got[rid] += 1
        eng.check()
        steps += 1
        assert steps < 5000, "scheduler stopped making progress"
    assert got == want
    assert eng.stats["preempted"] > 0


def test_request_larger_than_the_pool_is_reported():
    eng = engine.Engine(_NoCompute(), 4, max_batch=2, token_budget=64)
    eng.add_request(synth.make_tokens(100, SPEC.vocab, seed=1), 4)
    with pytest.raises(Exception, match="VD_ERR_CAPACITY"):
        for _ in range(4):  # the first 64-token chunk fits in the 4 pages, the rest cannot
            eng.step()
