"""Graph replay of steps: bitwise the eager path, across split and stride changes."""

import numpy as np
import pytest
import torch

from gpu_util import bits, ready
from invariant_vd_step_gb300 import synth, vd

pytestmark = pytest.mark.gpu


def _schedule():
    """Prefill chunks, then decode steps whose contexts cross 512 and 1024
    (new KV splits, so new attention item counts), with one mixed step that
    holds a decode-class (8 tokens) and a prefill-class (9 tokens) chunk."""
    prompts = [500, 1015, 40, 509]
    steps = [[(0, 500), (3, 509)], [(1, 1015)], [(2, 40)]]
    steps += [[(0, 1), (1, 1), (2, 1), (3, 1)] for _ in range(12)]
    steps += [[(0, 1), (1, 8), (2, 9), (3, 1)]]
    steps += [[(0, 1), (1, 1), (2, 1), (3, 1)] for _ in range(12)]
    total = [p + sum(n for st in steps[3:] for r, n in st if r == i) for i, p in enumerate(prompts)]
    return total, steps


class Pair:
    def __init__(self, spec, num_pages=320, max_context=2048):
        self.spec = spec
        W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=5, gain_std=0.1).items()}
        kw = dict(max_tokens=1024, max_seqs=8, max_logit_rows=1024, max_context=max_context)
        self.eager = vd.Model(spec, W, **kw)
        self.graph = vd.Model(spec, W, **kw)
        self.graph.set_graph_mode(16)
        self.pa = vd.KVPool(self.eager, num_pages)
        self.pb = vd.KVPool(self.graph, num_pages)
        self.W = W
        self.la = torch.empty(1024, spec.vocab, device="cuda")
        self.lb = torch.empty(1024, spec.vocab, device="cuda")

    def run(self, hist, steps, perm, swap_logits_at=None):
        tables = {r: [] for r in range(len(hist))}
        done = {r: 0 for r in range(len(hist))}
        nxt = 0
        for si, step in enumerate(steps):
            seqs = []
            for r, n in step:
                c = done[r]
                while len(tables[r]) < (c + n + 15) // 16:
                    tables[r].append(int(perm[nxt]))
                    nxt += 1
                seqs.append((hist[r][c:c + n], c, np.array(tables[r], np.int32)))
                done[r] = c + n
            batch = vd.StepBatch(seqs, logit_rows=range(sum(n for _, n in step)))
            R = batch.num_logit_rows
            self.eager.step(self.pa, batch, self.la)
            lb = self.lb if si != swap_logits_at else torch.empty_like(self.lb)
            self.graph.step(self.pb, batch, lb)
            torch.cuda.synchronize()
            assert np.array_equal(bits(self.la[:R]), bits(lb[:R])), f"step {si}: graph logits differ"
        assert self.eager.device_status() == 0 and self.graph.device_status() == 0


def test_graph_replay_bitwise_matches_eager():
    ready()
    spec = synth.TINY
    total, steps = _schedule()
    hist = [synth.make_tokens(n, spec.vocab, seed=40 + i) for i, n in enumerate(total)]
    p = Pair(spec)
    p.run(hist, steps, synth.page_permutation(320, seed=6))
    st = p.graph.graph_stats()
    assert st["captures"] + st["replays"] + st["eager"] == len(steps)
    assert st["replays"] >= 10, st  # steady decode steps share graphs
    assert st["captures"] <= st["eager"]  # a key is captured only on its second sighting
    assert st["cached"] <= 16


def test_graph_cache_bound_and_new_logits_buffer():
    ready()
    spec = synth.TINY
    total, steps = _schedule()
    hist = [synth.make_tokens(n, spec.vocab, seed=50 + i) for i, n in enumerate(total)]
    p = Pair(spec)
    p.graph.set_graph_mode(2)
    p.run(hist, steps, synth.page_permutation(320, seed=7), swap_logits_at=10)
    st = p.graph.graph_stats()
    assert st["cached"] <= 2
    assert st["captures"] + st["replays"] + st["eager"] == len(steps)
    p.graph.set_graph_mode(0)
    assert p.graph.graph_stats()["cached"] == 0


def test_graph_mode_rejects_negative():
    ready()
    spec = synth.TINY
    W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=1).items()}
    m = vd.Model(spec, W, max_tokens=64, max_seqs=4, max_logit_rows=64, max_context=256)
    with pytest.raises(vd.VDError):
        m.set_graph_mode(-1)


def test_a_new_gemm_plan_is_captured_not_replayed_stale():
    """A captured step graph holds its GEMM launches with the tile shapes of
    its capture; after vd_set_gemm_plan the same step key is seen afresh
    (captured again on its second sighting), and its logits stay bitwise
    those of the eager step either way."""
    ready()
    spec = synth.TINY
    W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=3, gain_std=0.1).items()}
    m = vd.Model(spec, W, max_tokens=64, max_seqs=4, max_logit_rows=8, max_context=256)
    e = vd.Model(spec, W, max_tokens=64, max_seqs=4, max_logit_rows=8, max_context=256)
    m.set_graph_mode(8)
    pm, pe = vd.KVPool(m, 32), vd.KVPool(e, 32)
    toks = synth.make_tokens(40, spec.vocab, seed=9)
    pages = np.arange(8, dtype=np.int32)
    lm, le = torch.empty(1, spec.vocab, device="cuda"), torch.empty(1, spec.vocab, device="cuda")
    pre = vd.StepBatch([(toks[:30], 0, pages)], logit_rows=[29])
    m.step(pm, pre, lm)
    e.step(pe, pre, le)
    try:
        for i, plan in enumerate([(0, 0, 0), (0, 0, 0), (0, 0, 0), (64, 16, 4), (64, 16, 4), (64, 16, 4)]):
            vd.set_gemm_plan(*plan)
            b = vd.StepBatch([(toks[30:31], 30, pages)], logit_rows=[0])  # the same step each time
            m.step(pm, b, lm)
            e.step(pe, b, le)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(bits(lm), bits(le), err_msg=f"step {i} plan {plan}")
            st = m.graph_stats()
            if i == 2:
                assert (st["captures"], st["replays"]) == (1, 1), st
        st = m.graph_stats()
        assert (st["captures"], st["replays"]) == (2, 2), st  # one capture and one replay per plan
    finally:
        vd.set_gemm_plan(0, 0, 0)
    assert m.device_status() == 0
