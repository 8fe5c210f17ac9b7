"""Agentic sessions: a shared prefix, several turns per session, a pool small
enough to force evictions and recomputation.  Every session's logits and
tokens must equal those of the same session served alone with an unlimited
pool (the agentic workload's invariance check), compared bitwise through
64-bit fingerprints of the logits rows."""

import collections

import numpy as np
import pytest
import torch

from gpu_util import ready
from invariant_vd_step_gb300 import engine, sessions, synth, vd

pytestmark = pytest.mark.gpu


def _fingerprint(rows: torch.Tensor) -> np.ndarray:
    g = torch.Generator(device="cuda")
    g.manual_seed(12345)
    w = torch.randint(-2 ** 62, 2 ** 62, (rows.shape[1],), generator=g, device="cuda", dtype=torch.int64)
    return (rows.contiguous().view(torch.int32).to(torch.int64) * w).sum(dim=1).cpu().numpy()


def _serve(model, work, conc, pages, budget, only=None, graphs=0):
    model.set_graph_mode(graphs)
    pool = vd.KVPool(model, pages)
    eng = engine.Engine(None, pages, max_batch=conc, token_budget=budget, prefix_reuse=True, placement_seed=4)
    logits = torch.empty((conc, work.vocab), device="cuda")
    tok = torch.empty(conc, dtype=torch.int32, device="cuda")
    seen = collections.defaultdict(list)

    def on_rows(sids, turns, rows, toks):
        for s, k, f, t in zip(sids, turns, _fingerprint(rows), toks):
            seen[(s, k)].append((int(f), int(t)))

    res = sessions.run_sessions(work, model, pool, eng, conc, logits, tok, on_rows=on_rows, only=only)
    assert model.device_status() == 0
    eng.check()
    return seen, res, eng.stats


@pytest.mark.parametrize("graphs", [0, 16])
def test_sessions_with_evictions_match_sessions_alone(graphs):
    ready()
    spec = synth.TINY
    W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=2, gain_std=0.1).items()}
    work = sessions.SessionWorkload(spec.vocab, 12, 3, 20, 80, 8, 24, prefix=synth.make_tokens(256, spec.vocab, seed=5),
                                    seed=3)
    model = vd.Model(spec, W, max_tokens=64, max_seqs=8, max_logit_rows=8, max_context=work.max_context())
    conc = 6
    mean_final = 256 + 3 * (50 + 16)
    pages = int(0.5 * conc * mean_final / 16)
    both, res, st = _serve(model, work, conc, pages, 64, graphs=graphs)
    assert st["evicted"] > 0, "the pool was meant to force evictions"
    assert st["prefix_hit_pages"] > 0, "turns and sessions were meant to share prefix pages"
    assert sum(len(o) for o in res.outputs.values()) == 12 * 3
    for sid in range(12):
        alone, _, _ = _serve(model, work, 1, 64, 64, only=[sid])
        for k in range(3):
            assert both[(sid, k)] == alone[(sid, k)], f"session {sid} turn {k} differs"
