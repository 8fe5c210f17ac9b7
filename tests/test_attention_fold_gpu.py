"""Decode attention in fold mode (one CTA walks all splits of its rows and
folds them) against split mode (one CTA per split plus the merge kernel):
logits bitwise equal, the cross-mapping check that workload-dependent
dispatch needs (深入解析 Vosti §八 8.1)."""

import numpy as np
import pytest
import torch

from gpu_util import bits, ready
from invariant_vd_step_gb300 import synth, vd

pytestmark = pytest.mark.gpu

# head dim 128, GQA 2, local sliding-window layers (window 300) between global ones
HD128_LOCAL = synth.TINY.with_(name="tiny-hd128-local", head_dim=128, sliding_window=300, local_global_period=2,
                               n_layers=3)


def _schedule(n_req=6):
    """Prompts of 1100..2100 tokens (3-5 KV splits of 512), then decode steps of
    1 token, steps of 3-8 tokens per request (several rows and positions in
    one decode-class CTA), and a step mixing decode rows with a prefill chunk."""
    rng = np.random.default_rng(3)
    lens = [int(x) for x in rng.integers(1100, 2100, size=n_req)]
    steps = [[(r, lens[r])] for r in range(n_req)]
    steps += [[(r, 1) for r in range(n_req)] for _ in range(3)]
    steps += [[(r, 3 + r) for r in range(n_req)]]
    steps += [[(r, 1) for r in range(n_req - 1)] + [(n_req - 1, 40)]]
    steps += [[(r, 2) for r in range(n_req)] for _ in range(2)]
    total = [lens[r] + sum(n for st in steps[n_req:] for rr, n in st if rr == r) for r in range(n_req)]
    return total, steps


@pytest.mark.parametrize("spec", [synth.TINY, HD128_LOCAL], ids=lambda s: s.name)
@pytest.mark.parametrize("graphs", [0, 8])
def test_fold_mode_bitwise_equals_split_mode(spec, graphs):
    ready()
    total, steps = _schedule()
    hist = [synth.make_tokens(n, spec.vocab, seed=60 + i) for i, n in enumerate(total)]
    W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=7, gain_std=0.1).items()}
    kw = dict(max_tokens=2200, max_seqs=8, max_logit_rows=64, max_context=2400)
    models = [vd.Model(spec, W, **kw), vd.Model(spec, W, **kw)]
    models[0].set_attention_fold(1)
    models[1].set_attention_fold(2)
    for m in models:
        m.set_graph_mode(graphs)
    npg = 160 * len(total)
    pools = [vd.KVPool(m, npg) for m in models]
    perm = synth.page_permutation(npg, seed=9)
    tables = {r: np.array(perm[160 * r:160 * r + 160], np.int32) for r in range(len(total))}
    done = {r: 0 for r in range(len(total))}
    logits = [torch.empty(64, spec.vocab, device="cuda") for _ in models]
    for si, step in enumerate(steps):
        seqs, rows, t = [], [], 0
        for r, n in step:
            seqs.append((hist[r][done[r]:done[r] + n], done[r], tables[r]))
            t += n
            rows.append(t - 1)
            if n <= 8:  # every row of the short chunks
                rows[-1:] = list(range(t - n, t))
            done[r] += n
        batch = vd.StepBatch(seqs, logit_rows=rows)
        for m, p, lg in zip(models, pools, logits):
            m.step(p, batch, lg)
        torch.cuda.synchronize()
        R = len(rows)
        assert np.array_equal(bits(logits[0][:R]), bits(logits[1][:R])), f"step {si}: fold and split modes differ"
    for m in models:
        assert m.device_status() == 0


def test_fold_mode_validation():
    ready()
    spec = synth.TINY
    W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=1).items()}
    m = vd.Model(spec, W, max_tokens=64, max_seqs=4, max_logit_rows=8, max_context=256)
    for bad in (-1, 3):
        with pytest.raises(vd.VDError):
            m.set_attention_fold(bad)
