"""vd_step_sample: the token choice fused into the LM-head GEMM epilogue.

The fused path must give the logits of vd_step bit for bit and the tokens
vd_sample picks from them (same scores, same (largest, lowest index) rule),
for greedy and Gumbel rows, eagerly and under graph replay, and with the
logits not stored at all.
"""

import numpy as np
import pytest
import torch

from gpu_util import bits, ready
from invariant_vd_step_gb300 import synth, vd

pytestmark = pytest.mark.gpu

# vocabulary of 393 LM-head tiles: not a multiple of the standalone sampler's chunk
WIDE = synth.TINY.with_(name="tiny-wide-vocab", vocab=50304)


def _samplers(R, salt):
    return [(salt * 100003 + r, 5 * r + salt, (0.0, 0.7, 1.3)[r % 3]) for r in range(R)]


class Twin:
    """One model, two pools: the two-call path on pool a, the fused path on pool b."""

    def __init__(self, spec, zero=False, graphs=0):
        self.spec = spec
        W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=3, gain_std=0.1, zero=zero).items()}
        self.W = W
        self.m = vd.Model(spec, W, max_tokens=256, max_seqs=16, max_logit_rows=256, max_context=512)
        self.m.set_graph_mode(graphs)
        self.pa, self.pb = vd.KVPool(self.m, 128), vd.KVPool(self.m, 128)
        self.la = torch.empty(256, spec.vocab, device="cuda")
        self.lb = torch.empty(256, spec.vocab, device="cuda")
        self.ta = torch.empty(256, dtype=torch.int32, device="cuda")
        self.tb = torch.empty(256, dtype=torch.int32, device="cuda")

    def both(self, batch, samplers, store_logits=True):
        R = batch.num_logit_rows
        self.m.step(self.pa, batch, self.la)
        self.m.sample(self.la, samplers, self.ta)
        self.m.step_sample(self.pb, batch, samplers, self.lb if store_logits else None, self.tb)
        torch.cuda.synchronize()
        if store_logits:
            assert np.array_equal(bits(self.la[:R]), bits(self.lb[:R])), "fused step changed the logits"
        ta, tb = self.ta[:R].cpu().numpy(), self.tb[:R].cpu().numpy()
        assert np.array_equal(ta, tb), f"tokens differ at rows {np.flatnonzero(ta != tb)[:8]}"
        return ta


@pytest.mark.parametrize("graphs", [0, 8])
def test_fused_tokens_and_logits_match_step_then_sample(graphs):
    ready()
    tw = Twin(WIDE, graphs=graphs)
    prompts = synth.make_prompts(6, 16, 40, WIDE.vocab, seed=11)
    perm = synth.page_permutation(128, seed=2)
    tables = [np.array(perm[8 * r:8 * r + 8], np.int32) for r in range(6)]
    seqs = [(p, 0, tables[r]) for r, p in enumerate(prompts)]
    T = sum(len(p) for p in prompts)
    # prefill with a logit row for every token
    toks = tw.both(vd.StepBatch(seqs, logit_rows=range(T)), _samplers(T, 1))
    last = [toks[int(np.sum([len(q) for q in prompts[:r + 1]])) - 1] for r in range(6)]
    ctx = [len(p) for p in prompts]
    for step in range(4):
        seqs = [(np.array([last[r]], np.int32), ctx[r], tables[r]) for r in range(6)]
        toks = tw.both(vd.StepBatch(seqs, logit_rows=range(6)), _samplers(6, 2 + step), store_logits=step != 2)
        last = list(toks)
        ctx = [c + 1 for c in ctx]
    assert tw.m.device_status() == 0


def test_fused_ties_and_zero_logits():
    ready()
    tw = Twin(WIDE, zero=True)
    prompts = synth.make_prompts(3, 17, 30, WIDE.vocab, seed=5)
    seqs = [(p, 0, np.arange(8 * r, 8 * r + 8, dtype=np.int32)) for r, p in enumerate(prompts)]
    T = sum(len(p) for p in prompts)
    toks = tw.both(vd.StepBatch(seqs, logit_rows=range(T)), _samplers(T, 9))
    greedy = np.arange(T) % 3 == 0
    assert np.all(toks[greedy] == 0), "all-equal logits must pick index 0"


def test_step_sample_validation():
    ready()
    tw = Twin(synth.TINY)
    seqs = [(np.array([1, 2, 3], np.int32), 0, np.array([0], np.int32))]
    b = vd.StepBatch(seqs, logit_rows=[2])
    with pytest.raises(vd.VDError):
        tw.m.step_sample(tw.pa, b, [(1, 0, 0.0)], tw.la, None)  # tokens_out required
    rows = vd.StepBatch([(np.arange(4, dtype=np.int32), 0, np.array([1], np.int32))], logit_rows=[])
    tw.m.step_sample(tw.pa, rows, [], None, None)  # no logit rows: nothing to choose
    torch.cuda.synchronize()


@pytest.mark.parametrize("graphs", [0, 8])
def test_device_fed_tokens_match_host_fed(graphs):
    """Decode steps whose tokens come from the previous step's device output
    equal steps fed the same tokens from the host, logits and tokens bitwise."""
    ready()
    tw = Twin(WIDE, graphs=graphs)
    prompts = synth.make_prompts(5, 16, 40, WIDE.vocab, seed=21)
    tables = [np.arange(8 * r, 8 * r + 8, dtype=np.int32) for r in range(5)]
    lens = [len(p) for p in prompts]
    rows = list(np.cumsum(lens) - 1)
    pre = vd.StepBatch([(p, 0, tables[r]) for r, p in enumerate(prompts)], logit_rows=rows)
    samp = _samplers(5, 4)
    # prefill both pools; tokens of the last prompt positions seed the decode loop
    tw.m.step_sample(tw.pa, pre, samp, tw.la, tw.ta)
    tw.m.step_sample(tw.pb, pre, samp, tw.lb, tw.tb)
    torch.cuda.synchronize()
    host_tok = tw.ta[:5].cpu().numpy()
    fed_logits = []
    ctx = list(lens)
    for step in range(6):
        zeros = [(np.zeros(1, np.int32), ctx[r], tables[r]) for r in range(5)]
        b_host = vd.StepBatch([(np.array([host_tok[r]], np.int32), ctx[r], tables[r]) for r in range(5)],
                              logit_rows=range(5))
        b_fed = vd.StepBatch(zeros, logit_rows=range(5))
        samp = _samplers(5, 10 + step)
        # fed path: never read back inside the loop; feed buffer = its own tokens_out
        lb = torch.empty(5, WIDE.vocab, device="cuda")
        tw.m.step_sample_fed(tw.pb, b_fed, np.arange(5), tw.tb, samp, lb, tw.tb)
        fed_logits.append(lb)
        tw.m.step_sample(tw.pa, b_host, samp, tw.la, tw.ta)
        torch.cuda.synchronize()
        assert np.array_equal(bits(tw.la[:5]), bits(lb)), f"step {step}: fed logits differ"
        host_tok = tw.ta[:5].cpu().numpy()
        assert np.array_equal(host_tok, tw.tb[:5].cpu().numpy())
        ctx = [c + 1 for c in ctx]
    assert tw.m.device_status() == 0


def test_fed_token_outside_vocabulary_is_reported():
    ready()
    tw = Twin(synth.TINY)
    seqs = [(np.array([1, 2, 3], np.int32), 0, np.array([3], np.int32))]
    feed = torch.tensor([synth.TINY.vocab + 5, 7], dtype=torch.int32, device="cuda")
    b = vd.StepBatch(seqs, logit_rows=[2])
    tw.m.step_sample_fed(tw.pa, b, [-1, 0, -1], feed, [(1, 0, 0.0)], tw.la, tw.ta)
    assert tw.m.device_status() == vd.VD_ERR_OUT_OF_RANGE
    assert tw.m.device_status() == 0  # reading clears it
    tw.m.step_sample_fed(tw.pa, b, [-1, 1, -1], feed, [(1, 0, 0.0)], tw.la, tw.ta)
    assert tw.m.device_status() == 0
    with pytest.raises(vd.VDError):
        tw.m.step_sample_fed(tw.pa, b, [-2, 0, -1], feed, [(1, 0, 0.0)], tw.la, tw.ta)
