"""The fast (split-K, non-invariant) path and decode-verify-rollback on top of it.

* The fast path computes the same model: its logits meet the oracle tolerance
  (a split-K bug would otherwise only show up as rollbacks).
* Decode-verify-rollback releases exactly the tokens of plain invariant
  decoding, and the verified logits are bitwise the invariant decode logits,
  with and without candidates corrupted on the host to force rollbacks.
"""

import numpy as np
import pytest
import torch

from gpu_util import assert_logits_close, bits, f64, ready
from invariant_vd_step_gb300 import llm42, synth, vd
from oracle.fp32 import Fp32Decoder

pytestmark = pytest.mark.gpu


def _model(spec, seed=3, max_rows=256):
    W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=seed, gain_std=0.1).items()}
    return W, vd.Model(spec, W, max_tokens=512, max_seqs=16, max_logit_rows=max_rows, max_context=1024)


@pytest.mark.parametrize("spec", [synth.TINY, synth.TINY.with_(name="tiny-geglu-hd128", head_dim=128,
                                                                act="geglu")], ids=lambda s: s.name)
def test_fast_path_logits_meet_the_oracle_tolerance(spec):
    ready()
    Wc = synth.make_weights(spec, seed=3, gain_std=0.1)
    W = {k: v.cuda() for k, v in Wc.items()}
    m = vd.Model(spec, W, max_tokens=512, max_seqs=16, max_logit_rows=256, max_context=1024)
    m.set_reduction_mode(1)
    pool = vd.KVPool(m, 64)
    h = synth.make_tokens(40, spec.vocab, seed=5)
    pt = np.arange(4, dtype=np.int32)
    lg = torch.empty(40, spec.vocab, device="cuda")
    m.step(pool, vd.StepBatch([(h[:30], 0, pt)], logit_rows=range(30)), lg[:30])
    for p in range(30, 40):  # decode steps on the fast path
        m.step(pool, vd.StepBatch([(h[p:p + 1], p, pt)], logit_rows=[0]), lg[p:p + 1])
    torch.cuda.synchronize()
    ref = Fp32Decoder(spec, synth.weights_to_numpy(Wc)).forward_all(h)
    assert_logits_close(f64(lg), ref)
    assert m.device_status() == 0


def _plain_invariant(m, pool, prompts, max_new, base_page=0):
    """Reference: invariant prefill, then one invariant decode step per token."""
    m.set_reduction_mode(0)
    out, lgs = {}, {}
    lg = torch.empty(1, m.spec.vocab, device="cuda")
    tok = torch.empty(1, dtype=torch.int32, device="cuda")
    for rid, p in enumerate(prompts):
        pages = np.arange(base_page + 16 * rid, base_page + 16 * rid + 16, dtype=np.int32)
        seq, toks = np.asarray(p, np.int32), []
        m.step_sample(pool, vd.StepBatch([(seq, 0, pages)], logit_rows=[len(seq) - 1]), [(100 + rid, 0, 0.0)], lg,
                      tok)
        toks.append(int(tok.item()))
        lgs[(rid, 0)] = lg[0].clone()
        for i in range(1, max_new):
            pos = len(seq) + i - 1
            m.step_sample(pool, vd.StepBatch([(np.array([toks[-1]], np.int32), pos, pages)], logit_rows=[0]),
                          [(100 + rid, i, 0.0)], lg, tok)
            toks.append(int(tok.item()))
            lgs[(rid, i)] = lg[0].clone()
        out[rid] = toks
    return out, lgs


class _Corrupting(llm42.SelectiveDecoder):
    """Host-side fault injection: every third candidate is replaced by another
    token, so verification must roll back and repair the K/V."""

    n = 0

    def _fast_step(self, live):
        super()._fast_step(live)
        for r in live:
            _Corrupting.n += 1
            if _Corrupting.n % 3 == 0:
                r.cand[-1] = (r.cand[-1] + 1) % self.m.spec.vocab


@pytest.mark.parametrize("window", [4, 8])
@pytest.mark.parametrize("corrupt", [False, True])
def test_decode_verify_rollback_releases_the_invariant_tokens(window, corrupt):
    ready()
    spec = synth.TINY
    W, m = _model(spec)
    pool = vd.KVPool(m, 256)
    prompts = synth.make_prompts(5, 20, 60, spec.vocab, seed=8)
    max_new = 30
    ref, ref_lg = _plain_invariant(m, pool, prompts, max_new)
    cls = _Corrupting if corrupt else llm42.SelectiveDecoder
    dec = cls(m, pool, pages=range(128, 256), window=window, max_batch=8, keep_logits=True)
    for rid, p in enumerate(prompts):
        assert dec.add_prompt(p, max_new, seed=100 + rid) == rid
    got = dec.run()
    for rid in range(len(prompts)):
        assert got[rid] == ref[rid], f"request {rid}: released tokens differ from invariant decoding"
        for i in range(max_new):
            assert np.array_equal(bits(dec.verified_logits[(rid, i)]), bits(ref_lg[(rid, i)])), (rid, i)
    st = dec.stats
    assert st.verify_steps > 0 and st.fast_steps > 0
    if corrupt:
        assert st.rolled_back > 0
    assert m.device_status() == 0


def test_a_changed_reduction_strategy_is_visible_in_the_bits():
    """Negative check for the first failure source the pages list (a kernel
    whose reduction strategy follows something other than the row): the same
    rows computed with split-K GEMMs differ from the invariant rows in their
    bits, though they agree within the stated tolerance, so the bitwise
    comparisons of the invariance tests do detect such a change."""
    ready()
    spec = synth.LLAMA8B_1L
    W = synth.make_weights(spec, seed=0, device="cuda")
    m = vd.Model(spec, W, max_tokens=256, max_seqs=8, max_logit_rows=8, max_context=1024)
    pool = vd.KVPool(m, 64)
    toks = synth.make_tokens(8 * 30, spec.vocab, seed=2).reshape(8, 30)  # 240 tokens: the fast path splits K
    seqs = [(toks[i], 0, np.arange(2 * i, 2 * i + 2, dtype=np.int32)) for i in range(8)]
    rows = [30 * i + 29 for i in range(8)]
    out = []
    for mode in (0, 1, 0):
        m.set_reduction_mode(mode)
        lg = torch.empty(8, spec.vocab, device="cuda")
        m.step(pool, vd.StepBatch(seqs, logit_rows=rows), lg)
        torch.cuda.synchronize()
        out.append(lg)
    assert np.array_equal(bits(out[0]), bits(out[2]))           # the invariant path repeats itself
    assert not np.array_equal(bits(out[0]), bits(out[1]))       # split-K changes bits
    d = (out[0] - out[1]).abs().max().item()
    assert d < 5e-2, d                                           # but computes the same model (noise floor)
