"""End-to-end engine step through the C ABI: oracle parity and invariance."""

import numpy as np
import pytest
import torch

from gpu_util import assert_logits_close, bits, f64, ready
from invariant_vd_step_gb300 import synth, vd
from oracle.fp32 import Fp32Decoder

pytestmark = pytest.mark.gpu

GEMMA_TINY = synth.ModelSpec("gemma-tiny", 3, 256, 2, 1, 256, 512, 512, act="geglu", qk_norm=True,
                             rope_theta=1e6, rope_theta_local=1e4, sliding_window=24, local_global_period=2,
                             rms_eps=1e-6, embed_scale=True, norm_offset=True, sandwich_norm=True)
LLAMA_TINY128 = synth.ModelSpec("llama-tiny-128", 2, 512, 8, 2, 128, 1024, 1024, rope_theta=5e5,
                                rope_theta_local=5e5)


class Runner:
    """Runs teacher-forced schedules of chunks; pages handed out from a permutation."""

    def __init__(self, spec, seed=0, gain_std=0.1, num_pages=256, zero=False, max_tokens=512, max_context=1024,
                 mode="eager"):
        self.spec = spec
        self.Wc = synth.make_weights(spec, seed=seed, gain_std=gain_std, zero=zero)
        self.W = {k: v.cuda() for k, v in self.Wc.items()}
        self.model = vd.Model(spec, self.W, max_tokens=max_tokens, max_seqs=32, max_logit_rows=max_tokens,
                              max_context=max_context)
        # launch modes that must not change a bit: graph replay of steps,
        # and decode attention folding all of a row's KV splits in one CTA
        if "graph" in mode:
            self.model.set_graph_mode(16)
        if "fold" in mode:
            self.model.set_attention_fold(1)
        self.pool = vd.KVPool(self.model, num_pages)
        self.num_pages = num_pages
        self.logits = torch.empty((max_tokens, spec.vocab), device="cuda")

    def execute(self, histories, steps, perm_seed=None):
        """steps: list of lists of (request, n_new_tokens).  Returns {(r, pos): logits bits row}."""
        perm = synth.page_permutation(self.num_pages, seed=perm_seed) if perm_seed is not None \
            else np.arange(self.num_pages, dtype=np.int32)
        nxt = 0
        tables = {r: [] for r in range(len(histories))}
        done = {r: 0 for r in range(len(histories))}
        out = {}
        for step in steps:
            seqs, keys = [], []
            for r, n in step:
                c = done[r]
                need = (c + n + 15) // 16
                while len(tables[r]) < need:
                    tables[r].append(int(perm[nxt]))
                    nxt += 1
                seqs.append((histories[r][c:c + n], c, np.array(tables[r], np.int32)))
                keys += [(r, c + i) for i in range(n)]
                done[r] = c + n
            T = len(keys)
            # one logits buffer for every step: graph replay keys a step on its output address
            logits = self.logits[:T]
            logits.fill_(float("nan"))
            self.model.step(self.pool, vd.StepBatch(seqs, logit_rows=range(T)), logits)
            torch.cuda.synchronize()
            for i, k in enumerate(keys):
                out[k] = logits[i].clone()
        self.tables = tables
        return out

    def oracle_all(self, history):
        return Fp32Decoder(self.spec, synth.weights_to_numpy(self.Wc)).forward_all(history)


MODES = ["eager", "graph", "fold", "graph+fold"]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("spec", [synth.TINY, GEMMA_TINY, LLAMA_TINY128], ids=lambda s: s.name)
def test_step_logits_vs_oracle(spec, mode):
    ready()
    run = Runner(spec, seed=1, mode=mode)
    hist = synth.make_prompts(3, 20, 70, spec.vocab, seed=2)
    hist = [np.concatenate([h, synth.make_tokens(5, spec.vocab, seed=10 + i)]) for i, h in enumerate(hist)]
    L = [len(h) for h in hist]
    steps = [[(0, L[0] - 5), (1, 16)], [(1, L[1] - 21), (2, L[2] - 5)]]
    steps += [[(0, 1), (1, 1), (2, 1)] for _ in range(5)]
    res = run.execute(hist, steps, perm_seed=3)
    if "graph" in mode:
        assert run.model.graph_stats()["replays"] >= 2
    for r, h in enumerate(hist):
        ref = run.oracle_all(h)
        got = np.stack([f64(res[(r, p)]) for p in range(len(h))])
        assert_logits_close(got, ref)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("spec", [synth.TINY, LLAMA_TINY128, GEMMA_TINY], ids=lambda s: s.name)
def test_long_context_decode_vs_oracle(spec, mode):
    """Contexts past one and two 512-key splits (decode rows of several
    splits, merged in split order or folded in one CTA), prefilled in chunks
    of up to 512 tokens, then decode steps: every row against the oracle."""
    ready()
    run = Runner(spec, seed=2, mode=mode, num_pages=400, max_tokens=1024, max_context=2048)
    hist = synth.make_prompts(3, 500, 1100, spec.vocab, seed=4)
    hist = [np.concatenate([h, synth.make_tokens(6, spec.vocab, seed=20 + i)]) for i, h in enumerate(hist)]
    L = [len(h) for h in hist]
    steps, done = [], [0, 0, 0]
    while any(done[r] < L[r] - 6 for r in range(3)):
        step = []
        for r in range(3):
            n = min(L[r] - 6 - done[r], (300, 512, 170)[r])
            if n > 0:
                step.append((r, n))
                done[r] += n
        steps.append(step)
    steps += [[(0, 1), (1, 1), (2, 1)] for _ in range(6)]
    res = run.execute(hist, steps, perm_seed=5)
    if "graph" in mode:
        assert run.model.graph_stats()["replays"] >= 1
    for r, h in enumerate(hist):
        ref = run.oracle_all(h)
        tail = range(len(h) - 8, len(h))  # the prompt's last rows and every decode row
        got = np.stack([f64(res[(r, p)]) for p in tail])
        assert_logits_close(got, ref[list(tail)])


def test_zero_model_gives_zero_logits_bitwise():
    """The all-zero model returns the golden outputs (tests/golden/zero_model_outputs.txt):
    every logit +0.0 bit for bit, and greedy token id 0."""
    ready()
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "zero_model_outputs.txt")) as f:
        kv = dict(line.split() for line in f if line.strip() and not line.startswith("#"))
    want_bits, want_token = int(kv["logit_float32_bits"], 16), int(kv["greedy_token"])
    run = Runner(synth.TINY, zero=True)
    hist = synth.make_prompts(2, 10, 40, synth.TINY.vocab, seed=4)
    res = run.execute(hist, [[(0, len(hist[0])), (1, len(hist[1]))]])
    rows = torch.stack(list(res.values()))
    assert torch.all(rows.contiguous().view(torch.int32) == want_bits)
    tok = torch.empty(rows.shape[0], dtype=torch.int32, device="cuda")
    run.model.sample(rows, [(1, i, 0.0) for i in range(rows.shape[0])], tok)
    torch.cuda.synchronize()
    assert torch.all(tok == want_token)


def test_invariance_across_batching_chunking_and_pages():
    # Definition 2.1: per-request logit views are equal bit for bit whatever
    # the batch composition, chunk budget, prefill/decode split and pages.
    ready()
    spec = synth.TINY
    hist = synth.make_prompts(4, 30, 60, spec.vocab, seed=5, shared_prefix=32, n_sharing=2)
    L = [len(h) for h in hist]
    schedules = [
        ([[(r, L[r])] for r in range(4)], None),                                  # one request at a time
        ([[(r, L[r]) for r in range(4)]], 1),                                     # all in one step
        ([[(r, 16) for r in range(4)]] + [[(r, L[r] - 16) for r in range(4)]], 2),  # chunk 16 then rest
        ([[(0, 5), (1, 30)], [(0, L[0] - 5), (2, L[2])], [(1, L[1] - 30), (3, L[3] - 1)], [(3, 1)]], 3),
        ([[(r, 1)] for r in range(4) for _ in range(1)] + [[(r, L[r] - 1) for r in (2, 0, 3, 1)]], 4),
    ]
    ref = None
    for steps, seed in schedules:
        run = Runner(spec, seed=7, num_pages=64)
        res = run.execute(hist, steps, perm_seed=seed)
        b = {k: bits(v) for k, v in res.items()}
        if ref is None:
            ref = b
            continue
        for k in ref:
            np.testing.assert_array_equal(b[k], ref[k], err_msg=f"row {k}")


def test_kv_written_by_chunked_and_whole_prefill_is_bitwise_equal():
    # KV-value invariant: the slot of position p holds fKV(W, h, p) however
    # the prefix was scheduled.
    ready()
    spec = synth.TINY
    h = synth.make_tokens(90, spec.vocab, seed=8)
    kv = []
    for steps in ([[(0, 90)]], [[(0, 7)], [(0, 40)], [(0, 43)]]):
        run = Runner(spec, seed=9, num_pages=32)
        run.execute([h], steps, perm_seed=len(steps))
        per_layer = []
        for layer in range(spec.n_layers):
            k = torch.empty((90, spec.n_kv_heads, spec.head_dim), dtype=torch.bfloat16, device="cuda")
            v = torch.empty_like(k)
            run.model.copy_kv(run.pool, layer, run.tables[0], 90, k, v)
            torch.cuda.synchronize()
            per_layer.append((bits(k), bits(v)))
        kv.append(per_layer)
    for (ka, va), (kb, vb) in zip(*kv):
        np.testing.assert_array_equal(ka, kb)
        np.testing.assert_array_equal(va, vb)


def test_descriptor_validation_rejects_bad_steps():
    ready()
    run = Runner(synth.TINY, num_pages=8)
    lg = torch.empty((4, synth.TINY.vocab), device="cuda")
    m, p = run.model, run.pool
    cases = [
        (vd.StepBatch([(np.array([1, 2]), 0, np.array([99]))], [0]), 3),        # page id out of range
        (vd.StepBatch([(np.array([1, 5000]), 0, np.array([1]))], [0]), 3),      # token id out of range
        (vd.StepBatch([(np.array([1] * 20), 0, np.array([1]))], [0]), 3),       # page table too narrow
        (vd.StepBatch([(np.array([1]), 0, np.array([1])), (np.array([2]), 0, np.array([1]))], [0]), 1),  # slot clash
        (vd.StepBatch([(np.array([1]), 0, np.array([1]))], [5]), 3),            # logit row out of range
    ]
    for b, code in cases:
        with pytest.raises(vd.VDError) as e:
            m.step(p, b, lg)
        assert e.value.code == code
    m.step(p, vd.StepBatch([]), lg)  # empty step is a no-op
    torch.cuda.synchronize()
    assert m.device_status() == 0
