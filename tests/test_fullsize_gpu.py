"""Full-size workloads of the pages' shapes: sampled oracle parity and invariance.

* 8B-shaped layer + LM head, decode batch of 256 over contexts U[512, 8192]
  (the bench workload): sampled rows against the oracle given the same
  cached K/V, and every row bitwise equal to the same request run alone.
* Full 32-layer 8B shape, continuous batching of 64 requests (prompts
  U[1024, 4096], 256 decode tokens) under chunk budgets 2048 and 8192:
  every emitted row bitwise equal across the two executions (compared
  through 64-bit fingerprints of the logits bits) and identical tokens.
* Gemma-3-4B shape (QK-norm, GeGLU, 5:1 local/global, window 1024),
  32 requests (prompts U[2048, 8192], 128 decode tokens) under batch sizes
  32 / 8 and budgets 4096 / 512, plus 4 requests run one at a time.
The oracle cannot compute a 32- or 34-layer forward over thousands of
tokens in test time, so the deep models are checked through the
invariance property, which holds at any size; their kernels are the same
ones the oracle checks on the smaller shapes.
"""

import numpy as np
import pytest
import torch

from gpu_util import ATOL, RTOL, bits, f64, ready
from invariant_vd_step_gb300 import engine, synth, vd

pytestmark = pytest.mark.gpu


def _fingerprint(rows: torch.Tensor) -> np.ndarray:
    w = _fingerprint.w
    if w is None or w.numel() != rows.shape[1]:
        g = torch.Generator(device="cuda")
        g.manual_seed(12345)
        w = torch.randint(-2 ** 62, 2 ** 62, (rows.shape[1],), generator=g, device="cuda", dtype=torch.int64)
        _fingerprint.w = w
    return (rows.contiguous().view(torch.int32).to(torch.int64) * w).sum(dim=1).cpu().numpy()


_fingerprint.w = None


def test_llama8b_layer_decode_b256_sampled_oracle_and_batch_invariance():
    ready()
    from oracle.decoder import OracleDecoder
    from oracle.bf16 import bits_to_f64
    spec = synth.LLAMA8B_1L
    B = 256
    ctx = synth.make_context_lengths(B, 512, 8192, seed=3)
    need = [(int(c) + 16) // 16 + 1 for c in ctx]
    perm = synth.page_permutation(int(sum(need)), seed=2)
    tables, k = [], 0
    for n in need:
        tables.append(perm[k:k + n])
        k += n
    W = synth.make_weights(spec, seed=0, device="cuda")
    model = vd.Model(spec, W, max_tokens=B, max_seqs=B, max_logit_rows=B, max_context=8192 + 32)
    mem = torch.empty(model.pool_bytes(len(perm)), dtype=torch.uint8, device="cuda")
    pool = vd.KVPool(model, len(perm), memory=mem)
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    pv = mem.view(torch.bfloat16)
    pv.copy_(torch.randn(pv.numel(), generator=g, device="cuda").to(torch.bfloat16))
    toks = synth.make_tokens(B, spec.vocab, seed=9)
    full = vd.StepBatch([(toks[i:i + 1], int(ctx[i]), tables[i]) for i in range(B)], logit_rows=range(B))
    logits = torch.empty((B, spec.vocab), device="cuda")
    model.step(pool, full, logits)
    torch.cuda.synchronize()
    # the same request alone (its K/V slot is rewritten with the same value)
    one = torch.empty((1, spec.vocab), device="cuda")
    for i in (0, 77, 255):
        model.step(pool, vd.StepBatch([(toks[i:i + 1], int(ctx[i]), tables[i])], logit_rows=[0]), one)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits(one)[0], bits(logits)[i])
    # sampled rows against the oracle over the same cached K/V
    dec = OracleDecoder(spec, synth.weights_to_numpy(W))
    pool6 = pv[: spec.n_layers * len(perm) * 2 * spec.n_kv_heads * 16 * spec.head_dim].view(
        spec.n_layers, len(perm), 2, spec.n_kv_heads, 16, spec.head_dim)
    for i in (3, 200):
        c = int(ctx[i])
        pg = torch.as_tensor(tables[i][:(c + 15) // 16], dtype=torch.long, device="cuda")
        kv = synth.bf16_to_u16(pool6[:, pg])  # [L][np][2][Hkv][16][hd]
        cache = []
        for layer in range(spec.n_layers):
            K = kv[layer][:, 0].transpose(0, 2, 1, 3).reshape(-1, spec.n_kv_heads, spec.head_dim)[:c]
            V = kv[layer][:, 1].transpose(0, 2, 1, 3).reshape(-1, spec.n_kv_heads, spec.head_dim)[:c]
            cache.append((bits_to_f64(K), bits_to_f64(V)))
        ref, _ = dec.step(np.array([toks[i]]), cache)
        got = f64(logits)[i]
        d = np.abs(got - ref[0])
        # At this shape a single bf16 flip anywhere in the layer moves the
        # logits by ~1e-2 (see test_oracle_noise_floor.py): the stated
        # tolerance must hold on >= 99.99% of the logits, and every logit
        # stays within twice it.
        within = d <= ATOL + RTOL * np.abs(ref[0])
        assert within.mean() >= 0.9999, (within.size - within.sum(), d.max())
        assert np.all(d <= 2 * (ATOL + RTOL * np.abs(ref[0]))), d.max()


def _run_engine(spec, W, prompts, max_new, budget, max_batch, num_pages, max_ctx, seed=5):
    model = vd.Model(spec, W, max_tokens=budget, max_seqs=max_batch, max_logit_rows=max_batch,
                     max_context=max_ctx)
    pool = vd.KVPool(model, num_pages)
    eng = engine.Engine(None, num_pages, max_batch=max_batch, token_budget=budget, prefix_reuse=True,
                        placement_seed=seed)
    rids = [eng.add_request(p, max_new, seed=1000 + i) for i, p in enumerate(prompts)]
    logits = torch.empty((max_batch, spec.vocab), device="cuda")
    tok = torch.empty(max_batch, dtype=torch.int32, device="cuda")
    fp = {r: [] for r in rids}

    def on_step(ids, rows, toks):
        for r, f, t in zip(ids, _fingerprint(rows), toks):
            fp[int(r)].append((int(f), int(t)))

    eng.run_native(model, pool, logits, tok, on_step=on_step)
    assert model.device_status() == 0
    st = eng.stats
    del pool
    model.close()
    return fp, st


def _assert_views_equal(a, b, rids=None):
    for r in (rids if rids is not None else a):
        assert len(a[r]) == len(b[r]) and a[r] == b[r], f"request {r} differs"


def test_llama8b_32_layers_continuous_batching_budgets_2048_vs_8192():
    ready()
    spec = synth.LLAMA8B
    prompts = synth.make_prompts(64, 1024, 4096, spec.vocab, seed=1)
    W = synth.make_weights(spec, seed=0, device="cuda")
    pages = sum((len(p) + 256 + 15) // 16 for p in prompts) + 64
    a, sa = _run_engine(spec, W, prompts, 256, 2048, 64, pages, 4096 + 256 + 16, seed=5)
    b, sb = _run_engine(spec, W, prompts, 256, 8192, 64, pages, 4096 + 256 + 16, seed=6)
    assert sum(len(v) for v in a.values()) == 64 * 256
    _assert_views_equal(a, b)


def test_gemma3_4b_batch_and_budget_invariance():
    ready()
    spec = synth.GEMMA3_4B
    prompts = synth.make_prompts(32, 2048, 8192, spec.vocab, seed=7)
    W = synth.make_weights(spec, seed=0, device="cuda")
    pages = sum((len(p) + 128 + 15) // 16 for p in prompts) + 32
    mc = 8192 + 128 + 16
    ref, _ = _run_engine(spec, W, prompts, 128, 4096, 32, pages, mc, seed=1)
    for budget, batch in ((512, 32), (4096, 8), (512, 8)):
        got, _ = _run_engine(spec, W, prompts, 128, budget, batch, pages, mc, seed=budget + batch)
        _assert_views_equal(ref, got)
    alone, _ = _run_engine(spec, W, prompts[:4], 128, 4096, 1, pages, mc, seed=9)
    _assert_views_equal(alone, {r: ref[r] for r in alone})


def test_gemma_block_32k_context_prefill_decode_pairs():
    """Prefill–decode pairs at a 32,768-token context on the Gemma-3 block
    (embedding scale, (1 + w) gains, sandwich norms, QK-norm, GeGLU, 5:1
    local/global with window 1024): logits of the last positions computed
    inside prefill chunks equal those computed by single-token decode steps
    over the same history, bitwise, under two chunk budgets."""
    ready()
    spec = synth.GEMMA3_4B.with_(name="gemma3-4b-shape-2layer", n_layers=2, local_global_period=2)
    n = 32768
    hist = synth.make_tokens(n, spec.vocab, seed=21)
    W = synth.make_weights(spec, seed=0, gain_std=0.1, device="cuda")
    tail = [n - 4, n - 3, n - 2, n - 1]
    pages = (n + 15) // 16
    table = np.arange(pages, dtype=np.int32)[::-1].copy()  # pages in reverse order

    def run(budget, decode_tail):
        model = vd.Model(spec, W, max_tokens=budget, max_seqs=1, max_logit_rows=budget, max_context=n + 16)
        pool = vd.KVPool(model, pages)
        logits = torch.empty((budget, spec.vocab), device="cuda")
        out = {}
        end = n - 4 if decode_tail else n
        for a in range(0, end, budget):
            b = min(end, a + budget)
            rows = [p - a for p in tail if a <= p < b]
            model.step(pool, vd.StepBatch([(hist[a:b], a, table)], logit_rows=rows), logits)
            for j, p in enumerate(p for p in tail if a <= p < b):
                out[p] = logits[j].clone()
        if decode_tail:
            for p in tail:
                model.step(pool, vd.StepBatch([(hist[p:p + 1], p, table)], logit_rows=[0]), logits)
                out[p] = logits[0].clone()
        torch.cuda.synchronize()
        assert model.device_status() == 0
        del pool
        model.close()
        return {p: bits(v) for p, v in out.items()}

    pre = run(4096, False)
    dec = run(4096, True)
    other = run(2048, True)
    for p in tail:
        assert np.array_equal(pre[p], dec[p]), f"position {p}: prefill and decode logits differ"
        assert np.array_equal(dec[p], other[p]), f"position {p}: budgets 4096 and 2048 differ"


def test_gemma3_block_decode_b32_sampled_oracle_and_batch_invariance():
    """Gemma-3-4B-shaped block (2 layers: one local window-1024, one global;
    hd 256, QK-norm, GeGLU, embedding scale, (1 + w) gains, sandwich norms,
    vocab 262144), 32 decode rows over contexts U[2048, 8192] with random
    cached K/V: rows alone equal the batch bitwise, and sampled rows meet the
    same derived criterion as the 8B layer against the oracle given the same
    cached K/V."""
    ready()
    from oracle.decoder import OracleDecoder
    from oracle.bf16 import bits_to_f64
    spec = synth.GEMMA3_4B.with_(name="gemma3-4b-shape-2layer", n_layers=2, local_global_period=2)
    B = 32
    ctx = synth.make_context_lengths(B, 2048, 8192, seed=13)
    need = [(int(c) + 16) // 16 + 1 for c in ctx]
    perm = synth.page_permutation(int(sum(need)), seed=14)
    tables, k = [], 0
    for n in need:
        tables.append(perm[k:k + n])
        k += n
    W = synth.make_weights(spec, seed=0, gain_std=0.1, device="cuda")
    model = vd.Model(spec, W, max_tokens=B, max_seqs=B, max_logit_rows=B, max_context=8192 + 32)
    mem = torch.empty(model.pool_bytes(len(perm)), dtype=torch.uint8, device="cuda")
    pool = vd.KVPool(model, len(perm), memory=mem)
    g = torch.Generator(device="cuda")
    g.manual_seed(15)
    pv = mem.view(torch.bfloat16)
    pv.copy_(torch.randn(pv.numel(), generator=g, device="cuda").to(torch.bfloat16))
    toks = synth.make_tokens(B, spec.vocab, seed=16)
    full = vd.StepBatch([(toks[i:i + 1], int(ctx[i]), tables[i]) for i in range(B)], logit_rows=range(B))
    logits = torch.empty((B, spec.vocab), device="cuda")
    model.step(pool, full, logits)
    torch.cuda.synchronize()
    one = torch.empty((1, spec.vocab), device="cuda")
    for i in (0, 17, 31):
        model.step(pool, vd.StepBatch([(toks[i:i + 1], int(ctx[i]), tables[i])], logit_rows=[0]), one)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits(one)[0], bits(logits)[i])
    assert model.device_status() == 0
    dec = OracleDecoder(spec, synth.weights_to_numpy(W))
    pool6 = pv[: spec.n_layers * len(perm) * 2 * spec.n_kv_heads * 16 * spec.head_dim].view(
        spec.n_layers, len(perm), 2, spec.n_kv_heads, 16, spec.head_dim)
    for i in (5, 26):
        c = int(ctx[i])
        pg = torch.as_tensor(tables[i][:(c + 15) // 16], dtype=torch.long, device="cuda")
        kv = synth.bf16_to_u16(pool6[:, pg])
        cache = []
        for layer in range(spec.n_layers):
            K = kv[layer][:, 0].transpose(0, 2, 1, 3).reshape(-1, spec.n_kv_heads, spec.head_dim)[:c]
            V = kv[layer][:, 1].transpose(0, 2, 1, 3).reshape(-1, spec.n_kv_heads, spec.head_dim)[:c]
            cache.append((bits_to_f64(K), bits_to_f64(V)))
        ref, _ = dec.step(np.array([toks[i]]), cache)
        d = np.abs(f64(logits)[i] - ref[0])
        # The Gemma block's noise floor is wider than the 8B layer's (one 1e-5
        # disagreement already puts ~1e-4 of the logits beyond the stated
        # tolerance; test_oracle_noise_floor.py): within it on >= 99.9 %, twice
        # it everywhere.
        within = d <= ATOL + RTOL * np.abs(ref[0])
        assert within.mean() >= 0.999, (within.size - within.sum(), d.max())
        assert np.all(d <= 2 * (ATOL + RTOL * np.abs(ref[0]))), d.max()
