"""Decode benchmark of the batch-invariant step on the Llama-3.1-8B shape.

Workload (one step = one pass of the whole hot path): one decoder layer of
the Llama-3.1-8B shape plus the LM head (d 4096, 32 q / 8 kv heads, hd 128,
SwiGLU 14336, vocab 128256), random-init bf16 weights N(0, 0.02), a pure
decode batch of B requests (default 256) whose cached contexts are
U[512, 8192] tokens, KV page size 16 with physical pages randomly permuted.
Each step: descriptor upload + validation, embedding, RMSNorm, QKV GEMM,
RoPE + KV write, paged attention + split merge, O GEMM + residual,
RMSNorm, gate/up GEMM + SwiGLU, down GEMM + residual, final norm, LM head
(fp32 logits), greedy token choice.  The cached K/V is seeded random
N(0, 1) bf16 (timing is independent of the values); each step appends one
token per request.

  value  -- decode tokens/s with inputs resident in HBM (device time, CUDA
            events on the launching stream, max over ranks).
  e2e    -- the same through the public API with host buffers: every step
            feeds the previous step's sampled tokens back, uploads the host
            descriptor and reads the sampled tokens back to the host.

The line also carries: the same step at B = 1, 8 and 64 (``decode_points``),
an 8192-token prefill step with each GEMM's TFLOP/s (``prefill``), repeated
K-step windows (``stability``), the 3,200-pair invariance matrix, and the
C++ oracle timed on the host cores for a sample of one step's rows
(``cpu_baseline``, with the GPU's parity on those rows).

Usage: python bench.py [--gpus N --steps K --warmup W --batch B]
       python bench.py --impl reference ...   (the C++ oracle, bounded sample)
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tok/s (Llama-8B shape, 1 GB300)"
UNIT = "tok/s"
CTX_LO, CTX_HI = 512, 8192


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def max_over_ranks(values, ws, device="cpu"):
    """Elementwise maximum of per-rank floats over all ranks: the slowest
    replica sets the job's time (a collective only when ws > 1)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if ws > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """Samples nvidia-smi clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), float(f[3]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        power_med = statistics.median(r[2] for r in rows)
        loaded = [r for r in rows if r[2] >= 0.5 * max(r[2] for r in rows)] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "power_w_median": power_med}


def make_workload(B: int, steps: int, seed_ctx: int = 3):
    from invariant_vd_step_gb300 import synth
    spec = synth.LLAMA8B_1L
    ctx = synth.make_context_lengths(B, CTX_LO, CTX_HI, seed=seed_ctx)
    need = [(int(c) + steps + 15) // 16 for c in ctx]
    num_pages = int(sum(need))
    perm = synth.page_permutation(num_pages, seed=2)
    tables, k = [], 0
    for n in need:
        tables.append(perm[k:k + n].copy())
        k += n
    return spec, ctx, tables, num_pages


def traffic_of(kernel, alg_bytes_per_launch):
    """DRAM bytes of one launch, scaled from the committed ncu capture of a
    smaller launch of the same kernel (traffic grows with the bytes
    streamed); None when no capture covers the kernel."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)[kernel]
        return int(round(t["dram_over_algorithmic"] * alg_bytes_per_launch))
    except Exception:
        return None


def algorithmic_bytes(spec, ctx_lens, B):
    """Per decode step: weights + KV read/write + activations, and per kernel."""
    d, hd, Hq, Hkv, F, V = spec.d_model, spec.head_dim, spec.n_heads, spec.n_kv_heads, spec.ffn_dim, spec.vocab
    L = spec.n_layers
    kv_tok = 2 * Hkv * hd * 2  # K+V bytes per token per layer
    attn = L * (int(np.sum(ctx_lens + 1)) * kv_tok + B * Hq * hd * 2)  # K/V read incl. the new token + q read
    w_layer = (spec.qkv_dim * d + d * spec.attn_dim + 2 * F * d + d * F) * 2 + 2 * d * 2
    lm = V * d * 2
    kernels = {
        "attention": attn,
        "gemm_qkv": L * (spec.qkv_dim * d * 2 + B * (d + spec.qkv_dim) * 2),
        "gemm_o": L * (d * spec.attn_dim * 2 + B * (spec.attn_dim + 2 * d) * 2),
        "gemm_gate_up": L * (2 * F * d * 2 + B * (d + F) * 2),
        "gemm_down": L * (d * F * 2 + B * (F + 2 * d) * 2),
        "gemm_lm_head": lm + B * (d * 2 + V * 4),
    }
    total = L * w_layer + lm + attn + L * B * kv_tok + B * V * 4
    return total, kernels


def gemm_plans(spec, T, R):
    """The tile shape (weight rows, tokens, K blocks per weight copy) each GEMM
    of a step over T tokens with R logit rows takes (LM head with the fused
    token choice)."""
    from invariant_vd_step_gb300 import vd
    d, F = spec.d_model, spec.ffn_dim
    glu = vd.EPI_GEGLU if spec.act == "geglu" else vd.EPI_SWIGLU
    return {
        "gemm_qkv": list(vd.gemm_plan(T, spec.qkv_dim, d, vd.EPI_BF16)),
        "gemm_o": list(vd.gemm_plan(T, d, spec.attn_dim, vd.EPI_RESIDUAL)),
        "gemm_gate_up": list(vd.gemm_plan(T, F, d, glu)),
        "gemm_down": list(vd.gemm_plan(T, d, F, vd.EPI_RESIDUAL)),
        "gemm_lm_head": list(vd.gemm_plan(R, spec.vocab, d, 5)),
    }


def decode_sweep_point(spec, weights, B, K, Wm, graphs, dev, hbm):
    """One point of the decode batch sweep: the bench workload at batch B
    (contexts U[512, 8192], permuted pages, random cached K/V), K timed steps
    of vd_step_sample after Wm warm-up steps, graph replay; device time."""
    import torch
    from invariant_vd_step_gb300 import synth, vd
    spec_, ctx, tables, num_pages = make_workload(B, Wm + K + 1)
    model = vd.Model(spec, weights, max_tokens=max(B, 16), max_seqs=B, max_logit_rows=B,
                     max_context=CTX_HI + Wm + K + 32)
    mem = torch.empty(model.pool_bytes(num_pages), dtype=torch.uint8, device=dev)
    pool = vd.KVPool(model, num_pages, memory=mem)
    g = torch.Generator(device=dev)
    g.manual_seed(4)
    pv = mem.view(torch.bfloat16)
    for i in range(0, pv.numel(), 1 << 28):
        n = min(1 << 28, pv.numel() - i)
        pv[i:i + n] = torch.randn(n, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    width = max(len(t) for t in tables)
    pt2d = np.zeros((B, width), dtype=np.int32)
    for i, t in enumerate(tables):
        pt2d[i, :len(t)] = t
    toks = synth.make_tokens(B * (Wm + K), spec.vocab, seed=1).reshape(Wm + K, B)
    cu, rows = np.arange(B + 1, dtype=np.int32), np.arange(B, dtype=np.int32)
    batches = [vd.StepBatch.from_arrays(toks[s], cu, ctx + s, pt2d, rows) for s in range(Wm + K)]
    logits = torch.empty((B, spec.vocab), dtype=torch.float32, device=dev)
    out_tok = torch.empty(B, dtype=torch.int32, device=dev)
    samplers = [(1000 + i, 0, 0.0) for i in range(B)]
    stream = torch.cuda.current_stream(dev)
    model.set_graph_mode(graphs)
    for s in range(Wm):
        model.step_sample(pool, batches[s], samplers, logits, out_tok, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(Wm, Wm + K):
        model.step_sample(pool, batches[s], samplers, logits, out_tok, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    assert model.device_status() == 0
    total, _ = algorithmic_bytes(spec, ctx + Wm, B)
    pool.close()
    model.close()
    del mem
    roof_ms = total / (hbm * 1e9) * 1e3
    return {"batch": B, "tok_s": round(B / (ms * 1e-3), 1), "ms_per_step": round(ms, 4),
            "step_roofline_frac": round(roof_ms / ms, 4), "roofline_tok_s": round(B / (roof_ms * 1e-3), 1)}


def run_gpu(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    import __graft_entry__
    __graft_entry__.build()
    from invariant_vd_step_gb300 import synth, vd

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B, K, Wm = args.batch, args.steps, args.warmup
    total_steps = Wm + K + 2 * args.e2e_steps + 2  # warm-up, timed, synchronous and pipelined e2e
    spec, ctx, tables, num_pages = make_workload(B, total_steps)
    weights = synth.make_weights(spec, seed=0, device=dev)
    model = vd.Model(spec, weights, max_tokens=max(B, 16), max_seqs=B, max_logit_rows=B,
                     max_context=CTX_HI + total_steps + 16)
    mem = torch.empty(model.pool_bytes(num_pages), dtype=torch.uint8, device=dev)
    pool = vd.KVPool(model, num_pages, memory=mem)
    g = torch.Generator(device=dev)
    g.manual_seed(4)
    pv = mem.view(torch.bfloat16)
    for i in range(0, pv.numel(), 1 << 28):  # random N(0,1) cached K/V
        n = min(1 << 28, pv.numel() - i)
        pv[i:i + n] = torch.randn(n, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    stream = torch.cuda.current_stream(dev)
    toks = synth.make_tokens(B * total_steps, spec.vocab, seed=1).reshape(total_steps, B)

    width = max(len(t) for t in tables)
    pt2d = np.zeros((B, width), dtype=np.int32)
    for i, t in enumerate(tables):
        pt2d[i, :len(t)] = t
    cu = np.arange(B + 1, dtype=np.int32)
    rows = np.arange(B, dtype=np.int32)

    def batch_at(step, tok_row):
        return vd.StepBatch.from_arrays(tok_row, cu, ctx + step, pt2d, rows)

    batches = [batch_at(s, toks[s]) for s in range(Wm + K)]
    logits = torch.empty((B, spec.vocab), dtype=torch.float32, device=dev)
    out_tok = torch.empty(B, dtype=torch.int32, device=dev)
    samplers = [(1000 + i, 0, 0.0) for i in range(B)]

    def one(s):
        model.step_sample(pool, batches[s], samplers, logits, out_tok, stream)

    model.set_graph_mode(args.graphs)  # 0: eager launches
    model.set_attention_fold(args.attention_fold)
    for s in range(Wm):
        one(s)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    windows = []
    with Clocks(local) as clk:
        ev0.record(stream)
        for s in range(Wm, Wm + K):
            one(s)
        ev1.record(stream)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        # the same K steps again, window after window (each step rewrites its
        # token's K/V slot with the same value), so that the clock record and
        # the spread of the step time cover at least 200 steps
        for _ in range(max(0, -(-200 // K) - 1)):
            w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            w0.record(stream)
            for s in range(Wm, Wm + K):
                one(s)
            w1.record(stream)
            torch.cuda.synchronize()
            windows.append(w0.elapsed_time(w1) / K)
    ms = ev0.elapsed_time(ev1)
    graph_stats = model.graph_stats()
    # Per-kernel times: the same K steps again, eager, with events around
    # every kernel class (profiling forces eager launches).
    model.profile_collect()
    model.profile(True)
    ep0, ep1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ep0.record(stream)
    for s in range(Wm, Wm + K):
        one(s)
    ep1.record(stream)
    torch.cuda.synchronize()
    model.profile(False)
    prof = model.profile_collect()
    prof_ms = ep0.elapsed_time(ep1)
    assert model.device_status() == 0, "a bounded on-device wait timed out"

    # ---- end to end through the C ABI from host buffers: every step uploads its
    # descriptor and sampler states from pinned host memory and reads its sampled
    # tokens back.  Synchronous loop: tokens go to the host and back each step.
    # Pipelined loop: step s+1 takes step s's tokens on the device
    # (vd_step_sample_fed) and is enqueued before step s's tokens are read.
    host_tok = torch.empty((2, B), dtype=torch.int32, pin_memory=True)
    last = toks[Wm + K - 1].astype(np.int32)
    base = Wm + K
    max_pages = (CTX_HI + total_steps + 16 + 15) // 16

    def h2d_bytes(step):
        need = (int(np.max(ctx)) + step + 16) // 16  # page-table columns the library uploads
        if args.graphs:  # graph mode rounds the stride up to 64 pages
            need = min((need + 63) // 64 * 64, max_pages)
        return 4 * (3 * B + 2 * (B + 1) + 3 * B + B * need + B) + 24 * B  # descriptor + sampler states

    E = args.e2e_steps
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(E):
        model.step_sample(pool, batch_at(base + s, last), samplers, logits, out_tok, stream)
        host_tok[0].copy_(out_tok, non_blocking=True)
        stream.synchronize()
        last = host_tok[0].numpy().copy()
    e2e_sync_s = time.perf_counter() - t0
    base += E
    feed_idx = np.arange(B, dtype=np.int32)
    zeros = np.zeros(B, dtype=np.int32)
    evs = [torch.cuda.Event(), torch.cuda.Event()]
    emitted = []
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(E):
        if s == 0:
            model.step_sample(pool, batch_at(base, last), samplers, logits, out_tok, stream)
        else:
            model.step_sample_fed(pool, batch_at(base + s, zeros), feed_idx, out_tok, samplers, logits, out_tok,
                                  stream)
        host_tok[s % 2].copy_(out_tok, non_blocking=True)
        evs[s % 2].record(stream)
        if s >= 1:
            evs[(s - 1) % 2].synchronize()
            emitted.append(host_tok[(s - 1) % 2].numpy().copy())
    evs[(E - 1) % 2].synchronize()
    emitted.append(host_tok[(E - 1) % 2].numpy().copy())
    e2e_s = time.perf_counter() - t0
    h2d = h2d_bytes(base + E - 1)
    assert len(emitted) == E and model.device_status() == 0
    # one more decode step, with every row's logits stored, for the CPU
    # baseline to recompute a sample of its rows (outside the timed region)
    check_step = base + E
    check_toks = toks[check_step % len(toks)]
    model.step(pool, batch_at(check_step, check_toks), logits, stream)
    torch.cuda.synchronize()
    check_logits = logits.cpu().numpy()

    ms_max, e2e_max, e2e_sync_max = max_over_ranks([ms, e2e_s, e2e_sync_s], ws,
                                                   dev if ws > 1 and dist.get_backend() == "nccl" else "cpu")
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    hbm, tf, peak_kind = load_peaks()
    total_bytes, kbytes = algorithmic_bytes(spec, ctx, B)
    plans = gemm_plans(spec, B, B)
    step_ms = ms_max / K
    kernels = {}
    for name, (n, nk, tot) in prof.items():
        per_step = tot / K
        e = {"launches_per_step": n / K, "kernels_per_step": nk / K, "ms_per_step": round(per_step, 5),
             "share": round(tot / prof_ms, 4)}
        if name in kbytes:
            gbs = kbytes[name] / (per_step * 1e-3) / 1e9
            e.update({"algorithmic_bytes": kbytes[name], "GB_s": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4)})
        if name in plans:
            e["plan_bm_bn_kpo"] = plans[name]
        kernels[name] = e
    dom = max((k for k in kernels if k in kbytes), key=lambda k: kernels[k]["ms_per_step"])
    dk = kernels[dom]
    launches = sum(int(round(v["kernels_per_step"])) for v in kernels.values())
    step_gbs = total_bytes / (step_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(ws * B * K / (ms_max * 1e-3), 1), "unit": UNIT, "n_gpus": ws,
        "steps": K, "warmup": Wm, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "llama3.1-8b-shape 1 decoder layer + LM head, pure decode",
                   "batch": B, "ctx": f"U[{CTX_LO},{CTX_HI}] mean {float(np.mean(ctx)):.0f}",
                   "page_size": 16, "pages": "randomly permuted", "parallelism": f"replicas x{ws}",
                   "launch": f"CUDA graph replay (<= {args.graphs} graphs)" if args.graphs else "eager launches",
                   "attention_fold": ["default (split)", "fold", "split"][args.attention_fold],
                   "l2": f"inputs larger than L2 ({total_bytes / 1e9:.2f} GB read+written per step)"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": dk["GB_s"], "peak": hbm, "unit": "GB/s",
                     "frac": dk["hbm_frac"], "traffic": traffic_of(dom, kbytes[dom] / max(1, round(dk["launches_per_step"]))),
                     "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": int(kbytes[dom] / max(1, round(dk["launches_per_step"])))},
        "step_roofline": {"algorithmic_bytes": total_bytes, "GB_s": round(step_gbs, 1),
                          "frac": round(step_gbs / hbm, 4)},
        "kernels": kernels,
        "gpu_launches": launches * K,
        "graphs": {"max_graphs": args.graphs, **graph_stats,
                   "eager_profiled_ms_per_step": round(prof_ms / K, 4)},
        "e2e": {"value": round(ws * B * args.e2e_steps / e2e_max, 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4 * B, "steps": args.e2e_steps,
                "loop": "pipelined: step s+1 takes step s's tokens on the device and is enqueued before "
                        "step s's tokens are read back",
                "synchronous_value": round(ws * B * args.e2e_steps / e2e_sync_max, 1)},
        "clocks": clk.summary(),
    }
    if not args.no_invariance:
        from invariant_vd_step_gb300 import invariance
        r = invariance.run_matrix()
        line["invariance"] = {"pairs": r.pairs, "bitwise_equal": r.equal, "pass_pct": round(r.pass_pct, 3),
                              "categories": r.categories, "runs": r.runs,
                              "workload": "tiny llama-style decoder, 8 requests, 16 greedy decode steps"}
    if windows:
        line["stability"] = {"windows": len(windows) + 1, "steps_per_window": K,
                             "ms_per_step_median": round(statistics.median([step_ms] + windows), 4),
                             "ms_per_step_min": round(min([step_ms] + windows), 4),
                             "ms_per_step_max": round(max([step_ms] + windows), 4),
                             "note": "value is the first window; the clock record covers all windows"}
    if not args.no_points:
        # decode at B = 1, 8 and 64 (same workload, graph replay) and the 8192-token prefill step
        line["decode_points"] = {str(b): decode_sweep_point(spec, weights, b, K, Wm, args.graphs, dev, hbm)
                                 for b in (1, 8, 64)}
        line["prefill"] = prefill_result(dev, 8192, 4, max(5, min(K, 20)), Wm)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, weights, ctx + check_step, tables, mem, check_toks, check_logits,
                                            args.cpu_sample)
    if args.sweep:
        line["sweep"] = [decode_sweep_point(spec, weights, b, 10, 3, args.graphs, dev, hbm)
                         for b in (1, 2, 4, 8, 16, 32, 64, 128, 256)]
    print(json.dumps(line))
    if ws > 1:
        dist.destroy_process_group()


def prefill_result(dev, T, nreq, K, Wm, attn_kernel=0):
    """One prefill step of T new tokens (nreq requests of T / nreq tokens
    from an empty cache) through the layer + LM head: prefill tok/s and each
    GEMM's TFLOP/s against the measured bf16 tensor peak (sustained).
    attn_kernel: the prefill-class attention kernel (0 tcgen05, 1 mma.sync)."""
    import torch
    from invariant_vd_step_gb300 import synth, vd
    spec = synth.LLAMA8B_1L
    per = T // nreq
    weights = synth.make_weights(spec, seed=0, device=dev)
    model = vd.Model(spec, weights, max_tokens=T, max_seqs=nreq, max_logit_rows=nreq, max_context=per + 16)
    model.set_attention_prefill(attn_kernel)
    npg = (per + 15) // 16
    pool = vd.KVPool(model, nreq * npg)
    toks = synth.make_tokens(T, spec.vocab, seed=1)
    tables = synth.page_permutation(nreq * npg, seed=2).reshape(nreq, npg)
    b = vd.StepBatch.from_arrays(toks[:per * nreq], np.arange(nreq + 1, dtype=np.int32) * per,
                                 np.zeros(nreq, np.int32), tables, np.arange(1, nreq + 1) * per - 1)
    logits = torch.empty((nreq, spec.vocab), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(Wm):
        model.step(pool, b, logits, stream)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(dev.index or 0) as clk:
        ev0.record(stream)
        for _ in range(K):
            model.step(pool, b, logits, stream)
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    # per-kernel times: the same K steps again with events around every kernel class
    model.profile_collect()
    model.profile(True)
    for _ in range(K):
        model.step(pool, b, logits, stream)
    torch.cuda.synchronize()
    model.profile(False)
    prof = model.profile_collect()
    assert model.device_status() == 0
    pool.close()
    model.close()
    hbm, tf_burst, peak_kind = load_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tf_sust = float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        tf_sust = 1700.0
    d, F = spec.d_model, spec.ffn_dim
    Tt = per * nreq
    flops = {"gemm_qkv": 2 * Tt * spec.qkv_dim * d, "gemm_o": 2 * Tt * d * spec.attn_dim,
             "gemm_gate_up": 2 * Tt * 2 * F * d, "gemm_down": 2 * Tt * d * F,
             "gemm_lm_head": 2 * nreq * spec.vocab * d}
    # causal attention: 4 * Hq * hd flops per visible key (QK^T and PV)
    flops_attn = 4 * spec.n_heads * spec.head_dim * nreq * per * (per + 1) // 2
    kernels = {}
    for name, (n, nk, tot) in prof.items():
        per_step = tot / K
        e = {"kernels_per_step": nk / K, "ms_per_step": round(per_step, 4), "share": round(tot / ms, 4)}
        if name in flops:
            tfs = flops[name] / (per_step * 1e-3) / 1e12
            e.update({"TFLOP_s": round(tfs, 1), "tensor_frac": round(tfs / tf_sust, 4)})
        if name == "attention":
            e["TFLOP_s"] = round(flops_attn / (per_step * 1e-3) / 1e12, 1)
        kernels[name] = e
    dom = max((k for k in kernels if k in flops), key=lambda k: kernels[k]["ms_per_step"])
    gemm_ms = sum(kernels[k]["ms_per_step"] for k in kernels if k in flops)
    gemm_tf = sum(flops.values()) / (gemm_ms * 1e-3) / 1e12
    return {
        "value": round(Tt * K / (ms * 1e-3), 1), "unit": "tok/s", "ms_per_step": round(ms / K, 4), "steps": K,
        "warmup": Wm, "tokens_per_step": Tt, "requests": nreq,
        "workload": "llama3.1-8b-shape 1 decoder layer + LM head, prefill from an empty cache",
        "attention_kernel": "tcgen05" if attn_kernel == 0 and spec.head_dim in (64, 128) else "mma.sync",
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": kernels[dom]["TFLOP_s"], "peak": tf_sust,
                     "unit": "TFLOP/s", "frac": kernels[dom]["tensor_frac"], "traffic": None,
                     "peak_source": peak_kind + " (sustained)"},
        "gemms": {"TFLOP_s": round(gemm_tf, 1), "frac_of_sustained": round(gemm_tf / tf_sust, 4),
                  "frac_of_burst": round(gemm_tf / tf_burst, 4)},
        "kernels": kernels, "clocks": clk.summary()}


def run_prefill(args):
    """Prefill mode: one step of --tokens new tokens (--prefill-requests
    requests from an empty cache) through the same layer + LM head."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    r = prefill_result(dev, args.tokens, args.prefill_requests, args.steps, args.warmup,
                       0 if args.prefill_attention == "tc" else 1)
    print(json.dumps({
        "metric": "prefill tok/s (Llama-8B shape, 1 GB300)", "value": r["value"], "unit": "tok/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": r["workload"], "tokens_per_step": r["tokens_per_step"], "requests": r["requests"],
                   "page_size": 16, "pages": "randomly permuted"},
        "roofline": r["roofline"], "gemms": r["gemms"], "kernels": r["kernels"], "clocks": r["clocks"]}))


def run_ceiling(args):
    """Ceiling mode: for each GEMM of the decode step (the Llama-3.1-8B-shaped
    layer + LM head) at B tokens, the time of one launch, replayed from a CUDA
    graph over copies of the weight matrix that together exceed L2, of
    (a) the plan's weight copies alone (vd_op_tma_stream), (b) the plan's
    weight and activation copies, (c) the same weight bytes over every SM
    (K cut into parts), and (d) the GEMM itself with that plan; each as
    weight GB/s and a fraction of the measured HBM peak."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from invariant_vd_step_gb300 import synth, vd
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm, _, peak_kind = load_peaks()
    spec = synth.LLAMA8B_1L
    d, F = spec.d_model, spec.ffn_dim
    glu = vd.EPI_SWIGLU
    gemms = [("gemm_qkv", spec.qkv_dim, d, vd.EPI_BF16), ("gemm_o", d, spec.attn_dim, vd.EPI_RESIDUAL),
             ("gemm_gate_up", F, d, glu), ("gemm_down", d, F, vd.EPI_RESIDUAL),
             ("gemm_lm_head", spec.vocab, d, vd.EPI_F32)]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rows_out = []

    def timed(fn, n):
        for i in range(n):  # warm-up (first launches set attributes; nothing is captured yet)
            fn(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream()
        with torch.cuda.graph(g, stream=cs):
            for i in range(n):
                fn(i)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (3 * n)

    # What one thread issuing MMAs costs (the GEMM's issuer is built around it):
    # 896 MMAs of 128 x N x 16, 16 per stage, with no test, a test_wait or a
    # try_wait of a completed mbarrier phase per stage (the stage's MMAs
    # waiting for its result), or the test issued one stage ahead; SM clock
    # cycles per MMA.
    issue = []
    cyc = torch.zeros(2, dtype=torch.int64, device=dev)
    for N in (16, 32, 64, 128, 256):
        for wait, wname in ((0, "none"), (1, "test_wait"), (2, "try_wait"), (3, "test_wait one stage ahead")):
            vals = []
            for _ in range(3):
                vd.mma_issue_probe(128, N, 896, wait, cyc)
                torch.cuda.synchronize()
                vals.append(cyc.cpu().tolist())
            best = min(vals, key=lambda v: v[1])
            issue.append({"M": 128, "N": N, "per_stage_wait": wname, "mmas": 896,
                          "cycles_per_mma_issue": round(best[0] / 896, 1),
                          "cycles_per_mma_complete": round(best[1] / 896, 1)})
    only = set(args.ceiling_gemms.split(",")) if args.ceiling_gemms else None
    for T in [int(t) for t in args.ceiling_batches.split(",")]:
        for name, N, K, epi in gemms:
            if only and name not in only:
                continue
            rows = 2 * N if epi == glu else N
            wbytes = rows * K * 2
            copies = max(1, -(-400_000_000 // wbytes))  # together past L2 (129 MB)
            Ws = [synth.make_normal_bf16((rows, K), seed=10 + i, std=0.02).to(dev) for i in range(copies)]
            bucket = 1
            while bucket < T:
                bucket <<= 1
            X = synth.make_normal_bf16((bucket, K), seed=3).to(dev)
            bm, bn, kpo = vd.gemm_plan(T, N, K, epi)
            xrows = min(bn, bucket)
            out_dt = torch.float32 if epi == vd.EPI_F32 else torch.bfloat16
            C = torch.empty((T, N), dtype=out_dt, device=dev)
            Xt = X[:T].contiguous()
            R = torch.zeros((T, N), dtype=torch.bfloat16, device=dev) if epi == vd.EPI_RESIDUAL else None
            kparts = 1
            while (rows // bm) * kparts * 2 <= sms and (K // 64) % (kpo * kparts * 2) == 0:
                kparts *= 2
            n = max(4, copies)
            t_w = timed(lambda i: vd.tma_stream(Ws[i % copies], bm, kpo), n)
            t_wx = timed(lambda i: vd.tma_stream(Ws[i % copies], bm, kpo, X, xrows), n)
            t_all = timed(lambda i: vd.tma_stream(Ws[i % copies], bm, kpo, k_parts=kparts), n)
            t_g = timed(lambda i: vd.gemm(Xt, Ws[i % copies], C, epi, R), n)
            row = {"gemm": name, "tokens": T, "weight_MB": round(wbytes / 1e6, 1), "plan_bm_bn_kpo": [bm, bn, kpo],
                   "row_tiles": rows // bm}
            if args.ceiling_sweep:  # the GEMM under every forced plan the matrix allows
                sweep = {}
                for fbm in (64, 128, 256):
                    for fbn in (16, 32, 64, 128, 256):
                        for fk in (1, 2, 4):
                            if rows % fbm or (K // 64) % fk or (fbm == 256 and fk > 1) or fbn > max(16, bucket):
                                continue
                            vd.set_gemm_plan(fbm, fbn, fk)
                            try:
                                if tuple(vd.gemm_plan(T, N, K, epi)) != (fbm, fbn, fk):
                                    continue
                                sweep[f"{fbm}x{fbn}x{fk}"] = round(timed(lambda i: vd.gemm(Xt, Ws[i % copies], C, epi, R), n) * 1e3, 2)
                            finally:
                                vd.set_gemm_plan(0, 0, 0)
                best = min(sweep, key=sweep.get)
                row["plan_sweep_us"] = sweep
                row["best_plan"] = {"plan": best, "us": sweep[best]}
            for tag, t in (("stream_plan", t_w), ("stream_plan_with_activations", t_wx),
                           (f"stream_all_sms_k{kparts}", t_all), ("gemm_launch", t_g)):
                gbs = wbytes / (t * 1e-3) / 1e9
                row[tag] = {"us": round(t * 1e3, 2), "GB_s": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4)}
            rows_out.append(row)
            del Ws, X, C, Xt, R
            torch.cuda.empty_cache()
    print(json.dumps({"metric": "decode GEMM weight-stream ceilings (Llama-8B shape, 1 GB300)", "unit": "GB/s",
                      "peak": hbm, "peak_source": peak_kind, "launch": "one launch per graph node, replayed",
                      "l2": "weight copies rotated, together > 400 MB", "mma_issue": issue, "rows": rows_out}))


def step_roofline_s(spec, seqs, R, hbm_gbs, tf_peak):
    """Roofline time of one engine step: max(algorithmic bytes / HBM, flops / tensor peak).

    seqs: (cached_len, q_len) per request.  Bytes: every layer's weights, the
    LM head and fp32 logits when rows are returned, each request's visible
    K/V read once per layer, its new K/V written.  Flops: the GEMMs over the
    step's tokens plus 4 * Hq * hd per (query, visible key) pair."""
    L, d, F, V = spec.n_layers, spec.d_model, spec.ffn_dim, spec.vocab
    per_layer = spec.qkv_dim * d + d * spec.attn_dim + 3 * F * d
    T = sum(q for _, q in seqs)
    kvb = 2 * spec.n_kv_heads * spec.head_dim * 2
    byts = L * per_layer * 2 + (V * d * 2 + R * V * 4 if R else 0)
    flops = 2 * per_layer * T * L + 2 * V * d * R
    for c, q in seqs:
        for i in range(L):
            w = spec.layer_window(i)
            vis_last = min(c + q, w) if w else c + q
            byts += vis_last * kvb + q * kvb
            if w:
                pairs = sum(min(t + 1, w) for t in range(c, c + q)) if q < 64 else q * min(c + q, w)
            else:
                pairs = q * c + q * (q + 1) // 2
            flops += 4 * spec.n_heads * spec.head_dim * pairs
    return max(byts / (hbm_gbs * 1e9), flops / (tf_peak * 1e12)), T


def run_serve(args):
    """Serving workloads through the native engine (plan -> vd_step_sample ->
    tokens to the host -> commit), full 32-layer Llama-3.1-8B shape:

    c3: 64 requests, prompts U[1024, 4096], 256 decode tokens each, chunk
        budget --budget (2048 or 8192), prefill and decode rows mixed.
    c5: agentic sessions: a shared 4096-token prefix; every turn appends
        U[200, 800] tokens and decodes U[128, 512]; --sessions x --turns at
        --concurrency sessions in flight; prefix reuse on and a pool of half of
        concurrency x mean final session length, which forces evictions and
        recomputation.

    A step that carries prompt tokens counts as prefill (its tokens minus its
    decode rows are prefill tokens); a step of decode rows only counts as
    decode.  Reports tok/s of each kind over its own steps, all computed
    tokens over the wall clock, and the wall-clock roofline fraction (sum of
    per-step roofline times / time)."""
    if args.workload == "c4":
        return run_serve_c4(args)
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from invariant_vd_step_gb300 import engine, sessions, synth, vd
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    spec = synth.LLAMA8B
    V = spec.vocab
    budget = args.budget
    if args.workload == "c3":
        prompts = synth.make_prompts(64, 1024, 4096, V, seed=1)
        work = sessions.SessionWorkload(V, 64, 1, decode_lo=256, decode_hi=256, prompts=prompts)
        conc = 64
        pages = sum((len(p) + 256 + 15) // 16 for p in prompts) + 64
    else:
        conc = args.concurrency
        work = sessions.SessionWorkload(V, args.sessions, args.turns, 200, 800, 128, 512,
                                        prefix=synth.make_tokens(4096, V, seed=11), seed=args.seed)
        mean_final = 4096 + args.turns * (500 + 320)
        pages = max(int(0.5 * conc * mean_final / 16), work.max_context() // 16 + 64)
    weights = synth.make_weights(spec, seed=0, device=dev)
    model = vd.Model(spec, weights, max_tokens=budget, max_seqs=conc, max_logit_rows=conc,
                     max_context=work.max_context())
    model.set_graph_mode(args.graphs)
    pool = vd.KVPool(model, pages)
    eng = engine.Engine(None, pages, max_batch=conc, token_budget=budget, prefix_reuse=True, placement_seed=2)
    stream = torch.cuda.current_stream(dev)
    logits = torch.empty((conc, V), dtype=torch.float32, device=dev)
    tok_dev = torch.empty(conc, dtype=torch.int32, device=dev)
    hbm, tf_burst, peak_kind = load_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tf_sust = float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        tf_sust = 1700.0
    torch.cuda.synchronize()
    t_start = time.perf_counter()
    with Clocks(local) as clk:
        res = sessions.run_sessions(work, model, pool, eng, conc, logits, tok_dev, stream)
    wall = time.perf_counter() - t_start
    assert model.device_status() == 0
    split = split_steps(spec, res.steps, hbm, tf_sust)
    total_T = split["tokens_computed"]
    gen = sum(len(t) for outs in res.outputs.values() for t in outs)
    print(json.dumps({
        "metric": f"serving tok/s ({args.workload}, Llama-3.1-8B shape 32 layers, 1 GB300)",
        "value": round(total_T / wall, 1), "unit": "tok/s (tokens computed: prefill chunks + decode)",
        "generated_tok_s": round(gen / wall, 1),
        "n_gpus": 1, "higher_is_better": True, "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "layers": spec.n_layers, "budget": budget, "max_batch": conc,
                   "sessions": work.n_sessions, "turns": work.turns, "pool_pages": pages, "graphs": args.graphs},
        "steps": len(res.steps), "wall_s": round(wall, 3),
        "prefill": split["prefill"], "decode": split["decode"],
        "roofline_frac": round(split["roofline_s"] / wall, 4),
        "tokens": {"prompt_submitted": res.submitted, "computed": total_T, "generated": gen},
        "engine": eng.stats, "graphs": model.graph_stats(), "clocks": clk.summary(),
        "peaks": {"hbm_gbs": hbm, "bf16_tflops_sustained": tf_sust, "source": peak_kind},
    }))


def split_steps(spec, steps, hbm, tf_sust):
    """Prefill and decode tok/s and roofline fractions over a run's steps.  A
    step that carries prompt tokens counts as prefill (its tokens minus its
    decode rows are prefill tokens); a step of decode rows only counts as
    decode."""
    t_pre = t_dec = roof_pre = roof_dec = 0.0
    n_pre_tok = n_dec_tok = total_T = 0
    for st in steps:
        T = sum(q for _, q in st.seqs)
        total_T += T
        roof, _ = step_roofline_s(spec, st.seqs, st.rows, hbm, tf_sust)
        if T > st.rows:  # the step carries prompt tokens
            t_pre += st.seconds
            roof_pre += roof
            n_pre_tok += T - sum(1 for c, q in st.seqs if q == 1 and c > 0)
        else:
            t_dec += st.seconds
            roof_dec += roof
            n_dec_tok += st.rows
    return {"steps": len(steps), "tokens_computed": total_T,
            "prefill": {"tok_s": round(n_pre_tok / max(t_pre, 1e-9), 1), "steps_s": round(t_pre, 3),
                        "roofline_frac": round(roof_pre / max(t_pre, 1e-9), 4)},
            "decode": {"tok_s": round(n_dec_tok / max(t_dec, 1e-9), 1), "steps_s": round(t_dec, 3),
                       "roofline_frac": round(roof_dec / max(t_dec, 1e-9), 4)},
            "gpu_steps_s": round(t_pre + t_dec, 3), "roofline_s": round(roof_pre + roof_dec, 4)}


def run_serve_c4(args):
    """C4: the Gemma-3-4B shape (34 layers: QK-norm, GeGLU, sandwich norms, 5
    local layers of window 1024 per global one) served by the native engine:
    32 requests, prompts U[2048, 8192], 128 decode tokens each, at batch
    {1, 8, 32} x chunk budget {512, 4096}.  Each run reports prefill and
    decode tok/s and roofline fractions over its own steps; every emitted
    row's logits (a fingerprint of their bits taken on the GPU: the sum and
    an index-weighted sum of the int32 views) and token are compared with
    the batch-1, budget-4096 run, the invariance pairs of this workload."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from invariant_vd_step_gb300 import engine, sessions, synth, vd
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    spec = synth.GEMMA3_4B
    V = spec.vocab
    n_req, dec = 32, 128
    prompts = synth.make_prompts(n_req, 2048, 8192, V, seed=1)
    work = sessions.SessionWorkload(V, n_req, 1, decode_lo=dec, decode_hi=dec, prompts=prompts)
    pages = sum((len(p) + dec + 15) // 16 for p in prompts) + 64
    weights = synth.make_weights(spec, seed=0, device=dev)
    model = vd.Model(spec, weights, max_tokens=4096, max_seqs=n_req, max_logit_rows=n_req,
                     max_context=work.max_context())
    model.set_graph_mode(args.graphs)
    pool = vd.KVPool(model, pages)
    stream = torch.cuda.current_stream(dev)
    logits = torch.empty((n_req, V), dtype=torch.float32, device=dev)
    tok_dev = torch.empty(n_req, dtype=torch.int32, device=dev)
    wvec = (torch.arange(V, device=dev, dtype=torch.int64) % 1021) + 1
    hbm, _, peak_kind = load_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tf_sust = float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        tf_sust = 1700.0
    runs = [(1, 4096), (1, 512), (8, 512), (8, 4096), (32, 512), (32, 4096)]  # the first is the reference
    out, prints = [], []
    with Clocks(local) as clk:
        for bsz, budget in runs:
            eng = engine.Engine(None, pages, max_batch=bsz, token_budget=budget, prefix_reuse=True, placement_seed=2)
            fp = {}

            def on_rows(sids, turns, lg, toks):
                bits = lg.view(torch.int32).to(torch.int64)
                f = torch.stack([bits.sum(dim=1), (bits * wvec).sum(dim=1)], 1).cpu().numpy()
                for i, sid in enumerate(sids):
                    fp.setdefault(sid, []).append((int(f[i, 0]), int(f[i, 1]), int(toks[i])))

            torch.cuda.synchronize()
            t0 = time.perf_counter()
            res = sessions.run_sessions(work, model, pool, eng, bsz, logits, tok_dev, stream, on_rows=on_rows)
            wall = time.perf_counter() - t0
            assert model.device_status() == 0
            row = {"batch": bsz, "budget": budget, "wall_s": round(wall, 3)}
            row.update(split_steps(spec, res.steps, hbm, tf_sust))
            out.append(row)
            prints.append(fp)
    ref = prints[0]
    pairs = equal = 0
    for fp in prints[1:]:
        for sid, rows in ref.items():
            for a, b in zip(rows, fp.get(sid, [])):
                pairs += 1
                equal += a == b
            pairs += abs(len(rows) - len(fp.get(sid, [])))
    print(json.dumps({
        "metric": "C4 serving (Gemma-3-4B shape, 34 layers, 1 GB300): tok/s and invariance pass %",
        "n_gpus": 1, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "c4", "requests": n_req, "prompts": "U[2048, 8192]", "decode_tokens": dec,
                   "pool_pages": pages, "graphs": args.graphs},
        "runs": out,
        "invariance": {"reference": "batch 1, budget 4096", "pairs": pairs, "bitwise_equal": equal,
                       "pass_pct": round(100.0 * equal / max(pairs, 1), 3),
                       "compared": "per emitted row: logits bit fingerprint and token"},
        "graphs": model.graph_stats(), "clocks": clk.summary(),
        "peaks": {"hbm_gbs": hbm, "bf16_tflops_sustained": tf_sust, "source": peak_kind},
    }))


def run_llm42(args):
    """Decode-verify-rollback against plain invariant decoding on the decode
    workload (Llama-3.1-8B-shaped layer + LM head, contexts U[lo, hi], random
    cached K/V, permuted pages): both loops emit --new-tokens tokens per
    request, one host sync per step; tok/s of released tokens."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from invariant_vd_step_gb300 import llm42, synth, vd
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B, N, Wn = args.batch, args.new_tokens, args.window
    spec, ctx, tables, num_pages = make_workload(B, N + Wn + 8)
    weights = synth.make_weights(spec, seed=0, device=dev)
    model = vd.Model(spec, weights, max_tokens=max(B * Wn, 16), max_seqs=B, max_logit_rows=B * Wn,
                     max_context=CTX_HI + N + Wn + 32)
    mem = torch.empty(model.pool_bytes(num_pages), dtype=torch.uint8, device=dev)
    pool = vd.KVPool(model, num_pages, memory=mem)
    g = torch.Generator(device=dev)
    g.manual_seed(4)
    pv = mem.view(torch.bfloat16)
    for i in range(0, pv.numel(), 1 << 28):
        n = min(1 << 28, pv.numel() - i)
        pv[i:i + n] = torch.randn(n, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    snapshot = mem.clone()  # both loops start from the same cached K/V
    first = synth.make_tokens(B, spec.vocab, seed=1)
    model.set_graph_mode(args.graphs)

    def plain():
        model.set_reduction_mode(0)
        lg = torch.empty((B, spec.vocab), dtype=torch.float32, device=dev)
        tok = torch.empty(B, dtype=torch.int32, device=dev)
        last, out = first.copy(), [[] for _ in range(B)]
        cu, rows = np.arange(B + 1, dtype=np.int32), np.arange(B, dtype=np.int32)
        width = max(len(t) for t in tables)
        pt = np.zeros((B, width), dtype=np.int32)
        for i, t in enumerate(tables):
            pt[i, :len(t)] = t
        for i in range(N):
            b = vd.StepBatch.from_arrays(last, cu, ctx + i, pt, rows)
            model.step_sample(pool, b, [(1000 + r, i, 0.0) for r in range(B)], lg, tok)
            last = tok.cpu().numpy()
            for r in range(B):
                out[r].append(int(last[r]))
        return out

    def selective():
        dec = llm42.SelectiveDecoder(model, pool, pages=[], window=Wn, max_batch=B)
        for r in range(B):
            dec.add_cached(int(ctx[r]), int(first[r]), tables[r], N, seed=1000 + r)
        got = dec.run()
        return [got[r] for r in range(B)], dec.stats

    for _ in range(2):  # warm-up both loops (graphs, split-K buffer)
        mem.copy_(snapshot)
        plain()
        mem.copy_(snapshot)
        selective()
    mem.copy_(snapshot)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ref = plain()
    t_plain = time.perf_counter() - t0
    mem.copy_(snapshot)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    got, st = selective()
    t_sel = time.perf_counter() - t0
    assert model.device_status() == 0
    same = sum(int(a == b) for a, b in zip(got, ref))
    print(json.dumps({
        "metric": "decode tok/s with decode-verify-rollback (Llama-8B shape, 1 GB300)",
        "value": round(B * N / t_sel, 1), "unit": "tok/s (released tokens)", "n_gpus": 1,
        "higher_is_better": True, "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "llama3.1-8b-shape 1 decoder layer + LM head, greedy decode from cached K/V",
                   "batch": B, "new_tokens": N, "window": Wn, "ctx": f"U[{CTX_LO},{CTX_HI}]",
                   "graphs": args.graphs},
        "invariant_decode_tok_s": round(B * N / t_plain, 1),
        "speedup": round(t_plain / t_sel, 3),
        "requests_identical_to_invariant_decoding": f"{same}/{B}",
        "fast_steps": st.fast_steps, "verify_steps": st.verify_steps, "candidates": st.candidates,
        "accepted": st.accepted, "rolled_back": st.rolled_back,
    }))


def oracle_decode_rows(spec, weights_np, caches, toks, threads):
    """The C++ oracle's decode step for each request over its cached K/V."""
    from oracle.fp32 import Fp32Decoder
    dec = Fp32Decoder(spec, weights_np, threads=threads)
    return [dec.step(np.array([toks[r]]), cache)[0][0] for r, cache in enumerate(caches)]


def cache_from_pages(spec, pages_u16, c):
    """pages_u16: [layers][n_pages][2][Hkv][16][hd] -> the oracle's cache of positions [0, c)."""
    from oracle.fp32 import KVCache
    kv = []
    for layer in range(spec.n_layers):
        p = pages_u16[layer]
        k = p[:, 0].transpose(0, 2, 1, 3).reshape(-1, spec.n_kv_heads, spec.head_dim)[:c]
        v = p[:, 1].transpose(0, 2, 1, 3).reshape(-1, spec.n_kv_heads, spec.head_dim)[:c]
        kv.append((k, v))
    return KVCache.from_bits(kv)


def literal_stats(got, ref):
    """The stated tolerance read literally (max-abs 2e-2 and max-rel 1e-2,
    each on its own) and combined as allclose combines them."""
    d, a = np.abs(got - ref), np.abs(ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(a > 0, d / a, np.where(d > 0, np.inf, 0.0))
    return {"logits": int(d.size), "max_abs": float(d.max()), "max_rel": float(rel.max()),
            "beyond_abs": int((d > 2e-2).sum()), "beyond_rel": int((d > 1e-2 * a).sum()),
            "beyond_combined": int((d > 2e-2 + 1e-2 * a).sum()),
            "beyond_twice_combined": int((d > 2 * (2e-2 + 1e-2 * a)).sum()), "mean_abs": float(d.mean())}


def cpu_model() -> str:
    """The host CPU's name from /proc/cpuinfo (x86 "model name"; on Arm the
    implementer/part codes), else the machine type."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if fields.get("model name"):
        return fields["model name"]
    if fields.get("CPU implementer"):
        return f"{platform.machine()} implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    return platform.machine() or "unknown"


def cpu_baseline(spec, weights, ctx_now, tables, mem, toks, gpu_logits, n_req):
    """Times the C++ oracle (as it stands) on this host's cores for a bounded
    sample of one decode step of the same workload: n_req rows spread over
    the context range on all cores, and 2 of them on one core.  The rows are
    the ones the GPU computed in its last (untimed) step, so the oracle's
    logits also give that step's parity against the stated tolerance."""
    from invariant_vd_step_gb300 import synth
    import torch
    w_np = synth.weights_to_numpy(weights)
    pool = mem.view(torch.int16)[: spec.n_layers * (mem.numel() // 2 // spec.n_layers)]
    pool = pool.view(spec.n_layers, -1, 2, spec.n_kv_heads, 16, spec.head_dim)
    order = np.argsort(ctx_now, kind="stable")
    rows = sorted({int(order[int(round(x))]) for x in np.linspace(0, len(ctx_now) - 1, n_req)})
    caches = []
    for r in rows:
        c = int(ctx_now[r])
        idx = torch.as_tensor(tables[r][:(c + 15) // 16], dtype=torch.long, device=mem.device)
        caches.append(cache_from_pages(spec, pool[:, idx].cpu().numpy().view(np.uint16), c))
    cores = os.cpu_count() or 1
    sel = [toks[r] for r in rows]
    t0 = time.perf_counter()
    refs = oracle_decode_rows(spec, w_np, caches, sel, cores)
    dt_all = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle_decode_rows(spec, w_np, caches[:2], sel[:2], 1)
    dt_one = time.perf_counter() - t0
    par = literal_stats(np.stack([gpu_logits[r].astype(np.float64) for r in rows]), np.stack(refs))
    return {"value": round(len(rows) / dt_all, 4), "unit": UNIT, "cores": cores, "cpu": cpu_model(), "kind": "oracle",
            "single_thread": {"value": round(2 / dt_one, 4), "unit": UNIT, "cores": 1},
            "sample": f"{len(rows)} decode rows of the same workload (1 layer + LM head, C++ float32 oracle) on "
                      f"{cores} threads in {dt_all:.1f} s; 2 of them on 1 thread in {dt_one:.1f} s",
            "parity_vs_gpu": dict(par, rows=len(rows),
                                  note="the GPU's logits of these rows against the oracle's, at the stated "
                                       "tolerance (max-abs 2e-2, max-rel 1e-2)")}


def run_cpu_baseline(args):
    """CPU-baseline mode (no GPU): the C++ oracle on the host cores, as it
    stands, on (a) the tiny-model workload end to end -- 8 requests with
    prompts of 17..64 tokens, 4 sharing a 32-token prefix, 16 greedy decode
    tokens each (cold prefill, then one decode step per token) -- and (b) one
    decode step of the Llama-3.1-8B-shaped layer + LM head at B = 1, 8 and
    32 over seeded N(0, 1) caches of U[512, 8192] tokens; each on one thread
    and on every core (threads split output features, so the results are
    the same bits)."""
    import torch
    from invariant_vd_step_gb300 import synth
    from oracle import sampler
    from oracle.fp32 import Fp32Decoder
    cores = os.cpu_count() or 1
    out = {"metric": "C++ oracle throughput on the host cores", "cpu": cpu_model(), "cores": cores, "kind": "oracle"}
    spec = synth.TINY
    W = synth.weights_to_numpy(synth.make_weights(spec, seed=0))
    prompts = synth.make_prompts(8, 17, 64, spec.vocab, seed=1, shared_prefix=32, n_sharing=4)
    tiny = {}
    for threads in (1, cores):
        dec = Fp32Decoder(spec, W, threads=threads)
        t0 = time.perf_counter()
        gen = 0
        for p in prompts:
            logits, cache = dec.step(p, dec.empty_cache())
            for _ in range(16):
                tok = sampler.argmax_lowest(logits[-1])
                gen += 1
                logits, cache = dec.step(np.array([tok]), cache)
        dt = time.perf_counter() - t0
        tiny[f"threads_{threads}"] = {"generated_tok_s": round(gen / dt, 1), "seconds": round(dt, 3)}
    out["tiny_end_to_end"] = dict(tiny, workload="tiny llama-style decoder, 8 requests (4 share a 32-token "
                                                  "prefix), prompts 17..64, 16 greedy tokens each")
    spec = synth.LLAMA8B_1L
    W = synth.weights_to_numpy(synth.make_weights(spec, seed=0))
    rng = np.random.default_rng(4)
    ctx = synth.make_context_lengths(32, CTX_LO, CTX_HI, seed=3)
    toks = synth.make_tokens(32, spec.vocab, seed=9)
    caches = []
    for r in range(32):
        c = int(ctx[r])
        shape = (spec.n_layers, (c + 15) // 16, 2, spec.n_kv_heads, 16, spec.head_dim)
        vals = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
        caches.append(cache_from_pages(spec, synth.bf16_to_u16(vals), c))
    decode = {}
    for B in (1, 8, 32):
        for threads in ((1, cores) if B == 1 else (cores,)):
            t0 = time.perf_counter()
            oracle_decode_rows(spec, W, caches[:B], toks[:B], threads)
            dt = time.perf_counter() - t0
            decode[f"B{B}_threads_{threads}"] = {"tok_s": round(B / dt, 3), "seconds": round(dt, 2)}
    out["decode_step_llama8b_layer"] = dict(decode, workload="llama3.1-8b-shape 1 decoder layer + LM head, one "
                                                            "decode step, contexts U[512,8192]")
    print(json.dumps(out))


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from invariant_vd_step_gb300 import synth
    B = args.batch
    spec, ctx, tables, num_pages = make_workload(B, 4)
    weights = synth.make_weights(spec, seed=0)
    w_np = synth.weights_to_numpy(weights)
    rng = np.random.default_rng(4)
    n_req = args.cpu_sample
    caches = []
    for r in range(n_req):  # seeded N(0,1) bf16 cached K/V of the sampled requests
        c = int(ctx[r])
        shape = (spec.n_layers, (c + 15) // 16, 2, spec.n_kv_heads, 16, spec.head_dim)
        import torch
        vals = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
        caches.append(cache_from_pages(spec, synth.bf16_to_u16(vals), c))
    toks = synth.make_tokens(n_req, spec.vocab, seed=9)
    cores = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle_decode_rows(spec, w_np, caches[:1], toks, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_decode_rows(spec, w_np, caches, toks, cores)
    dt = time.perf_counter() - t0
    v = round(n_req * args.steps / dt, 4)
    sample = f"{n_req} of the {B} decode rows per step (1 layer + LM head, C++ float32 oracle, {cores} threads)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "llama3.1-8b-shape 1 decoder layer + LM head, pure decode", "batch": B,
                   "ctx": f"U[{CTX_LO},{CTX_HI}]", "page_size": 16},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "cpu": cpu_model(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--batch", type=int, default=256)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--graphs", type=int, default=64,
                    help="decode: keep up to N captured step graphs (0 = eager launches)")
    ap.add_argument("--cpu-sample", type=int, default=8)
    ap.add_argument("--no-points", action="store_true", help="decode: leave out the B = 1 / 64 points and the prefill step")
    ap.add_argument("--prefill-attention", choices=["tc", "mma"], default="tc",
                    help="prefill mode: the prefill-class attention kernel (tcgen05 or mma.sync; the same bits)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-invariance", action="store_true")
    ap.add_argument("--sweep", action="store_true", help="decode: add the batch sweep 1..256 to the line")
    ap.add_argument("--ctx", default="512,8192", help="decode: context lengths U[lo, hi] (lo,hi)")
    ap.add_argument("--attention-fold", type=int, default=0, choices=[0, 1, 2],
                    help="decode attention mapping: 0 default (one CTA per split), 1 fold splits in one CTA, 2 split")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--mode", default="decode",
                    choices=["decode", "prefill", "serve", "llm42", "ceiling", "cpu-baseline"])
    ap.add_argument("--ceiling-batches", default="1,256", help="ceiling mode: token counts")
    ap.add_argument("--ceiling-sweep", action="store_true", help="ceiling mode: also time every forced GEMM plan")
    ap.add_argument("--ceiling-gemms", default="", help="ceiling mode: only these GEMMs (comma-separated names)")
    ap.add_argument("--window", type=int, default=8, help="llm42 mode: verification window")
    ap.add_argument("--new-tokens", type=int, default=64, help="llm42 mode: tokens per request")
    ap.add_argument("--workload", default="c3", choices=["c3", "c4", "c5"], help="serve mode workload")
    ap.add_argument("--budget", type=int, default=2048, help="serve mode: chunked-prefill token budget")
    ap.add_argument("--sessions", type=int, default=128, help="serve c5: sessions")
    ap.add_argument("--turns", type=int, default=8, help="serve c5: turns per session")
    ap.add_argument("--concurrency", type=int, default=64, help="serve c5: sessions in flight")
    ap.add_argument("--seed", type=int, default=7, help="serve c5: turn-length seed")
    ap.add_argument("--tokens", type=int, default=8192, help="prefill mode: tokens per step")
    ap.add_argument("--prefill-requests", type=int, default=4)
    args = ap.parse_args()
    global CTX_LO, CTX_HI  # the decode workload's context range
    CTX_LO, CTX_HI = (int(v) for v in args.ctx.split(","))
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.mode == "prefill":
        run_prefill(args)
    elif args.mode == "serve":
        run_serve(args)
    elif args.mode == "llm42":
        run_llm42(args)
    elif args.mode == "ceiling":
        run_ceiling(args)
    elif args.mode == "cpu-baseline":
        run_cpu_baseline(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
