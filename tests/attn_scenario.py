"""Paged-attention test scenarios: seeded K/V written straight into
caller-owned pool memory ([layer][page][K/V][kv_head][16][hd]) and q rows
seeded per (request, position), so the same logical row can be recomputed
under any batch composition, chunking, page placement or split placement."""

import numpy as np
import torch

from gpu_util import f64
from invariant_vd_step_gb300 import synth, vd
from oracle import decoder as od

SPECS = {
    64: synth.TINY,
    128: synth.ModelSpec("att128", 1, 256, 8, 2, 128, 256, 256),
    256: synth.ModelSpec("att256", 1, 256, 4, 2, 256, 256, 256),
}


class Scenario:
    def __init__(self, spec, kv_lens, num_pages, seed=0, max_tokens=2048):
        self.spec = spec
        self.kv_lens = list(kv_lens)
        W = {k: v.cuda() for k, v in synth.make_weights(spec, seed=seed).items()}
        self.model = vd.Model(spec, W, max_tokens=max_tokens, max_seqs=64, max_logit_rows=8,
                              max_context=max(kv_lens) + 16)
        self.num_pages = num_pages
        mem = torch.zeros(self.model.pool_bytes(num_pages), dtype=torch.uint8, device="cuda")
        self.pool = vd.KVPool(self.model, num_pages, memory=mem)
        Hq, Hkv, hd = spec.n_heads, spec.n_kv_heads, spec.head_dim
        self.K, self.V, self.Q = [], [], []
        for r, n in enumerate(kv_lens):
            self.K.append(synth.make_normal_bf16((n, Hkv, hd), seed=1000 * seed + 3 * r))
            self.V.append(synth.make_normal_bf16((n, Hkv, hd), seed=1000 * seed + 3 * r + 1))
            self.Q.append(synth.make_normal_bf16((n, Hq, hd), seed=1000 * seed + 3 * r + 2))
        self.place(synth.page_permutation(num_pages, seed=seed + 7))

    def place(self, perm):
        """Assign physical pages from the permutation and write K/V there."""
        view = self.pool.view()
        view.zero_()
        self.tables, k = [], 0
        for r, n in enumerate(self.kv_lens):
            npg = (n + 15) // 16
            pt = np.asarray(perm[k:k + npg], dtype=np.int32)
            k += npg
            self.tables.append(pt)
            for i in range(npg):
                m = min(16, n - 16 * i)
                for layer in range(self.spec.n_layers):
                    view[layer, pt[i], 0, :, :m] = self.K[r][16 * i:16 * i + m].transpose(0, 1).cuda()
                    view[layer, pt[i], 1, :, :m] = self.V[r][16 * i:16 * i + m].transpose(0, 1).cuda()
        assert k <= self.num_pages

    def run(self, parts, layer=0, tables=None):
        """parts: list of (request, cached, q_len); tables: optional {request: page table} overriding the
        placed ones (e.g. padded with trailing entries).  Returns {(r, pos): out row bits/values}."""
        seqs, keys, qs = [], [], []
        for r, c, ql in parts:
            pt = tables[r] if tables is not None and r in tables else self.tables[r]
            seqs.append((np.zeros(ql, np.int32), c, pt))
            keys += [(r, c + i) for i in range(ql)]
            qs.append(self.Q[r][c:c + ql])
        q = torch.cat(qs).cuda().contiguous()
        out = torch.full_like(q, float("nan"))
        self.model.attention(self.pool, layer, vd.StepBatch(seqs), q, out)
        torch.cuda.synchronize()
        return {k: out[i] for i, k in enumerate(keys)}

    def oracle(self, r, positions, window):
        K, V, Q = f64(self.K[r]), f64(self.V[r]), f64(self.Q[r])
        return od.attention(Q[positions], K, V, positions, window)


def check_parity(sc, res, window=0):
    by_req = {}
    for (r, p), row in res.items():
        by_req.setdefault(r, []).append((p, row))
    for r, rows in by_req.items():
        rows.sort(key=lambda x: x[0])
        pos = [p for p, _ in rows]
        ref = sc.oracle(r, pos, window)
        got = np.stack([f64(x) for _, x in rows])
        vmax = np.abs(f64(sc.V[r])).max()
        # P is rounded to bf16 (<= 2^-9 relative per weight) and both sides round the output once
        tol = 2.0 ** -8 * vmax + 2.0 ** -7 * np.abs(ref)
        assert np.all(np.abs(got - ref) <= tol), f"req {r}: max |d| {np.abs(got - ref).max():.3g}"
