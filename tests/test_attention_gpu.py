"""Unified paged attention: parity with the oracle and the causal contract.

K/V are seeded synthetic values written straight into caller-owned pool
memory ([layer][page][K/V][kv_head][16][hd]); q rows are seeded per
(request, position), so the same logical row can be recomputed under any
batch composition, chunking, page placement or split placement.
"""

import numpy as np
import pytest
import torch

from gpu_util import bits, f64, ready
from invariant_vd_step_gb300 import synth, vd
from oracle import decoder as od

pytestmark = pytest.mark.gpu

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

    def run(self, parts, layer=0):
        """parts: list of (request, cached, q_len). Returns {(r, pos): out row bits/values}."""
        seqs, keys, qs = [], [], []
        for r, c, ql in parts:
            seqs.append((np.zeros(ql, np.int32), c, self.tables[r]))
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


def _check_parity(sc, res, window=0):
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


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_decode_and_prefill_rows_vs_oracle(hd):
    ready()
    lens = [1, 17, 64, 65, 511, 512, 513, 1100]
    sc = Scenario(SPECS[hd], lens, num_pages=200, seed=hd)
    # decode rows (last position), a full prefill of one request, and a chunk
    res = sc.run([(r, n - 1, 1) for r, n in enumerate(lens)])
    _check_parity(sc, res)
    res = sc.run([(6, 0, 513), (7, 1000, 100), (2, 3, 61)])
    _check_parity(sc, res)


def test_sliding_window_vs_oracle():
    ready()
    spec = SPECS[128].with_(sliding_window=100, local_global_period=1000)
    lens = [50, 99, 100, 101, 700]
    sc = Scenario(spec, lens, num_pages=120, seed=3)
    res = sc.run([(r, n - 1, 1) for r, n in enumerate(lens)])
    _check_parity(sc, res, window=100)
    res = sc.run([(4, 0, 700)])
    _check_parity(sc, res, window=100)


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_causal_contract_bitwise_across_schedules(hd):
    # The same (request, position) row must be bit-identical whatever the
    # query length, row index, batch, chunking and split placement.
    ready()
    lens = [300, 1030, 77]
    sc = Scenario(SPECS[hd], lens, num_pages=120, seed=11 + hd)
    runs = [
        [(0, 0, 300), (1, 0, 1030), (2, 0, 77)],                  # one prefill each
        [(1, 0, 500), (0, 0, 150), (2, 0, 10)],                   # chunks ...
        [(1, 500, 530), (0, 150, 150), (2, 10, 67)],              # ... continued
        [(2, 76, 1), (0, 299, 1), (1, 1029, 1)],                  # decode rows
        [(0, 299, 1)], [(1, 511, 1)], [(1, 512, 1)],              # alone, at split edges
        [(1, 1000, 30), (0, 290, 10)],
        [(0, 63, 2), (1, 63, 2)],
    ]
    seen = {}
    for parts in runs:
        for key, row in sc.run(parts).items():
            b = bits(row)
            if key in seen:
                np.testing.assert_array_equal(b, seen[key], err_msg=f"row {key} differs in {parts}")
            else:
                seen[key] = b
    assert len(seen) > 1400


def test_page_placement_does_not_change_bits():
    ready()
    lens = [333, 700]
    sc = Scenario(SPECS[128], lens, num_pages=80, seed=5)
    a = sc.run([(0, 0, 333), (1, 650, 50)])
    sc.place(np.arange(80)[::-1].copy())  # a different physical layout of the same logical K/V
    b = sc.run([(0, 0, 333), (1, 650, 50)])
    for k in a:
        np.testing.assert_array_equal(bits(a[k]), bits(b[k]))
