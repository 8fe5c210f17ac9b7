"""Engine executor that emulates the paged KV pool on the CPU with the oracle.

K/V live in a numpy pool indexed by (layer, physical page, slot); every step
reads the request's cached prefix through its page table and writes the new
tokens' K/V into their slots, so any bookkeeping error of the block manager
(a wrong page reused, a shared page overwritten) changes the logits or trips
the write guard.  Test infrastructure only.
"""

import numpy as np

from oracle import sampler as osm
from oracle.decoder import OracleDecoder


class OracleExecutor:
    def __init__(self, spec, weights_u16, num_pages, write_guard=None):
        self.spec = spec
        self.dec = OracleDecoder(spec, weights_u16)
        L, Hkv, hd = spec.n_layers, spec.n_kv_heads, spec.head_dim
        self.K = np.zeros((L, num_pages, 16, Hkv, hd))
        self.V = np.zeros_like(self.K)
        self.written = np.zeros((num_pages, 16), dtype=bool)
        self.guard = write_guard
        self.steps = []

    def step(self, seqs, rows):
        self.steps.append([(len(t), c) for t, c, _ in seqs])
        out = []
        for toks, cached, pt in seqs:
            pos = np.arange(cached)
            pages, slots = pt[pos // 16], pos % 16
            assert np.all(self.written[pages, slots]), "reading a slot that was never written"
            cache = [(self.K[l][pages, slots], self.V[l][pages, slots]) for l in range(self.spec.n_layers)]
            lg, new = self.dec.step(toks, cache, logit_rows=range(len(toks)))
            for i in range(len(toks)):
                p = cached + i
                pg, sl = pt[p // 16], p % 16
                if self.guard is not None:
                    assert self.guard(int(pg)), f"write into shared/registered page {pg}"
                for l in range(self.spec.n_layers):
                    self.K[l, pg, sl] = new[l][0][p]
                    self.V[l, pg, sl] = new[l][1][p]
                self.written[pg, sl] = True
            out.append(lg)
        allrows = np.concatenate(out) if out else np.zeros((0, self.spec.vocab))
        return allrows[list(rows)]

    def sample(self, logits, samplers):
        return np.array([osm.sample(l, t, s, k) for l, (s, k, t) in zip(logits, samplers)], dtype=np.int32)
