"""Host engine: continuous-batching scheduler and paged block manager.

Follows the engine structure and rules of 深入解析 Vosti §三 3.2 and §五:

* Paged KV pool; each request owns a page table mapping logical page i
  (tokens 16i..16i+15) to a physical page (Invariant 1: 0 <= cached <=
  |history|, page tables map the prefix to allocated, in-range slots).
* Exact prefix matching (§五 5.4): a rolling hash only *finds* candidate
  pages; a full page is reused only if its tokens, its depth in the prefix
  and its physical parent page all match.  A hash collision never causes
  reuse.
* Reuse before registration (§三 3.2): a step first resolves every prefix
  hit, then allocates and registers the private pages it will write.
  Shared and registered pages are never written again (Invariant 3, write
  isolation): the last prompt token always lands in a private page.
* Leaf-only eviction (§五 5.4): under memory pressure only registered,
  unreferenced pages without registered children are evicted, so a parent
  page id is never recycled while a retained child refers to it.
* Recompute: a request whose pages cannot be allocated is preempted; its
  private pages are freed and its history is recomputed later (prefix hits
  shorten the recomputation).
* Scheduling decisions (batch size, chunk budget, prefix reuse on/off,
  page placement, pool size) are free: they change when and where K/V is
  computed, never its value (Invariant 2, KV-value consistency), so the
  logits of a request depend on its history only (Theorem 4.1).

The engine calls an *executor* with a duck-typed interface:
``step(seqs, logit_rows) -> logits`` (seqs: list of (token_ids, cached_len,
page_table)) and ``sample(logits, samplers) -> tokens``.  ``GpuExecutor``
drives libvd.so.
"""

from __future__ import annotations

import collections
import dataclasses
import zlib

import numpy as np

PAGE = 16


def default_page_hash(parent_hash: int, tokens) -> int:
    """Rolling hash of a full page chained on its parent's hash (candidate lookup only)."""
    return zlib.crc32(np.asarray(tokens, dtype=np.int32).tobytes(), parent_hash & 0xFFFFFFFF)


@dataclasses.dataclass
class PageMeta:
    parent: int          # physical parent page (-1 for depth 0)
    depth: int           # logical page index in the prefix
    tokens: tuple        # the 16 tokens of the page
    hash: int
    children: int = 0    # registered children


class BlockManager:
    """Physical pages, reference counts, the prefix index and eviction."""

    def __init__(self, num_pages: int, placement_seed: int | None = None, prefix_reuse: bool = True,
                 page_hash=default_page_hash):
        self.num_pages = num_pages
        order = np.arange(num_pages)
        if placement_seed is not None:
            order = np.random.default_rng(placement_seed).permutation(num_pages)
        self.free = collections.deque(int(p) for p in order)
        self.ref = np.zeros(num_pages, dtype=np.int64)
        self.meta: dict[int, PageMeta] = {}          # registered pages
        self.index: dict[int, list] = collections.defaultdict(list)  # hash -> pages
        self.evictable: collections.OrderedDict = collections.OrderedDict()  # LRU of evictable leaves
        self.prefix_reuse = prefix_reuse
        self.page_hash = page_hash
        self.stats = collections.Counter()

    # -- invariants ------------------------------------------------------
    def check(self):
        """Invariant checks used by tests: no page is both free and referenced
        or registered, and every registered page's parent is registered."""
        free = set(self.free)
        for p in free:
            assert self.ref[p] == 0 and p not in self.meta
        for p, m in self.meta.items():
            assert m.parent == -1 or m.parent in self.meta, "parent recycled under a retained child"
            kids = sum(1 for q in self.meta.values() if q.parent == p)
            assert kids == m.children
        for p in self.evictable:
            assert self.ref[p] == 0 and self.meta[p].children == 0

    # -- lookup ------------------------------------------------------------
    def match_prefix(self, tokens, max_pages: int) -> list:
        """Longest chain of registered pages whose tokens, depth and parent
        match ``tokens`` exactly (at most ``max_pages`` pages)."""
        if not self.prefix_reuse:
            return []
        chain, parent, ph = [], -1, 0
        for i in range(max_pages):
            toks = tuple(int(t) for t in tokens[PAGE * i:PAGE * (i + 1)])
            h = self.page_hash(ph, toks)
            hit = -1
            for cand in self.index.get(h, ()):
                m = self.meta[cand]
                if m.tokens == toks and m.depth == i and m.parent == parent:
                    hit = cand
                    break
                self.stats["hash_candidates_rejected"] += 1
            if hit < 0:
                break
            chain.append(hit)
            parent, ph = hit, h
        return chain

    def acquire(self, pages):
        for p in pages:
            if self.ref[p] == 0:
                self.evictable.pop(p, None)
            self.ref[p] += 1

    def release(self, pages):
        for p in pages:
            self.ref[p] -= 1
            assert self.ref[p] >= 0
            if self.ref[p] == 0:
                if p in self.meta:
                    if self.meta[p].children == 0:
                        self.evictable[p] = True
                else:
                    self.free.append(p)

    # -- allocation ----------------------------------------------------------
    def _evict_one(self) -> bool:
        if not self.evictable:
            return False
        p, _ = self.evictable.popitem(last=False)  # least recently released leaf
        m = self.meta.pop(p)
        self.index[m.hash].remove(p)
        if not self.index[m.hash]:
            del self.index[m.hash]
        if m.parent >= 0:
            pm = self.meta[m.parent]
            pm.children -= 1
            if pm.children == 0 and self.ref[m.parent] == 0:
                self.evictable[m.parent] = True
        self.free.append(p)
        self.stats["evicted"] += 1
        return True

    def allocate(self, n: int):
        """n private pages, evicting unreferenced leaves if needed; None if impossible."""
        while len(self.free) < n:
            if not self._evict_one():
                return None
        out = [self.free.popleft() for _ in range(n)]
        for p in out:
            self.ref[p] = 1
        return out

    def register(self, page: int, parent: int, depth: int, tokens, parent_hash: int):
        """Offers a full, written page to the prefix index.

        ``parent`` is the registered page standing for the previous prefix
        page (-1 at depth 0).  Returns (hash, canonical page): ``page`` itself
        if it was registered, the identical page already registered if there
        is one (``page`` then stays private), or -1 when reuse is off.
        """
        toks = tuple(int(t) for t in tokens)
        h = self.page_hash(parent_hash, toks)
        if not self.prefix_reuse:
            return h, -1
        if page in self.meta:
            return h, page
        for cand in self.index.get(h, ()):
            m = self.meta[cand]
            if m.tokens == toks and m.depth == depth and m.parent == parent:
                return h, cand
        self.meta[page] = PageMeta(parent, depth, toks, h)
        self.index[h].append(page)
        if parent >= 0:
            self.meta[parent].children += 1
            self.evictable.pop(parent, None)
        self.stats["registered"] += 1
        return h, page


@dataclasses.dataclass
class Request:
    rid: int
    prompt: np.ndarray
    max_new: int
    seed: int
    temperature: float = 0.0
    history: list = dataclasses.field(default_factory=list)
    generated: int = 0
    cached: int = 0                  # tokens whose K/V is in this request's pages
    pages: list = dataclasses.field(default_factory=list)
    hashes: list = dataclasses.field(default_factory=list)  # chain hash per full page
    canon: list = dataclasses.field(default_factory=list)   # registered page standing for each full page
    registered_upto: int = 0         # full pages already offered to the index
    admitted: bool = False

    @property
    def done(self) -> bool:
        return self.generated >= self.max_new


class Engine:
    """Continuous batching with chunked prefill over a paged, prefix-sharing pool."""

    def __init__(self, executor, num_pages: int, max_batch: int = 8, token_budget: int = 64,
                 prefix_reuse: bool = True, placement_seed: int | None = None, page_hash=default_page_hash):
        self.ex = executor
        self.bm = BlockManager(num_pages, placement_seed, prefix_reuse, page_hash)
        self.max_batch = max_batch
        self.budget = token_budget
        self.waiting: collections.deque = collections.deque()
        self.running: list = []
        self.requests: dict = {}
        self.views: dict = collections.defaultdict(list)   # rid -> [(logits, token)]
        self.steps = 0
        self._next_id = 0

    def add_request(self, prompt, max_new: int, seed: int = 0, temperature: float = 0.0) -> int:
        rid = self._next_id
        self._next_id += 1
        r = Request(rid, np.asarray(prompt, dtype=np.int32), max_new, seed, temperature)
        r.history = [int(t) for t in r.prompt]
        self.requests[rid] = r
        self.waiting.append(r)
        return rid

    # -- scheduling ------------------------------------------------------------
    def _admit(self):
        while self.waiting and len(self.running) < self.max_batch:
            r = self.waiting.popleft()
            # Resolve prefix hits first; the last history token stays private.
            hits = self.bm.match_prefix(r.history, (len(r.history) - 1) // PAGE)
            self.bm.acquire(hits)
            r.pages = list(hits)
            r.cached = PAGE * len(hits)
            r.hashes, r.canon = [], list(hits)
            ph = 0
            for i in range(len(hits)):
                ph = self.bm.page_hash(ph, tuple(int(t) for t in r.history[PAGE * i:PAGE * (i + 1)]))
                r.hashes.append(ph)
            r.registered_upto = len(hits)
            r.admitted = True
            self.bm.stats["prefix_hit_pages"] += len(hits)
            self.running.append(r)

    def _preempt(self, r: Request):
        """Frees the request's pages; it is recomputed from its history later."""
        self.bm.release(r.pages)
        r.pages, r.hashes, r.canon, r.cached, r.registered_upto, r.admitted = [], [], [], 0, 0, False
        self.running.remove(r)
        self.waiting.appendleft(r)
        self.bm.stats["preempted"] += 1

    def _ensure_pages(self, r: Request, upto: int) -> bool:
        need = (upto + PAGE - 1) // PAGE - len(r.pages)
        if need <= 0:
            return True
        got = self.bm.allocate(need)
        if got is None:
            return False
        r.pages += got
        return True

    def plan(self):
        """Chooses (request, n_tokens) for this step under the token budget."""
        self._admit()
        plan, budget = [], self.budget
        # decode rows first, then prefill chunks, in admission order
        order = sorted(self.running, key=lambda r: (len(r.history) - r.cached > 1, r.rid))
        for r in order:
            todo = len(r.history) - r.cached
            if todo <= 0 or budget <= 0:
                continue
            n = min(todo, budget)
            if not self._ensure_pages(r, r.cached + n):
                continue
            plan.append((r, n))
            budget -= n
        if not plan and self.running:
            # nothing fits: preempt the newest request and retry once
            victim = max(self.running, key=lambda r: r.rid)
            self._preempt(victim)
            return self.plan() if self.running else []
        return plan

    def step(self) -> dict:
        """One engine step; returns the output record {rid: (logits, token)}."""
        plan = self.plan()
        if not plan:
            return {}
        seqs, rows, outs, t = [], [], [], 0
        for r, n in plan:
            seqs.append((np.asarray(r.history[r.cached:r.cached + n], dtype=np.int32), r.cached,
                         np.asarray(r.pages, dtype=np.int32)))
            t += n
            if r.cached + n == len(r.history):  # caught up: this row's logits choose the next token
                rows.append(t - 1)
                outs.append(r)
        logits = self.ex.step(seqs, rows)
        samplers = [(r.seed, r.generated, r.temperature) for r in outs]
        tokens = self.ex.sample(logits, samplers) if outs else []
        record = {}
        for (r, n) in plan:
            r.cached += n
            self._register_full_pages(r)
        for i, r in enumerate(outs):
            tok = int(tokens[i])
            record[r.rid] = (logits[i], tok)
            self.views[r.rid].append((logits[i], tok))
            r.history.append(tok)
            r.generated += 1
        for r in outs:
            if r.done:
                self.bm.release(r.pages)
                r.pages = []
                self.running.remove(r)
        self.steps += 1
        return record

    def _register_full_pages(self, r: Request):
        # Registration of pages written in this step happens after the step's
        # prefix hits were resolved (reuse before registration).
        full = r.cached // PAGE
        while r.registered_upto < full:
            i = r.registered_upto
            parent = r.canon[i - 1] if i > 0 else -1
            if i > 0 and parent < 0:
                break  # no registered chain to hang this page on
            ph = r.hashes[i - 1] if i > 0 else 0
            h, canon = self.bm.register(r.pages[i], parent, i, r.history[PAGE * i:PAGE * (i + 1)], ph)
            r.hashes.append(h)
            r.canon.append(canon)
            r.registered_upto += 1

    def run(self, max_steps: int = 100000):
        while (self.waiting or self.running) and self.steps < max_steps:
            self.step()
        return self.views


class GpuExecutor:
    """Executor over libvd.so: logits stay on the device; tokens come back to the host."""

    def __init__(self, model, pool, keep_logits: bool = True, stream=None):
        import torch
        self.torch = torch
        self.model, self.pool, self.keep, self.stream = model, pool, keep_logits, stream

    def step(self, seqs, rows):
        from . import vd
        torch = self.torch
        V = self.model.spec.vocab
        logits = torch.empty((max(len(rows), 1), V), dtype=torch.float32, device="cuda")
        self.model.step(self.pool, vd.StepBatch(seqs, logit_rows=rows), logits, self.stream)
        return logits[:len(rows)]

    def sample(self, logits, samplers):
        torch = self.torch
        out = torch.empty(len(samplers), dtype=torch.int32, device="cuda")
        self.model.sample(logits, samplers, out, self.stream)
        return out.cpu().numpy()
