// Host engine: continuous-batching scheduler and paged block manager.
//
// Rules (深入解析 Vosti §三 3.2 and §五):
//  * paged KV pool with per-request page tables (Invariant 1: 0 <= cached <=
//    |history|; tables map the prefix to allocated, in-range pages);
//  * exact prefix matching (§五 5.4): a rolling hash only finds candidate
//    pages; reuse needs the same 16 tokens, the same depth and the same
//    physical parent page, so a hash collision never causes reuse;
//  * reuse before registration (§三 3.2): prefix hits are resolved when a
//    request is admitted, before the step registers the pages it writes;
//    registered pages are read-only and the last history token always lands
//    in a private page (Invariant 3, write isolation);
//  * leaf-only eviction (§五 5.4): only registered, unreferenced pages with
//    no registered child are evicted, so a parent id is never recycled while
//    a retained child refers to it;
//  * preemption with recomputation when a step cannot get pages.
// Scheduling decisions never change a value: K/V is a function of the token
// prefix (Invariant 2), so a request's logits depend on its history only.
//
// The engine plans a step (vd_engine_plan), the caller executes it, and the
// engine commits the sampled tokens (vd_engine_commit); vd_engine_run_step
// does all three with libvd's kernels.
#include <cuda_runtime.h>
#include <string.h>

#include <algorithm>
#include <array>
#include <deque>
#include <list>
#include <memory>
#include <string>
#include <unordered_map>
#include <vector>

#include "vd_internal.h"

using vd::fail;

namespace {

constexpr int kPage = 16;

uint64_t page_hash(uint64_t parent_hash, const int32_t* toks, int mode) {
  if (mode == 1) return 7;  // every page collides (used to test exact matching)
  uint64_t h = 1469598103934665603ull ^ parent_hash;  // FNV-1a chained on the parent
  for (int i = 0; i < kPage; ++i) {
    uint32_t v = static_cast<uint32_t>(toks[i]);
    for (int b = 0; b < 4; ++b) {
      h ^= (v >> (8 * b)) & 0xFF;
      h *= 1099511628211ull;
    }
  }
  return h;
}

struct PageMeta {
  int parent;
  int depth;
  std::array<int32_t, kPage> tokens;
  uint64_t hash;
  int children = 0;
};

struct BlockManager {
  int num_pages = 0;
  bool reuse = true;
  int hash_mode = 0;
  std::deque<int> free_list;
  std::vector<int> ref;
  std::unordered_map<int, PageMeta> meta;
  std::unordered_map<uint64_t, std::vector<int>> index;
  std::list<int> lru;  // evictable leaves, oldest first
  int idle = 0;        // registered pages with no reference (all evictable, leaves first)
  std::unordered_map<int, std::list<int>::iterator> lru_pos;
  vd_engine_stats stats{};

  void lru_add(int p) {
    if (lru_pos.count(p)) return;
    lru.push_back(p);
    lru_pos[p] = std::prev(lru.end());
  }
  void lru_del(int p) {
    auto it = lru_pos.find(p);
    if (it == lru_pos.end()) return;
    lru.erase(it->second);
    lru_pos.erase(it);
  }
  bool same(const PageMeta& m, const int32_t* toks, int depth, int parent) const {
    return m.depth == depth && m.parent == parent && std::equal(m.tokens.begin(), m.tokens.end(), toks);
  }

  std::vector<int> match_prefix(const int32_t* tokens, int max_pages) {
    std::vector<int> chain;
    if (!reuse) return chain;
    int parent = -1;
    uint64_t ph = 0;
    for (int i = 0; i < max_pages; ++i) {
      const int32_t* toks = tokens + kPage * i;
      const uint64_t h = page_hash(ph, toks, hash_mode);
      int hit = -1;
      auto it = index.find(h);
      if (it != index.end()) {
        for (int cand : it->second) {
          if (same(meta.at(cand), toks, i, parent)) {
            hit = cand;
            break;
          }
          stats.hash_candidates_rejected++;
        }
      }
      if (hit < 0) break;
      chain.push_back(hit);
      parent = hit;
      ph = h;
    }
    return chain;
  }
  void acquire(const std::vector<int>& pages) {
    for (int p : pages) {
      if (ref[p] == 0) {
        lru_del(p);
        if (meta.count(p)) idle--;
      }
      ref[p]++;
    }
  }
  void release(const std::vector<int>& pages) {
    for (int p : pages) {
      ref[p]--;
      if (ref[p] == 0) {
        auto it = meta.find(p);
        if (it != meta.end()) {
          idle++;
          if (it->second.children == 0) lru_add(p);
        } else {
          free_list.push_back(p);
        }
      }
    }
  }
  // Pages obtainable without preempting anyone: free ones plus every
  // registered page nobody references.  A request references its whole
  // chain, so an unreferenced page's subtree is unreferenced too and leaf-
  // first eviction reaches all of them.
  int reclaimable() const { return static_cast<int>(free_list.size()) + idle; }
  bool evict_one() {
    if (lru.empty()) return false;
    const int p = lru.front();
    lru_del(p);
    const PageMeta m = meta.at(p);
    meta.erase(p);
    idle--;
    auto& v = index[m.hash];
    v.erase(std::find(v.begin(), v.end(), p));
    if (v.empty()) index.erase(m.hash);
    if (m.parent >= 0) {
      PageMeta& pm = meta.at(m.parent);
      if (--pm.children == 0 && ref[m.parent] == 0) lru_add(m.parent);
    }
    free_list.push_back(p);
    stats.evicted++;
    return true;
  }
  bool allocate(int n, std::vector<int>& out) {
    while (static_cast<int>(free_list.size()) < n)
      if (!evict_one()) return false;
    for (int i = 0; i < n; ++i) {
      const int p = free_list.front();
      free_list.pop_front();
      ref[p] = 1;
      out.push_back(p);
    }
    return true;
  }
  // Offers a full, written page; returns the page standing for this prefix
  // page in the index (itself, an identical registered page, or -1).
  int register_page(int page, int parent, int depth, const int32_t* toks, uint64_t ph, uint64_t* h_out) {
    const uint64_t h = page_hash(ph, toks, hash_mode);
    *h_out = h;
    if (!reuse) return -1;
    if (meta.count(page)) return page;
    auto it = index.find(h);
    if (it != index.end())
      for (int cand : it->second)
        if (same(meta.at(cand), toks, depth, parent)) return cand;
    PageMeta m;
    m.parent = parent;
    m.depth = depth;
    std::copy(toks, toks + kPage, m.tokens.begin());
    m.hash = h;
    meta.emplace(page, m);
    index[h].push_back(page);
    if (parent >= 0) {
      meta.at(parent).children++;
      lru_del(parent);
    }
    stats.registered++;
    return page;
  }
  int check() const {
    for (int p : free_list)
      if (ref[p] != 0 || meta.count(p)) return fail(VD_ERR_INVALID_ARG, "free page is referenced or registered");
    for (const auto& kv : meta) {
      if (kv.second.parent != -1 && !meta.count(kv.second.parent))
        return fail(VD_ERR_INVALID_ARG, "parent recycled under a retained child");
      int kids = 0;
      for (const auto& q : meta) kids += q.second.parent == kv.first;
      if (kids != kv.second.children) return fail(VD_ERR_INVALID_ARG, "child count mismatch");
    }
    for (int p : lru)
      if (ref[p] != 0 || meta.at(p).children != 0) return fail(VD_ERR_INVALID_ARG, "evictable page in use");
    int n_idle = 0;
    for (const auto& kv : meta) n_idle += ref[kv.first] == 0;
    if (n_idle != idle) return fail(VD_ERR_INVALID_ARG, "idle page count mismatch");
    return VD_OK;
  }
};

struct Request {
  int64_t rid;
  int prompt_len;
  std::vector<int32_t> history;
  int max_new;
  int generated = 0;
  int cached = 0;
  uint64_t seed;
  float temperature;
  std::vector<int> pages, canon;
  std::vector<uint64_t> hashes;
  int registered_upto = 0;
  bool done() const { return generated >= max_new; }
};

}  // namespace

struct vd_engine {
  vd_engine_config cfg{};
  BlockManager bm;
  std::deque<Request*> waiting;
  std::vector<Request*> running;
  std::unordered_map<int64_t, std::unique_ptr<Request>> reqs;
  int64_t next_id = 0;
  // current plan
  std::vector<std::pair<Request*, int>> plan;
  std::vector<Request*> outs;
  std::vector<int32_t> tok, pos, cu, cached, pt, rows;
  std::vector<int64_t> out_rids;
  std::vector<vd_sampler> samplers;
  int pt_stride = 0;
  bool planned = false;
  int32_t* h_tokens = nullptr;  // pinned, for run_step
  size_t h_tokens_cap = 0;
};

namespace {

// Admission (running < max_batch) takes the waiting queue in order while the
// pool can hold the next request's uncached prompt plus one page; with
// nothing running the front request is admitted unconditionally.
void admit(vd_engine* e) {
  while (!e->waiting.empty() && static_cast<int>(e->running.size()) < e->cfg.max_batch) {
    Request* r = e->waiting.front();
    const int hist_pages = (static_cast<int>(r->history.size()) + kPage - 1) / kPage;
    const int max_pages = (static_cast<int>(r->history.size()) - 1) / kPage;
    std::vector<int> hits = e->bm.match_prefix(r->history.data(), max_pages);
    if (!e->running.empty()) {
      int idle_hits = 0;  // hit pages now evictable: acquiring them removes them from the reclaimable set
      for (int p : hits) idle_hits += e->bm.ref[p] == 0;
      const int need = hist_pages - static_cast<int>(hits.size()) + 1;
      if (need > e->bm.reclaimable() - idle_hits) break;
    }
    e->waiting.pop_front();
    e->bm.acquire(hits);
    r->pages = hits;
    r->canon = hits;
    r->cached = kPage * static_cast<int>(hits.size());
    r->hashes.clear();
    uint64_t ph = 0;
    for (size_t i = 0; i < hits.size(); ++i) {
      ph = page_hash(ph, r->history.data() + kPage * i, e->bm.hash_mode);
      r->hashes.push_back(ph);
    }
    r->registered_upto = static_cast<int>(hits.size());
    e->bm.stats.prefix_hit_pages += static_cast<int64_t>(hits.size());
    e->running.push_back(r);
  }
}

void preempt(vd_engine* e, Request* r) {
  e->bm.release(r->pages);
  r->pages.clear();
  r->canon.clear();
  r->hashes.clear();
  r->cached = 0;
  r->registered_upto = 0;
  e->running.erase(std::find(e->running.begin(), e->running.end(), r));
  e->waiting.push_front(r);
  e->bm.stats.preempted++;
}

bool ensure_pages(vd_engine* e, Request* r, int upto) {
  const int need = (upto + kPage - 1) / kPage - static_cast<int>(r->pages.size());
  if (need <= 0) return true;
  return e->bm.allocate(need, r->pages);
}

// Plans one step.  Decode rows first, then prompt chunks in admission order,
// within the token budget; a request that cannot get its pages this step
// waits.  If nothing fits, the newest running request is preempted (its
// pages released, its K/V recomputed later) and nothing is admitted for the
// rest of this planning pass, so the victim cannot take its pages straight
// back; this repeats until something fits.  A request that cannot get its
// pages while running alone does not fit in the pool: VD_ERR_CAPACITY.
int make_plan(vd_engine* e) {
  bool allow_admit = true;
  for (;;) {
    if (allow_admit || e->running.empty()) admit(e);
    e->plan.clear();
    int budget = e->cfg.token_budget;
    std::vector<Request*> order(e->running);
    std::stable_sort(order.begin(), order.end(), [](const Request* a, const Request* b) {
      const bool pa = static_cast<int>(a->history.size()) - a->cached > 1;
      const bool pb = static_cast<int>(b->history.size()) - b->cached > 1;
      return pa != pb ? !pa : a->rid < b->rid;  // decode rows first, then admission order
    });
    for (Request* r : order) {
      const int todo = static_cast<int>(r->history.size()) - r->cached;
      if (todo <= 0 || budget <= 0) continue;
      const int n = std::min(todo, budget);
      if (!ensure_pages(e, r, r->cached + n)) continue;
      e->plan.push_back({r, n});
      budget -= n;
    }
    if (!e->plan.empty() || e->running.empty()) return VD_OK;
    if (e->running.size() == 1) return fail(VD_ERR_CAPACITY, "a request does not fit in the KV pool on its own");
    Request* victim = *std::max_element(e->running.begin(), e->running.end(),
                                        [](const Request* a, const Request* b) { return a->rid < b->rid; });
    preempt(e, victim);
    allow_admit = false;
  }
}

void register_full_pages(vd_engine* e, Request* r) {
  const int full = r->cached / kPage;
  while (r->registered_upto < full) {
    const int i = r->registered_upto;
    const int parent = i > 0 ? r->canon[i - 1] : -1;
    if (i > 0 && parent < 0) break;  // no registered chain to hang this page on
    const uint64_t ph = i > 0 ? r->hashes[i - 1] : 0;
    uint64_t h = 0;
    const int c = e->bm.register_page(r->pages[i], parent, i, r->history.data() + kPage * i, ph, &h);
    r->hashes.push_back(h);
    r->canon.push_back(c);
    r->registered_upto++;
  }
}

}  // namespace

extern "C" {

int vd_engine_create(const vd_engine_config* cfg, vd_engine** out) {
  if (!cfg || !out) return fail(VD_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  if (cfg->num_pages < 1 || cfg->max_batch < 1 || cfg->token_budget < 1)
    return fail(VD_ERR_INVALID_ARG, "num_pages, max_batch and token_budget must be >= 1");
  if (cfg->hash_mode != 0 && cfg->hash_mode != 1) return fail(VD_ERR_INVALID_ARG, "unknown hash_mode");
  vd_engine* e = new vd_engine();
  e->cfg = *cfg;
  BlockManager& bm = e->bm;
  bm.num_pages = cfg->num_pages;
  bm.reuse = cfg->prefix_reuse != 0;
  bm.hash_mode = cfg->hash_mode;
  bm.ref.assign(cfg->num_pages, 0);
  std::vector<int> order(cfg->num_pages);
  for (int i = 0; i < cfg->num_pages; ++i) order[i] = i;
  if (cfg->placement_seed >= 0) {  // seeded Fisher-Yates permutation (splitmix64 stream)
    uint64_t x = static_cast<uint64_t>(cfg->placement_seed);
    for (int i = cfg->num_pages - 1; i > 0; --i) {
      x += 0x9E3779B97F4A7C15ull;
      uint64_t z = x;
      z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
      z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
      z ^= z >> 31;
      std::swap(order[i], order[z % static_cast<uint64_t>(i + 1)]);
    }
  }
  bm.free_list.assign(order.begin(), order.end());
  *out = e;
  return VD_OK;
}

void vd_engine_destroy(vd_engine* e) {
  if (!e) return;
  if (e->h_tokens) cudaFreeHost(e->h_tokens);
  delete e;
}

int vd_engine_add_request(vd_engine* e, const int32_t* prompt, int32_t len, int32_t max_new, uint64_t seed,
                          float temperature, int64_t* rid_out) {
  if (!e || !prompt || !rid_out) return fail(VD_ERR_INVALID_ARG, "null argument");
  if (len < 1 || max_new < 1) return fail(VD_ERR_INVALID_ARG, "prompt length and max_new must be >= 1");
  auto r = std::make_unique<Request>();
  r->rid = e->next_id++;
  r->prompt_len = len;
  r->history.assign(prompt, prompt + len);
  r->max_new = max_new;
  r->seed = seed;
  r->temperature = temperature;
  e->waiting.push_back(r.get());
  *rid_out = r->rid;
  e->reqs.emplace(r->rid, std::move(r));
  return VD_OK;
}

int vd_engine_plan(vd_engine* e, vd_engine_plan_out* out) {
  if (!e || !out) return fail(VD_ERR_INVALID_ARG, "null argument");
  if (e->planned) return fail(VD_ERR_INVALID_ARG, "previous plan not committed");
  memset(out, 0, sizeof(*out));
  if (const int rc = make_plan(e)) return rc;
  if (e->plan.empty()) return VD_OK;
  e->tok.clear();
  e->pos.clear();
  e->cu.assign(1, 0);
  e->cached.clear();
  e->rows.clear();
  e->outs.clear();
  e->out_rids.clear();
  e->samplers.clear();
  e->pt_stride = 1;
  for (auto& pn : e->plan) e->pt_stride = std::max(e->pt_stride, static_cast<int>(pn.first->pages.size()));
  e->pt.assign(e->plan.size() * e->pt_stride, 0);
  int t = 0;
  for (size_t b = 0; b < e->plan.size(); ++b) {
    Request* r = e->plan[b].first;
    const int n = e->plan[b].second;
    for (int i = 0; i < n; ++i) {
      e->tok.push_back(r->history[r->cached + i]);
      e->pos.push_back(r->cached + i);
    }
    t += n;
    e->cu.push_back(t);
    e->cached.push_back(r->cached);
    std::copy(r->pages.begin(), r->pages.end(), e->pt.begin() + b * e->pt_stride);
    if (r->cached + n == static_cast<int>(r->history.size())) {  // caught up: this row chooses a token
      e->rows.push_back(t - 1);
      e->outs.push_back(r);
      e->out_rids.push_back(r->rid);
      e->samplers.push_back({r->seed, static_cast<uint64_t>(r->generated), r->temperature, 0.f});
    }
  }
  vd_batch& bt = out->batch;
  bt.num_tokens = t;
  bt.num_seqs = static_cast<int32_t>(e->plan.size());
  bt.num_logit_rows = static_cast<int32_t>(e->rows.size());
  bt.page_table_stride = e->pt_stride;
  bt.token_ids = e->tok.data();
  bt.positions = e->pos.data();
  bt.cu_q = e->cu.data();
  bt.cached_len = e->cached.data();
  bt.page_table = e->pt.data();
  bt.logit_rows = e->rows.data();
  out->rids = e->out_rids.data();
  out->samplers = e->samplers.data();
  e->planned = true;
  return VD_OK;
}

int vd_engine_commit(vd_engine* e, const int32_t* tokens) {
  if (!e) return fail(VD_ERR_INVALID_ARG, "null engine");
  if (!e->planned) return fail(VD_ERR_INVALID_ARG, "nothing planned");
  if (!e->outs.empty() && !tokens) return fail(VD_ERR_INVALID_ARG, "null tokens");
  for (auto& pn : e->plan) {
    pn.first->cached += pn.second;
    register_full_pages(e, pn.first);
  }
  for (size_t i = 0; i < e->outs.size(); ++i) {
    e->outs[i]->history.push_back(tokens[i]);
    e->outs[i]->generated++;
  }
  for (Request* r : e->outs)
    if (r->done()) {
      e->bm.release(r->pages);
      r->pages.clear();
      e->running.erase(std::find(e->running.begin(), e->running.end(), r));
    }
  e->bm.stats.steps++;
  e->planned = false;
  e->plan.clear();
  return VD_OK;
}

int vd_engine_run_step(vd_engine* e, vd_model* m, vd_kv_pool* pool, float* logits, int32_t* tokens_dev,
                       int64_t* rids_out, int32_t* tokens_out, int32_t* n_out, void* stream) {
  if (!e || !m || !pool || !logits || !tokens_dev || !n_out) return fail(VD_ERR_INVALID_ARG, "null argument");
  *n_out = 0;
  vd_engine_plan_out p;
  int rc = vd_engine_plan(e, &p);
  if (rc) return rc;
  if (p.batch.num_tokens == 0) return VD_OK;
  const int R = p.batch.num_logit_rows;
  if ((rc = vd_step_sample(m, pool, &p.batch, p.samplers, logits, tokens_dev, stream))) return rc;
  if (R > 0) {
    if (e->h_tokens_cap < static_cast<size_t>(R)) {
      if (e->h_tokens) cudaFreeHost(e->h_tokens);
      e->h_tokens = nullptr;
      if (cudaMallocHost(reinterpret_cast<void**>(&e->h_tokens), R * sizeof(int32_t)) != cudaSuccess)
        return fail(VD_ERR_CUDA, "pinned token buffer");
      e->h_tokens_cap = R;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    VD_CUDA_TRY(cudaMemcpyAsync(e->h_tokens, tokens_dev, R * sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    VD_CUDA_TRY(cudaStreamSynchronize(s));
    if (rids_out) memcpy(rids_out, p.rids, R * sizeof(int64_t));
    if (tokens_out) memcpy(tokens_out, e->h_tokens, R * sizeof(int32_t));
  }
  *n_out = R;
  return vd_engine_commit(e, e->h_tokens);
}

int vd_engine_pending(vd_engine* e) {
  if (!e) return 0;
  return static_cast<int>(e->waiting.size() + e->running.size());
}

int vd_engine_get_stats(vd_engine* e, vd_engine_stats* out) {
  if (!e || !out) return fail(VD_ERR_INVALID_ARG, "null argument");
  *out = e->bm.stats;
  return VD_OK;
}

int vd_engine_check(vd_engine* e) {
  if (!e) return fail(VD_ERR_INVALID_ARG, "null engine");
  return e->bm.check();
}

int vd_engine_page_info(vd_engine* e, int32_t page, int32_t* ref, int32_t* registered) {
  if (!e || !ref || !registered) return fail(VD_ERR_INVALID_ARG, "null argument");
  if (page < 0 || page >= e->bm.num_pages) return fail(VD_ERR_OUT_OF_RANGE, "page out of range");
  *ref = e->bm.ref[page];
  *registered = e->bm.meta.count(page) ? 1 : 0;
  return VD_OK;
}

int vd_engine_history(vd_engine* e, int64_t rid, int32_t* out, int32_t cap, int32_t* len, int32_t* prompt_len) {
  if (!e || !len) return fail(VD_ERR_INVALID_ARG, "null argument");
  auto it = e->reqs.find(rid);
  if (it == e->reqs.end()) return fail(VD_ERR_OUT_OF_RANGE, "unknown request id");
  const Request& r = *it->second;
  *len = static_cast<int32_t>(r.history.size());
  if (prompt_len) *prompt_len = r.prompt_len;
  if (out) memcpy(out, r.history.data(), std::min<size_t>(cap, r.history.size()) * sizeof(int32_t));
  return VD_OK;
}

}  // extern "C"
