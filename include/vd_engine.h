/*
 * vd_engine.h -- host engine of libvd.so: continuous batching with chunked
 * prefill over the paged, prefix-sharing KV pool.
 *
 * Rules followed (深入解析 Vosti §三 3.2, §五 5.4): exact prefix matching (a
 * rolling hash only finds candidates; reuse needs equal tokens, depth and
 * physical parent page), prefix hits resolved before the pages a step writes
 * are registered, registered pages read-only, leaf-only eviction under memory
 * pressure, preemption with recomputation.  Scheduling choices (batch size,
 * token budget, reuse on/off, page placement, pool size) never change a
 * value: the logits of a request depend on its token history only
 * (深入解析 Vosti §二 Theorem 4.1).
 *
 * Use: vd_engine_add_request() any number of times, then repeat either
 * vd_engine_run_step() (plan, vd_step_sample, copy tokens back, commit),
 * or vd_engine_plan() / execute the returned vd_batch yourself /
 * vd_engine_commit(tokens), until vd_engine_pending() is 0.  Host-only except
 * vd_engine_run_step.  An engine is not thread-safe.  Errors as in vd.h.
 */
#ifndef VD_ENGINE_H_
#define VD_ENGINE_H_

#include <stdint.h>

#include "vd.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct vd_engine vd_engine;

typedef struct vd_engine_config {
  int32_t num_pages;       /* pool pages the engine may hand out: ids 0 .. num_pages-1 */
  int32_t max_batch;       /* requests running at once                                 */
  int32_t token_budget;    /* tokens per step (decode rows first, then prefill chunks) */
  int32_t prefix_reuse;    /* 1: share registered full pages between requests          */
  int64_t placement_seed;  /* < 0: pages handed out in id order; else a seeded shuffle */
  int32_t hash_mode;       /* 0: rolling hash; 1: every page hashes alike (tests)      */
  int32_t pad_;
} vd_engine_config;

typedef struct vd_engine_stats {
  int64_t steps;
  int64_t prefix_hit_pages;
  int64_t registered;
  int64_t evicted;
  int64_t preempted;
  int64_t hash_candidates_rejected;
} vd_engine_stats;

/* A planned step: a vd_batch over engine-owned host arrays (valid until the
 * next plan or commit), and for each logit row its request id and sampler. */
typedef struct vd_engine_plan_out {
  vd_batch batch;
  const int64_t* rids;
  const vd_sampler* samplers;
} vd_engine_plan_out;

int vd_engine_create(const vd_engine_config* cfg, vd_engine** out);
void vd_engine_destroy(vd_engine* e);
/* Queues a request; prompt (host) is copied.  sampler state = (seed, output index). */
int vd_engine_add_request(vd_engine* e, const int32_t* prompt, int32_t len, int32_t max_new, uint64_t seed,
                          float temperature, int64_t* rid_out);
/* Plans the next step.  batch.num_tokens == 0: nothing to do. */
int vd_engine_plan(vd_engine* e, vd_engine_plan_out* out);
/* Commits the planned step: tokens (host [num_logit_rows]) are appended to the
 * requests of the logit rows; finished requests release their pages. */
int vd_engine_commit(vd_engine* e, const int32_t* tokens);
/* Plan + vd_step_sample + token copy to the host + commit.  logits: dev
 * fp32 [>= rows][V]; tokens_dev: dev int32 [>= rows]; rids_out / tokens_out:
 * host arrays [>= rows] or null; *n_out = rows emitted.  Synchronises the stream. */
int vd_engine_run_step(vd_engine* e, vd_model* m, vd_kv_pool* pool, float* logits, int32_t* tokens_dev,
                       int64_t* rids_out, int32_t* tokens_out, int32_t* n_out, void* stream);
/* Requests waiting or running. */
int vd_engine_pending(vd_engine* e);
int vd_engine_get_stats(vd_engine* e, vd_engine_stats* out);
/* Checks the block manager's invariants; VD_ERR_INVALID_ARG with a message if one fails. */
int vd_engine_check(vd_engine* e);
/* Page state for tests: *ref = holders of the page, *registered = 1 if it is
 * in the prefix index (and therefore must never be written again). */
int vd_engine_page_info(vd_engine* e, int32_t page, int32_t* ref, int32_t* registered);
/* History (prompt + generated tokens) of a request into out[cap]; *len = its length. */
int vd_engine_history(vd_engine* e, int64_t rid, int32_t* out, int32_t cap, int32_t* len, int32_t* prompt_len);

#ifdef __cplusplus
}
#endif
#endif /* VD_ENGINE_H_ */
