/*
 * vd.h -- C ABI of the batch-invariant decoder step (libvd.so).
 *
 * One engine step runs a Llama/Gemma-style decoder over a batch of
 * requests whose K/V lives in a paged, prefix-sharing cache, and returns
 * float32 logits for selected rows.  Every kernel choice (GEMM tile, KV
 * split size, key tile) is fixed when the model is created, from the model
 * shape alone, so that for every request u the logits equal
 * Forward(W, history_u) bit for bit whatever the batch composition, chunked
 * prefill budget, prefill/decode split, prefix reuse, recomputation or
 * physical page placement.
 *
 * Sources (cited by page title and section):
 *   [V]  "Vosti: Specifying, Implementing, and Verifying Deterministic LLM
 *        Inference" (arXiv 2609.38981), abstract.
 *   [B]  深入解析 Vosti (blog deep-dive on the same paper): §二 Definition 2.1
 *        and Theorem 4.1; §三 3.2 engine invariants and the three engineering
 *        rules (fixed kernel choices, exact prefix matching, reuse before
 *        registration); §五 5.1 KV-value invariant; §六 6.1 matmul contract,
 *        6.2 attention causal contract, masking rules and tile traversal.
 *   [T]  "Deterministic and bit-exact inference" (catalogue record M-0002),
 *        technical section: fixed KV split *size*, batch-invariant RMSNorm,
 *        matmul and attention.
 *   [L]  "LLM-42: Enabling Determinism in LLM Inference with Verified
 *        Speculation" (arXiv 2601.17768), §4 decode-verify-rollback.
 *
 * Conventions for every entry point:
 *   - Return value: VD_OK (0) or a VD_ERR_* code; vd_last_error() then gives
 *     a message (thread-local, valid until the next call on this thread).
 *   - Arguments are validated on the host before anything is launched; a
 *     call that fails validation has launched nothing and changed nothing.
 *   - "dev" pointers are CUDA device pointers of the current device; "host"
 *     pointers are ordinary host memory (pageable or pinned) read during the
 *     call and not retained.
 *   - bf16 tensors are row-major; matrices are stored [out][in].
 *   - Work is enqueued on the given stream (0 = legacy default stream); the
 *     call returns before the GPU finishes unless stated otherwise.
 */
#ifndef VD_H_
#define VD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  VD_OK = 0,
  VD_ERR_INVALID_ARG = 1,  /* malformed descriptor, null pointer, bad size      */
  VD_ERR_UNSUPPORTED = 2,  /* no fixed kernel configuration for this shape      */
  VD_ERR_OUT_OF_RANGE = 3, /* page id, position, token id or row out of range   */
  VD_ERR_CAPACITY = 4,     /* step exceeds the sizes fixed at model creation    */
  VD_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed                 */
  VD_ERR_TIMEOUT = 6       /* a bounded on-device wait gave up (device status)  */
};

enum { VD_ACT_SWIGLU = 0, VD_ACT_GEGLU = 1 };

typedef struct vd_model vd_model;
typedef struct vd_kv_pool vd_kv_pool;

/* Model shape and numerics.  Layer i is a global attention layer iff
 * local_global_period == 0 or (i + 1) % local_global_period == 0; other
 * layers are local with a window of sliding_window keys (the row's own key
 * included) [B §六 6.2, sliding-window traversal]. */
typedef struct vd_model_config {
  int32_t n_layers;
  int32_t d_model;
  int32_t n_heads;           /* query heads Hq                                */
  int32_t n_kv_heads;        /* KV heads Hkv; Hq % Hkv == 0                   */
  int32_t head_dim;          /* 64, 128 or 256                                */
  int32_t ffn_dim;           /* F                                             */
  int32_t vocab;             /* V                                             */
  float rms_eps;
  int32_t act;               /* VD_ACT_SWIGLU or VD_ACT_GEGLU (tanh GELU)     */
  int32_t qk_norm;           /* 1: per-head RMSNorm of q and k before RoPE    */
  float rope_theta;          /* global layers                                 */
  float rope_theta_local;    /* local layers                                  */
  int32_t sliding_window;    /* 0: no local layers                            */
  int32_t local_global_period;
  int32_t page_size;         /* must be 16                                    */
  /* capacities: fix workspace sizes at creation, never numerics */
  int32_t max_tokens;        /* max tokens (rows) per step                    */
  int32_t max_seqs;          /* max requests per step                         */
  int32_t max_logit_rows;    /* max rows returning logits per step            */
  int32_t max_context;       /* max cached + new tokens of one request        */
  /* Gemma-3 block (the published Gemma 3 architecture; the pages name the
   * model, not its block): */
  int32_t embed_scale;       /* 1: embeddings times bf16(sqrt(d_model))       */
  int32_t norm_offset;       /* 1: every RMSNorm gain is (1 + w), fp32        */
  int32_t sandwich_norm;     /* 1: x = x + rms_post(sub-layer output), both
                                sub-layers (post_attn_norm, post_ffn_norm)    */
} vd_model_config;

/* Per-layer weights: bf16 device pointers, borrowed (caller keeps them
 * alive and unchanged until vd_destroy_model). */
typedef struct vd_layer_weights {
  const void* attn_norm;   /* [d]                                             */
  const void* wqkv;        /* [(Hq + 2 Hkv) hd][d]; rows q heads, k, v        */
  const void* q_norm;      /* [hd] (only if qk_norm)                          */
  const void* k_norm;      /* [hd] (only if qk_norm)                          */
  const void* wo;          /* [d][Hq hd]                                      */
  const void* ffn_norm;    /* [d]                                             */
  const void* w_gate_up;   /* [2F][d]; rows 0..F-1 gate, F..2F-1 up           */
  const void* w_down;      /* [d][F]                                          */
  const void* post_attn_norm; /* [d] (only if sandwich_norm)                  */
  const void* post_ffn_norm;  /* [d] (only if sandwich_norm)                  */
} vd_layer_weights;

typedef struct vd_weight_ptrs {
  const void* embed;                /* dev bf16 [V][d]                          */
  const vd_layer_weights* layers;   /* host array [n_layers], copied            */
  const void* final_norm;           /* dev bf16 [d]                             */
  const void* lm_head;              /* dev bf16 [V][d]                          */
} vd_weight_ptrs;

/* One engine step.  Request b owns tokens cu_q[b] .. cu_q[b+1]-1 (q_len >= 1),
 * at positions cached_len[b] .. cached_len[b] + q_len - 1; its logical page i
 * (tokens 16i .. 16i+15) is physical page page_table[b * page_table_stride + i].
 * The step writes the K/V of its new tokens into their slots and reads the
 * cached prefix [0, cached_len[b]) from the pool [B §三 3.2 Invariant 1;
 * §五 5.1].  All arrays are host memory. */
typedef struct vd_batch {
  int32_t num_tokens;          /* T = cu_q[B]                                 */
  int32_t num_seqs;            /* B                                           */
  int32_t num_logit_rows;      /* R                                           */
  int32_t page_table_stride;   /* columns of page_table                       */
  const int32_t* token_ids;    /* [T]                                         */
  const int32_t* positions;    /* [T]; must equal cached_len[b] + i           */
  const int32_t* cu_q;         /* [B + 1], cu_q[0] = 0, strictly increasing   */
  const int32_t* cached_len;   /* [B]                                         */
  const int32_t* page_table;   /* [B * page_table_stride]                     */
  const int32_t* logit_rows;   /* [R] token indices in [0, T)                 */
} vd_batch;

/* Per-row sampler state [B §二 Definition 2.1, sampler_0]: Philox4x32-10 key
 * = seed, counter from (vocabulary index, step).  temperature <= 0: greedy. */
typedef struct vd_sampler {
  uint64_t seed;
  uint64_t step;
  float temperature;
  float pad_;
} vd_sampler;

typedef struct vd_kernel_stat {
  char name[32];
  int32_t launches;   /* timed regions (event pairs) of this class     */
  int32_t kernels;    /* kernel launches inside those regions          */
  double total_ms;
} vd_kernel_stat;

/* Creates a model over borrowed weights and fixes every kernel choice from
 * the shape alone [B §三 3.2, fixed kernel choices: bound at initialisation
 * from weight dims, dtype, head geometry and page size; no runtime tuning;
 * a shape without a fixed configuration is rejected].  Allocates the
 * library-owned workspace (activations, split partials, RoPE tables) on the
 * current device.  Errors: VD_ERR_INVALID_ARG (null/inconsistent),
 * VD_ERR_UNSUPPORTED (head_dim not 64/128/256, page_size != 16, d or 2F
 * or V not a multiple of 128, ...), VD_ERR_CUDA. */
int vd_create_model(const vd_model_config* cfg, const vd_weight_ptrs* w, vd_model** out);
void vd_destroy_model(vd_model* m);

/* Paged KV pool of num_pages pages [B §三 3.2: paged KV with page tables;
 * §五 5.1: each slot holds fKV of its logical prefix].  Layout, per layer:
 * [page][K=0,V=1][kv_head][16 slots][head_dim] bf16, layers contiguous, so
 * one page of one layer is 2*Hkv*16*hd*2 bytes.  dev_mem (nullable): caller
 * memory of at least vd_kv_pool_bytes() bytes, 256-byte aligned, borrowed;
 * null makes the library allocate.  The pool is zero-filled on creation.
 * Errors: VD_ERR_INVALID_ARG, VD_ERR_CAPACITY (bytes too small), VD_ERR_CUDA. */
size_t vd_kv_pool_bytes(const vd_model* m, int32_t num_pages);
int vd_kv_pool_alloc(vd_model* m, int32_t num_pages, void* dev_mem, size_t bytes, vd_kv_pool** out);
void vd_destroy_kv_pool(vd_kv_pool* p);
/* Device address of the pool (for tests that fill it directly). */
void* vd_kv_pool_data(vd_kv_pool* p);

/* One engine step [B §二 Theorem 4.1: o_u.logits = Forward(W, history_u)].
 * logits_out: dev float32 [R][V], row j = logits of token logit_rows[j].
 * Validates the descriptor (S5 layout consistency: positions, page ids in
 * range, capacity; S7 write isolation: no two new tokens share a slot),
 * uploads it, then enqueues the whole decoder forward.  Errors:
 * VD_ERR_INVALID_ARG, VD_ERR_OUT_OF_RANGE, VD_ERR_CAPACITY, VD_ERR_CUDA.
 * T == 0 is a no-op. */
int vd_step(vd_model* m, vd_kv_pool* pool, const vd_batch* b, float* logits_out, void* stream);

/* Reduction mode (the fast path of LLM-42's decode-verify-rollback [L, design:
 * a non-invariant fast path verified by fixed-shape replay]).  mode 0
 * (default): every step is batch-invariant.  mode 1: GEMMs with fewer weight
 * tiles than SMs split K across CTAs (fp32 partials summed in split order,
 * then the same epilogue) when a step has at most 256 tokens; logits then
 * depend on the batch and are not guaranteed to equal the invariant path's.
 * Use mode 1 only for candidates that an invariant step verifies.  Switching
 * is cheap (the partial buffer is allocated on first use).
 * Errors: VD_ERR_INVALID_ARG, VD_ERR_CUDA. */
int vd_set_reduction_mode(vd_model* m, int32_t mode);

/* Workload-dependent decode attention mapping [B §八 8.1: one SM per
 * sequence for full waves, several SMs for partially filled waves, both with
 * the same accumulation order; named there as future work that needs a
 * cross-kernel bitwise check].  Decode-class rows
 * (q_len * Hq/Hkv <= 16) normally get one CTA per (request, KV head, split)
 * and a merge kernel folds the split partials.  In fold mode one CTA per
 * (request, KV head) walks all its splits and folds them itself, with the
 * merge kernel's arithmetic and order, writing the output directly: no
 * partials round trip and no merge launch for those rows.  Logits are bitwise
 * identical in both modes.  mode 0 (default) and 2: split mode; 1: fold
 * mode.  On GB300 fold mode measured slower or equal (a fold CTA walks its
 * splits serially, so a long request sets the launch's critical path, and
 * the merged state costs registers), so the default does not use it.
 * Head dimensions above 128 never fold.  Errors: VD_ERR_INVALID_ARG. */
int vd_set_attention_fold(vd_model* m, int32_t mode);

/* Kernel of the prefill-class attention rows (q_len * Hq/Hkv > 16), with the
 * per-row traversal and arithmetic of 深入解析 Vosti §六 6.2 either way.
 * kernel 0 (default): 5th-generation tensor cores (tcgen05, accumulators in
 * tensor memory, 128 rows per CTA) for head dimensions 64, 128 and 256;
 * kernel 1: mma.sync (64 rows per CTA) for every head dimension.  A
 * tcgen05 K = 16 MMA step computes what an mma.sync m16n8k16 step computes,
 * bit for bit, and both kernels take the same steps in the same order, so
 * logits are bitwise identical under either choice.  Applies to the steps
 * and attention ops issued after the call (captured step graphs are keyed
 * on it).  Errors: VD_ERR_INVALID_ARG. */
int vd_set_attention_prefill(vd_model* m, int32_t kernel);

/* Graph replay of steps (an engineering addition; the pages' design has no
 * counterpart).  With max_graphs > 0, vd_step keeps the descriptor upload as
 * an ordinary copy on the stream and replays the step's kernel sequence as
 * one CUDA graph, captured the second time its key is seen (the first time
 * runs eagerly, so one-off shapes never pay for a capture).  The key is
 * (pool, logits_out address, T, B, R, page-table stride, number of decode-
 * and prefill-class requests, attention grid sizes); in this mode the
 * stride is rounded up to 64 pages and each attention grid to a 1/16
 * quantum of its item count (extra CTAs exit at once), so steady decode
 * steps share a graph.  The kernels, their arguments and every row's
 * arithmetic are those of the eager path: logits are bitwise identical.
 * At most max_graphs executables are kept (least recently replayed goes
 * first); 0 turns the mode off and frees them.  Profiling (vd_profile_enable)
 * forces the eager path.  A capture costs milliseconds of host time.  Not
 * thread-safe: one host thread drives a model.
 * Errors: VD_ERR_INVALID_ARG (null model, max_graphs < 0). */
int vd_set_graph_mode(vd_model* m, int32_t max_graphs);
/* out4[0] = graphs captured, out4[1] = replays of a cached graph, out4[2] =
 * graphs currently cached, out4[3] = steps run eagerly because their key was
 * new (a key is captured the second time it is seen) (host int64 [4]). */
int vd_graph_stats(const vd_model* m, int64_t* out4);

/* Token choice for R rows of dev float32 logits [R][V] (16-byte aligned) ->
 * dev int32 [R]: the sampler of the engine-step outputs, whose state is
 * part of a request's configuration [B §二 Definition 2.1: sampler_0 and the
 * per-request view (logits, token)], and whose choice is a fixed-order
 * function of the logits row and that state [B §六 6.3: argmax / sampling
 * take finite logits].  Temperature 0: greedy argmax, lowest index on ties.
 * Temperature T > 0: Gumbel-max argmax_i(l_i / T - log(-log(u_i))) with u_i
 * from Philox4x32-10 (Salmon et al., SC'11) keyed by the row's (seed, step)
 * (host array per_row[R]; the generator is this library's choice).  The
 * result depends on the row and its state only, never on R or the other
 * rows.  Errors: VD_ERR_INVALID_ARG (null or misaligned pointers, R < 0). */
int vd_sample(vd_model* m, const float* logits, int32_t R, const vd_sampler* per_row,
              int32_t* tokens_out, void* stream);

/* One engine step with the token choice fused into the LM-head GEMM
 * [B §二 Definition 2.1: per-request sampler_0; Theorem 4.1 for the logits].
 * Same validation, errors and logits as vd_step (logits_out may be NULL:
 * then logits are computed but not stored), and tokens_out (dev int32 [R])
 * holds exactly what vd_sample would choose from those logits: the GEMM
 * epilogue scores each 32-row vocabulary group per token (greedy or
 * Gumbel-max, per-row state in host per_row[R]) and a second kernel picks
 * the (largest score, lowest index) winner, so the logits are never read
 * back.  per_row is copied before the call returns. */
int vd_step_sample(vd_model* m, vd_kv_pool* pool, const vd_batch* b, const vd_sampler* per_row,
                   float* logits_out, int32_t* tokens_out, void* stream);

/* vd_step_sample with device-side token feedback (an engineering addition;
 * the pages have no counterpart).  feed_index: host int32 [num_tokens]; for
 * each t with feed_index[t] >= 0 the step's token t is feed_tokens[feed_index[t]]
 * (dev int32, typically an earlier step's tokens_out; it may be this call's
 * own tokens_out), read on the device when the step runs, and token_ids[t] is
 * ignored; -1 takes token_ids[t] as usual.  A host can thus enqueue step s+1
 * before it has read step s's tokens back.  The caller keeps every index
 * inside its feed buffer.  A fed id outside [0, V) is not read: the step
 * records VD_ERR_OUT_OF_RANGE in the device status word (vd_device_status)
 * and the rest of the step is skipped.  Host-side errors as vd_step_sample,
 * plus VD_ERR_INVALID_ARG for entries below -1 or a null feed_tokens. */
int vd_step_sample_fed(vd_model* m, vd_kv_pool* pool, const vd_batch* b, const int32_t* feed_index,
                       const int32_t* feed_tokens, const vd_sampler* per_row, float* logits_out,
                       int32_t* tokens_out, void* stream);

/* Debug: copies the K and V of `layer` for logical positions [0, n_tokens)
 * of one request (host page table) into dev bf16 out_k / out_v
 * [n_tokens][Hkv][hd], for bitwise checks of the KV-value invariant
 * [B §五 5.1]. */
int vd_copy_kv(vd_model* m, vd_kv_pool* pool, int32_t layer, const int32_t* page_table,
               int32_t n_tokens, void* out_k, void* out_v, void* stream);

/* Reads (synchronising the device) the on-device status word: VD_OK,
 * VD_ERR_TIMEOUT if a bounded wait in a kernel gave up, or VD_ERR_OUT_OF_RANGE
 * if a token fed on the device was outside the vocabulary; clears it.  While
 * it is set, the GEMM and attention kernels skip their work.  They read it
 * before waiting for the kernel ahead of them, so the kernel right after a
 * failing one may still run; every result of a step that set the word is to
 * be discarded either way. */
int vd_device_status(vd_model* m);

/* Per-kernel timing with CUDA events on the launching stream. */
int vd_profile_enable(vd_model* m, int32_t on);
/* Synchronises, returns the number of kernel classes written to out. */
int vd_profile_collect(vd_model* m, vd_kernel_stat* out, int32_t max_out);

const char* vd_last_error(void);
const char* vd_version(void);

#ifdef __cplusplus
}
#endif
#endif /* VD_H_ */
