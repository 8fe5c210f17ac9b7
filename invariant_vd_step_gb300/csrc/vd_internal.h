// Host-side declarations shared by the translation units of libvd.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "vd.h"
#include "vd_ops.h"
#include "vd_engine.h"

namespace vd {

// ---------------------------------------------------------------- errors
void set_error(const std::string& msg);
int fail(int code, const std::string& msg);
#define VD_CUDA_TRY(expr)                                                          \
  do {                                                                             \
    cudaError_t e_ = (expr);                                                       \
    if (e_ != cudaSuccess)                                                         \
      return ::vd::fail(VD_ERR_CUDA, std::string(#expr) + ": " + cudaGetErrorString(e_)); \
  } while (0)

// ---------------------------------------------------------------- launches
// Every kernel of the library is launched with the programmatic-stream-
// serialisation attribute, so it may be scheduled while the previous kernel
// of the stream drains; each kernel waits (griddepcontrol.wait) before it
// touches memory.  VD_PDL=0 in the environment launches without it.
bool pdl_enabled();
template <typename... Exp, typename... Act>
cudaError_t launch_k(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Act&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Act&&>(args)...);
}

// ---------------------------------------------------------------- TMA maps
// 2-D bf16 map over a row-major [rows][cols] matrix; box = box_rows x 64
// columns (128 bytes), 128-byte swizzle, zero fill outside the matrix.
int make_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
// 3-D bf16 map for the KV pool: dims (64, hd/64, rows), box (64, hd/64, 16).
int make_map_kv(CUtensorMap* map, const void* base, uint64_t rows, int hd, int box_blocks);

// ---------------------------------------------------------------- GEMM
// EPI_F32_SAMPLE: fp32 logits (stored unless out is null) plus, per token and
// 32-row vocabulary group, the best (score, index) of the token choice.
// EPI_PARTIAL: fp32 partial sums of one K split (the fast, non-invariant path;
// splitk_reduce applies the real epilogue).
enum Epilogue {
  EPI_BF16 = 0, EPI_RESIDUAL = 1, EPI_F32 = 2, EPI_SWIGLU = 3, EPI_GEGLU = 4, EPI_F32_SAMPLE = 5, EPI_PARTIAL = 6
};
constexpr int kGemmBM = 128;  // weight rows per tile (MMA M); tiles of 64 and 256 rows too
constexpr int kGemmBN = 256;  // most tokens per tile (MMA N)
constexpr int kGemmBK = 64;   // K per block (one 128-byte swizzle row)
constexpr int kNumKpo = 3;    // K blocks per weight copy: 1, 2 or 4
constexpr int kNumBn = 5;     // token tile widths 16, 32, 64, 128, 256

// Launch shape of one GEMM: weight rows per tile (64, 128, or 256 = two
// M = 128 instructions sharing each activation block), tokens per tile
// (16 .. 256, a power of two) and K blocks per weight copy (1, 2, 4).  None
// of them changes the arithmetic of an output element: every element is the
// same chain of K = 16 MMA steps in ascending K order into a zeroed fp32
// accumulator, whatever the instruction's M and N.
struct GemmPlan {
  int bm = 0, bn = 0, kpo = 0;
};

// A weight matrix with one TMA map per (tile height, K blocks per copy):
// plain [rows][K] as (64, row, K block); gate/up [2F][K] as
// (64, half, feature, K block), so a tile stages each gate row next to its up
// row (tile rows 2f, 2f + 1).
struct WeightMaps {
  CUtensorMap m[3][kNumKpo];  // [0: 128 rows, 1: 64 rows, 2: 256 rows (kpo 1 only)][log2 kpo]
  int rows = 0;               // output rows (2F for gate/up)
  int K = 0;
  bool glu = false;
};
int make_weight_maps(WeightMaps* w, const void* base, uint64_t rows, uint64_t K, bool glu);

// Activation rows [rows][cols] with one map per token tile width: map i has a
// box of min(16 << i, rows) rows.
struct ActMaps {
  const CUtensorMap* maps = nullptr;  // [kNumBn]
  int rows = 0;
};

struct GemmArgs {
  void* out;             // [T][ldo] bf16 (or fp32 for EPI_F32)
  const void* residual;  // [T][ldo] bf16 (EPI_RESIDUAL; may alias out)
  int T;                 // valid tokens
  int K;                 // reduction length
  int ldo;               // output row stride (elements)
  int glu_up_row;        // GLU: first row of the up half in the weight matrix (= F)
  int n_wtiles;          // weight tiles (set by launch_gemm)
  const vd_sampler* samp;  // EPI_F32_SAMPLE: per-token sampler state [T]
  float* part_v;           // EPI_F32_SAMPLE: [T][part_stride] group winners' scores
  int* part_i;             //                 and indices
  int part_stride;         //                 = vocab / 32
  int k_splits;          // K splits (1: the invariant path; > 1 only with EPI_PARTIAL)
  int glu;               // EPI_PARTIAL over a GLU weight matrix (gate/up tile layout)
  // set by launch_gemm:
  int bm, bn, kpo;       // the plan
  int b_box_rows;        // rows of the activation TMA box (min(bn, activation rows))
  int b_sub;             // bytes of one K block of B in a stage (>= bn * 128, 1 KB multiple)
  int stage_bytes;       // kpo * (bm * 128 + b_sub)
  int stages;            // pipeline depth
  int* status;           // device status word
};
// Fast path: out = epilogue(sum over ks of part[ks][t][n]) for the T x N
// output (N = 2F for GLU: z[t][f] = act(bf16(gate)) * bf16(up)), summed in
// split order.  epi: EPI_BF16, EPI_RESIDUAL, EPI_SWIGLU or EPI_GEGLU.
int launch_splitk_reduce(const float* part, int k_splits, int T, int N, int epi, void* out, const void* residual,
                         cudaStream_t s);
// The plan launch_gemm takes for T tokens against this matrix (the forced
// plan where one is set, else the estimated fastest).
GemmPlan gemm_plan(const WeightMaps& w, int T, int epi, int k_splits);
// Forced plan for every later launch (fields 0: chosen per launch).
// gemm_plan_epoch() changes whenever the forced plan does.
int set_forced_gemm_plan(GemmPlan p);
unsigned gemm_plan_epoch();
int launch_gemm(const WeightMaps& w, const ActMaps& x, const GemmArgs& a, int epi, cudaStream_t s);
// Once per device: every tile shape on seeded operands, raw fp32 results
// compared bit for bit; *result = 1 if all agree (shapes stay per launch),
// 0 if not (every later launch takes one fixed shape).
int gemm_shapes_self_check(int* result);

// ---------------------------------------------------------------- attention
struct AttnArgs {
  const __nv_bfloat16* q;  // [T][Hq][hd]
  float* part_o;           // [T][Hq][max_splits][hd]
  float* part_ml;          // [T][Hq][max_splits][2]
  const int* cu_q;         // [B+1]
  const int* cached_len;   // [B]
  const int* page_table;   // [B][pt_stride]
  const int* cls_seq;      // seqs of this launch class
  const int* cls_start;    // [n + 1] item prefix sums
  int n_cls;
  int pt_stride;
  int Hq, Hkv;
  int layer_row0;          // first pool row of this layer
  int pool_rows;           // total pool rows (zero-fill coordinate)
  int window;              // 0: global
  int split;               // S_kv keys
  int max_splits;
  float scale_log2;        // log2(e) / sqrt(hd)
  int stages;              // K/V tiles in flight (set by launch_attention)
  int fold;                // decode class: 1 = a CTA walks all splits of its rows and folds them,
                           // writing out directly (no partials); 0 = one CTA per split
  __nv_bfloat16* out;      // [T][Hq][hd] (fold mode)
  int* status;
};
struct MergeArgs {
  const float* part_o;
  const float* part_ml;
  __nv_bfloat16* out;      // [T][Hq][hd]
  const int* positions;    // [T]
  const int* tokens;       // tokens to merge (T of them), or null for 0..T-1
  int T, Hq, window, split, max_splits;
};
int attn_key_tile(int hd);
// Items of one sequence (both host and device use the same formula).
int launch_attention(const CUtensorMap& kvmap, const AttnArgs& a, int hd, bool prefill_class, int n_items,
                     cudaStream_t s);
int launch_merge(const MergeArgs& a, int hd, cudaStream_t s);
// Prefill-class attention on tcgen05 (128 rows per CTA), same per-row
// arithmetic as launch_attention's kernels; kvmap_tc has one-page boxes of
// 64 head dims.
bool attn_tc_supported(int hd);
int launch_attention_tc(const CUtensorMap& kvmap_tc, const AttnArgs& a, int hd, int n_items, cudaStream_t s);
// Fixed-size device scratch of vd_op_attention_static (bytes) and its
// device address on the current device (looked up once per device).
constexpr size_t kAttnStaticScratchBytes = static_cast<size_t>(16) << 20;
int attn_static_scratch(void** ptr);

// ---------------------------------------------------------------- elementwise
// tokens[t] < 0 refers to feed[-1 - tokens[t]] (device tokens of an earlier step).
// scale != 0: x = bf16(E[token] * scale) (Gemma-3 embedding scale).
int launch_embed(const void* embed, const int* tokens, const int* feed, int V, int* status, float scale, void* x,
                 int T, int d, cudaStream_t s);
// y[r] = bf16(x[row_idx[r]] * (1 / sqrt(mean(x^2) + eps)) * (w + gain_offset)).
int launch_rmsnorm(const void* x, const int* row_idx, const void* w, void* y, int rows, int d, float eps,
                   float gain_offset, cudaStream_t s);
// Sandwich norm + residual (+ the next pre-norm): x = bf16(x + rms(h; w_post));
// then, if w_pre is not null, y = rms(x; w_pre).  Gains are w + gain_offset.
int launch_postnorm_residual(const void* h, void* x, const void* w_post, const void* w_pre, void* y, int rows, int d,
                             float eps, float gain_offset, cudaStream_t s);
struct RopeArgs {
  const __nv_bfloat16* qkv;   // [T][(Hq+2Hkv) hd]
  __nv_bfloat16* q_out;       // [T][Hq][hd]
  __nv_bfloat16* pool;        // pool base
  const int* positions;       // [T]
  const int* slot_page;       // [T] physical page of the token's slot
  const float* cos_t;         // [max_ctx][hd/2]
  const float* sin_t;
  const __nv_bfloat16* q_norm;  // nullable
  const __nv_bfloat16* k_norm;
  float eps;
  float gain_offset;          // QK-norm gains are w + gain_offset
  int T, Hq, Hkv, hd;
  long long layer_elem0;      // first element of this layer in the pool
};
int launch_rope_kv(const RopeArgs& a, cudaStream_t s);

// ---------------------------------------------------------------- sampling
// Two passes over [R][V] logits; part_v / part_i hold R * sample_chunks(V) winners.
int sample_chunks(int V);
int launch_sample(const float* logits, int R, int V, const vd_sampler* dev_params, float* part_v, int* part_i,
                  int* out, cudaStream_t s);
// Second pass alone: per row, the best of nchunk (score, index) partials.
int launch_sample_final(const float* part_v, const int* part_i, int R, int nchunk, int* out, cudaStream_t s);
int launch_philox(uint64_t seed, uint64_t step, int n, uint32_t* out, cudaStream_t s);
int launch_wait_probe(int* status, uint64_t limit_ns, int* out, cudaStream_t s);
// Streams a [rows][K] bf16 weight matrix through shared memory with a GEMM
// plan's weight copies (and, if x_box_rows > 0, its activation copies); no
// arithmetic.  ctas = 0: one CTA per SM (at most one per tile).
int launch_tma_stream(const CUtensorMap& wmap, const CUtensorMap& xmap, int rows, int K, int box_rows, int kpo,
                      int x_box_rows, int k_parts, int ctas, int* status, cudaStream_t s);
// One thread issuing n_mma MMAs (M x N x 16), 16 per stage, with an optional
// test (wait 1: test_wait, 2: try_wait) of a completed mbarrier phase per
// stage; out: dev int64 [2] cycles to the last issue and to completion.
int launch_mma_issue_probe(int M, int N, int n_mma, int wait, long long* out, int* status, cudaStream_t s);

}  // namespace vd
