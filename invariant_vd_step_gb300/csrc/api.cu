// C ABI of libvd.so: model creation with kernel choices fixed from the
// model shape, the paged KV pool, descriptor validation and upload, and the
// kernel sequence of one engine step.
//
// Fixed kernel choices (深入解析 Vosti §三 3.2): every constant that shapes a
// reduction -- GEMM tile 128 weight rows x 256 tokens x 64 (MMA 128x256x16),
// attention key tile B_N (32 keys), KV split size S_kv (512 keys), RMSNorm
// lane layout -- is chosen here from (dims, dtype, head geometry, page size)
// and never from a batch.  What varies per step (grid sizes, which TMA map
// bucket covers the T activation rows, the attention CTA shape) changes no
// row's arithmetic.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <array>
#include <atomic>
#include <mutex>
#include <string>
#include <unordered_set>
#include <vector>

#include <cudaTypedefs.h>

#include "vd_device.cuh"
#include "vd_internal.h"

namespace vd {

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("VD_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

static thread_local std::string g_err;
void set_error(const std::string& msg) { g_err = msg; }
int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

// ---------------------------------------------------------------- TMA maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int make_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(VD_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (cols * 2) % 16) return fail(VD_ERR_INVALID_ARG, "TMA base/stride not 16-byte aligned");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(VD_ERR_CUDA, "cuTensorMapEncodeTiled(2d) failed: " + std::to_string(r));
  return VD_OK;
}

int make_weight_maps(WeightMaps* w, const void* base, uint64_t rows, uint64_t K, bool glu) {
  auto fn = encode_fn();
  if (!fn) return fail(VD_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  if ((reinterpret_cast<uintptr_t>(base) & 15) || K % kGemmBK || (glu && rows % 2))
    return fail(VD_ERR_INVALID_ARG, "weight matrix: base not 16-byte aligned or K not a multiple of 64");
  *w = WeightMaps{};
  w->rows = static_cast<int>(rows);
  w->K = static_cast<int>(K);
  w->glu = glu;
  const uint64_t KB = K / kGemmBK, F = rows / 2;
  for (int bi = 0; bi < 3; ++bi)
    for (int ki = 0; ki < kNumKpo; ++ki) {
      const uint32_t bm = bi == 0 ? kGemmBM : bi == 1 ? kGemmBM / 2 : 2 * kGemmBM, kpo = 1u << ki;
      if (KB % kpo) continue;  // never used: a plan's kpo divides the K blocks
      if (bi == 2 && (kpo > 1 || rows % bm)) continue;  // 256-row tiles: one K block per copy
      CUresult r;
      if (!glu) {  // (64, row, K block)
        cuuint64_t dims[3] = {64, rows, KB};
        cuuint64_t strides[2] = {K * 2, 128};
        cuuint32_t box[3] = {64, bm, kpo};
        cuuint32_t estr[3] = {1, 1, 1};
        r = fn(&w->m[bi][ki], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      } else {  // (64, half, feature, K block): gate rows 0..F-1, up rows F..2F-1
        cuuint64_t dims[4] = {64, 2, F, KB};
        cuuint64_t strides[3] = {F * K * 2, K * 2, 128};
        cuuint32_t box[4] = {64, 2, bm / 2, kpo};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        r = fn(&w->m[bi][ki], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      }
      if (r != CUDA_SUCCESS) return fail(VD_ERR_CUDA, "cuTensorMapEncodeTiled(weights) failed: " + std::to_string(r));
    }
  return VD_OK;
}

// K/V pool rows as (64 head dims, hd / 64 blocks, rows).  A box is one page
// (16 rows) of `box_blocks` 64-wide blocks: all hd / 64 for the mma.sync
// kernels (a key's head dims side by side), 1 for the tcgen05 kernel (one
// block of 16 keys, the MMA's canonical operand layout).
int make_map_kv(CUtensorMap* map, const void* base, uint64_t rows, int hd, int box_blocks) {
  auto fn = encode_fn();
  if (!fn) return fail(VD_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(hd / 64), rows};
  cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(hd) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_blocks), 16};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(VD_ERR_CUDA, "cuTensorMapEncodeTiled(kv) failed: " + std::to_string(r));
  return VD_OK;
}

}  // namespace vd

using namespace vd;

namespace {

constexpr int kSplitKeys = 512;  // S_kv, fixed for every model

struct ProfRec {
  int cls;
  int kernels;  // kernel launches between the two events
  cudaEvent_t a, b;
};
const char* const kKernelNames[] = {"embed",     "rmsnorm",  "gemm_qkv",     "rope_kv",   "attention",
                                    "attn_merge", "gemm_o",  "gemm_gate_up", "gemm_down", "final_norm",
                                    "gemm_lm_head", "sample"};
enum KernelClass {
  K_EMBED, K_RMSNORM, K_GEMM_QKV, K_ROPE, K_ATTN, K_MERGE, K_GEMM_O, K_GEMM_GU, K_GEMM_DOWN, K_FINAL_NORM,
  K_GEMM_LM, K_SAMPLE, K_COUNT
};

// Activation buffer with TMA maps for row counts 1, 2, 4, ... (capped at
// the capacity), each in every token tile width: a GEMM over T rows uses the
// smallest row count covering T, so rows past T are either never fetched or
// (within the bucket) computed and discarded -- a GEMM column depends on its
// own row only.
struct ActBuf {
  __nv_bfloat16* ptr = nullptr;
  int cols = 0;
  std::vector<int> rows;
  std::vector<std::array<CUtensorMap, kNumBn>> maps;
  size_t bucket(int T) const {
    for (size_t i = 0; i < rows.size(); ++i)
      if (rows[i] >= T) return i;
    return rows.size() - 1;
  }
  ActMaps view(int T) const {
    ActMaps v;
    v.maps = maps[bucket(T)].data();
    v.rows = rows[bucket(T)];
    return v;
  }
};

// Host-side layout of the uploaded step descriptor (int32 offsets).
struct Desc {
  int T = 0, B = 0, R = 0, stride = 0;
  int tokens, positions, slot_page, cu_q, cached, page_table, logit_rows, dec_seq, dec_start, pre_seq, pre_start;
  // (merge_tok: offset of the token list the merge kernel folds)
  int n_dec = 0, n_pre = 0, items_dec = 0, items_pre = 0;
  bool fold = false;  // decode class in fold mode
  bool pre_tc = false;  // prefill class on the tcgen05 kernel (128 rows per CTA), else mma.sync (64)
  int merge_tok = 0, n_merge = 0;
  int grid_dec = 0, grid_pre = 0;  // attention CTAs launched (>= items; extra CTAs exit)
  int total = 0;
  const int* feed = nullptr;  // device tokens that entries -(1 + i) of `tokens` refer to
};

// What a captured step graph depends on beyond the model: every kernel
// argument and grid size of a step is a function of these fields.
struct GraphKey {
  unsigned long long pool_id = 0;
  const void* logits = nullptr;
  const void* tokens = nullptr;  // fused token choice (vd_step_sample) or null
  const void* feed = nullptr;    // device-side token feedback or null
  int T = 0, B = 0, R = 0, stride = 0, n_dec = 0, n_pre = 0, grid_dec = 0, grid_pre = 0, fold = 0, n_merge = 0;
  int pre_tc = 0;
  int fast = 0;
  unsigned plan_epoch = 0;  // GEMM plan override in force
  bool operator==(const GraphKey& o) const {
    return pool_id == o.pool_id && logits == o.logits && tokens == o.tokens && feed == o.feed && T == o.T && B == o.B && R == o.R && stride == o.stride &&
           n_dec == o.n_dec && n_pre == o.n_pre && grid_dec == o.grid_dec && grid_pre == o.grid_pre &&
           fold == o.fold && pre_tc == o.pre_tc && n_merge == o.n_merge && fast == o.fast &&
           plan_epoch == o.plan_epoch;
  }
};
struct GraphEntry {
  GraphKey key;
  cudaGraphExec_t exec = nullptr;
  long long used = 0;
};

}  // namespace

struct vd_model {
  vd_model_config cfg{};
  int device = 0;
  const __nv_bfloat16* embed = nullptr;
  const __nv_bfloat16* final_norm = nullptr;
  const __nv_bfloat16* lm_head = nullptr;
  std::vector<vd_layer_weights> layers;
  // fixed kernel choices
  int split = kSplitKeys;
  int key_tile = 64;
  int max_splits = 0;
  int G = 1;
  // TMA maps
  std::vector<WeightMaps> m_qkv, m_o, m_gu, m_down;
  WeightMaps m_lm{};
  ActBuf a, o, z, ar;
  // workspace
  __nv_bfloat16 *x = nullptr, *qkv = nullptr, *q = nullptr;
  __nv_bfloat16* hsub = nullptr;  // sandwich norms: a sub-layer's output before its norm
  float embed_scale = 0.f;        // 0: none, else bf16(sqrt(d)) as float
  int fold_mode = 0;              // 0: default (split mode), 1: fold the decode class whenever legal, 2: never
  int prefill_kernel = 0;         // 0: tcgen05 attention for the prefill class where hd allows, 1: mma.sync
  // fast (non-invariant) path: split-K for GEMMs with too few weight tiles
  int fast = 0;
  int n_sm = 0;
  float* splitk_part = nullptr;
  size_t splitk_cap = 0;          // floats
  std::vector<int> scratch_dec;   // host scratch of build_desc
  float gain_offset = 0.f;        // RMSNorm gains are w + gain_offset
  float *part_o = nullptr, *part_ml = nullptr;
  float *cos_g = nullptr, *sin_g = nullptr, *cos_l = nullptr, *sin_l = nullptr;
  int* status = nullptr;
  int* d_desc = nullptr;
  int* h_desc[2] = {nullptr, nullptr};
  cudaEvent_t desc_ev[2] = {nullptr, nullptr};
  int desc_slot = 0;
  size_t desc_cap = 0;
  vd_sampler* d_samp = nullptr;
  float* samp_part_v = nullptr;  // per-chunk winners of the sampler's first pass
  int* samp_part_i = nullptr;
  float* fused_part_v = nullptr;  // per-32-row-group winners of the fused LM-head epilogue
  int* fused_part_i = nullptr;
  vd_sampler* h_samp = nullptr;
  cudaEvent_t samp_ev = nullptr;
  std::vector<void*> dev_allocs;
  // profiling
  bool profiling = false;
  std::vector<ProfRec> recs;
  std::vector<cudaEvent_t> ev_pool;
  double prof_ms[K_COUNT] = {};
  int prof_n[K_COUNT] = {};
  int prof_k[K_COUNT] = {};
  // graph replay of steps
  int graph_max = 0;
  cudaStream_t cap_stream = nullptr;
  std::vector<GraphEntry> graphs;
  long long graph_clock = 0, graph_captures = 0, graph_replays = 0, graph_eager = 0;
};

struct vd_kv_pool {
  vd_model* m = nullptr;
  unsigned long long id = 0;  // never reused, unlike the host address
  int num_pages = 0;
  void* data = nullptr;
  bool owned = false;
  long long rows = 0;  // 16-slot rows of hd elements
  CUtensorMap map{};     // boxes for the mma.sync attention kernels
  CUtensorMap map_tc{};  // boxes for the tcgen05 attention kernel
};

namespace {

// ---------------------------------------------------------------- profiling
cudaEvent_t take_event(vd_model* m) {
  if (!m->ev_pool.empty()) {
    cudaEvent_t e = m->ev_pool.back();
    m->ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
struct Prof {
  vd_model* m;
  int cls;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  int kernels = 1;
  Prof(vd_model* m_, int cls_, cudaStream_t s_) : m(m_), cls(cls_), s(s_) {
    if (m->profiling) {
      a = take_event(m);
      cudaEventRecord(a, s);
    }
  }
  ~Prof() {
    if (m->profiling) {
      cudaEvent_t b = take_event(m);
      cudaEventRecord(b, s);
      m->recs.push_back({cls, kernels, a, b});
    }
  }
};

int dev_alloc(vd_model* m, void** p, size_t bytes) {
  if (bytes == 0) bytes = 256;
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) return fail(VD_ERR_CUDA, std::string("cudaMalloc: ") + cudaGetErrorString(e));
  m->dev_allocs.push_back(*p);
  cudaMemset(*p, 0, bytes);
  return VD_OK;
}

int make_act(vd_model* m, ActBuf& buf, int cap_rows, int cols) {
  int rc = dev_alloc(m, reinterpret_cast<void**>(&buf.ptr), static_cast<size_t>(cap_rows) * cols * 2);
  if (rc) return rc;
  buf.cols = cols;
  for (int r = 1;; r *= 2) {
    const int rows = std::min(r, cap_rows);
    std::array<CUtensorMap, kNumBn> mp;
    for (int i = 0; i < kNumBn; ++i)
      if ((rc = make_map_2d(&mp[i], buf.ptr, rows, cols, std::min(rows, 16 << i)))) return rc;
    buf.rows.push_back(rows);
    buf.maps.push_back(mp);
    if (rows >= cap_rows) break;
  }
  return VD_OK;
}

int rope_table(vd_model* m, float theta, int hd, float** cs, float** sn) {
  const int half = hd / 2;
  const size_t n = static_cast<size_t>(m->cfg.max_context) * half;
  std::vector<float> c(n), s(n);
  for (int p = 0; p < m->cfg.max_context; ++p)
    for (int i = 0; i < half; ++i) {
      const double inv = pow(static_cast<double>(theta), -2.0 * i / hd);
      const double ang = static_cast<double>(p) * inv;
      c[static_cast<size_t>(p) * half + i] = static_cast<float>(cos(ang));
      s[static_cast<size_t>(p) * half + i] = static_cast<float>(sin(ang));
    }
  int rc;
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(cs), n * 4))) return rc;
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(sn), n * 4))) return rc;
  VD_CUDA_TRY(cudaMemcpy(*cs, c.data(), n * 4, cudaMemcpyHostToDevice));
  VD_CUDA_TRY(cudaMemcpy(*sn, s.data(), n * 4, cudaMemcpyHostToDevice));
  return VD_OK;
}

bool layer_is_local(const vd_model_config& c, int i) {
  return c.sliding_window > 0 && c.local_global_period > 0 && ((i + 1) % c.local_global_period) != 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Items of one attention work class for request with q_len, kv_len.
int attn_items(int qlen, int kv_len, int G, int Hkv, int rows_per_cta) {
  const int rows = qlen * G;
  const int nrb = (rows + rows_per_cta - 1) / rows_per_cta;
  const int nsplit = (kv_len - 1) / kSplitKeys + 1;
  return nrb * Hkv * nsplit;
}

// Validates a step descriptor and builds the upload image in h.
// Highest power of two <= n, divided by 16, is the rounding quantum: at most
// 1/16 of the CTAs are extra, and the rounded count changes rarely as
// contexts grow.
int bucket_items(int n) {
  if (n <= 16) return n;
  int p = 1;
  while (p <= n / 2) p *= 2;
  const int q = p / 16;
  return (n + q - 1) / q * q;
}

// graph_shape rounds the page-table stride up to 64 pages and the attention
// grids with bucket_items(), so that consecutive decode steps share one
// captured graph; neither changes any row's arithmetic.
// feed_index (host [T] or null): token t with feed_index[t] >= 0 is taken on
// the device from the step's feed buffer; its descriptor entry is
// -(1 + feed_index[t]).
int build_desc(vd_model* m, vd_kv_pool* pool, const vd_batch* b, bool need_tokens, Desc& d, int* h,
               bool graph_shape = false, const int32_t* feed_index = nullptr) {
  const vd_model_config& c = m->cfg;
  if (!b) return fail(VD_ERR_INVALID_ARG, "null batch");
  const int T = b->num_tokens, B = b->num_seqs, R = b->num_logit_rows;
  if (T < 0 || B < 0 || R < 0) return fail(VD_ERR_INVALID_ARG, "negative size");
  if (T > c.max_tokens || B > c.max_seqs || R > c.max_logit_rows)
    return fail(VD_ERR_CAPACITY, "step exceeds max_tokens / max_seqs / max_logit_rows");
  if (T == 0) {
    d.T = 0;
    return VD_OK;
  }
  if (B == 0 || !b->cu_q || !b->cached_len || !b->page_table || !b->positions)
    return fail(VD_ERR_INVALID_ARG, "missing descriptor array");
  if (need_tokens && !b->token_ids) return fail(VD_ERR_INVALID_ARG, "missing token_ids");
  if (R > 0 && !b->logit_rows) return fail(VD_ERR_INVALID_ARG, "missing logit_rows");
  if (b->cu_q[0] != 0 || b->cu_q[B] != T) return fail(VD_ERR_INVALID_ARG, "cu_q must run from 0 to num_tokens");
  int stride = 0;
  for (int s = 0; s < B; ++s) {
    const int ql = b->cu_q[s + 1] - b->cu_q[s];
    if (ql < 1) return fail(VD_ERR_INVALID_ARG, "every request needs q_len >= 1");
    if (b->cached_len[s] < 0) return fail(VD_ERR_INVALID_ARG, "negative cached_len");
    const long long kv = static_cast<long long>(b->cached_len[s]) + ql;
    if (kv > c.max_context) return fail(VD_ERR_CAPACITY, "request exceeds max_context");
    const int np = static_cast<int>((kv + 15) / 16);
    if (np > b->page_table_stride) return fail(VD_ERR_OUT_OF_RANGE, "page table narrower than the request");
    stride = std::max(stride, np);
  }
  if (graph_shape) stride = std::min((stride + 63) / 64 * 64, (c.max_context + 15) / 16);
  d.T = T;
  d.B = B;
  d.R = R;
  d.stride = stride;
  int off = 0;
  auto take = [&](int n) {
    const int o = off;
    off += n;
    return o;
  };
  d.tokens = take(T);
  d.positions = take(T);
  d.slot_page = take(T);
  d.cu_q = take(B + 1);
  d.cached = take(B);
  d.page_table = take(B * stride);
  d.logit_rows = take(R);
  d.dec_seq = take(B);
  d.dec_start = take(B + 1);
  d.pre_seq = take(B);
  d.pre_start = take(B + 1);
  d.merge_tok = take(T);
  d.total = off;
  if (static_cast<size_t>(off) > m->desc_cap) return fail(VD_ERR_CAPACITY, "descriptor exceeds capacity");
  std::unordered_set<long long> slots;
  slots.reserve(static_cast<size_t>(T) * 2);
  const int V = c.vocab;
  for (int s = 0; s < B; ++s) {
    const int q0 = b->cu_q[s], ql = b->cu_q[s + 1] - q0, cached = b->cached_len[s];
    const int np = (cached + ql + 15) / 16;
    for (int i = 0; i < np; ++i) {
      const int pg = b->page_table[static_cast<size_t>(s) * b->page_table_stride + i];
      if (pg < 0 || pg >= pool->num_pages) return fail(VD_ERR_OUT_OF_RANGE, "page id out of range");
      h[d.page_table + s * stride + i] = pg;
    }
    for (int i = np; i < stride; ++i) h[d.page_table + s * stride + i] = 0;
    for (int i = 0; i < ql; ++i) {
      const int t = q0 + i, p = cached + i;
      if (b->positions[t] != p) return fail(VD_ERR_INVALID_ARG, "positions[t] must equal cached_len + offset");
      const bool fed = feed_index && feed_index[t] >= 0;
      if (feed_index && feed_index[t] < -1) return fail(VD_ERR_INVALID_ARG, "feed_index entries must be >= -1");
      if (need_tokens && !fed && (b->token_ids[t] < 0 || b->token_ids[t] >= V))
        return fail(VD_ERR_OUT_OF_RANGE, "token id out of range");
      const int pg = h[d.page_table + s * stride + p / 16];
      if (!slots.insert(static_cast<long long>(pg) * 16 + (p & 15)).second)
        return fail(VD_ERR_INVALID_ARG, "two new tokens of the step write the same KV slot");
      h[d.tokens + t] = fed ? -1 - feed_index[t] : need_tokens ? b->token_ids[t] : 0;
      h[d.positions + t] = p;
      h[d.slot_page + t] = pg;
    }
    h[d.cu_q + s] = q0;
    h[d.cached + s] = cached;
  }
  h[d.cu_q + B] = T;
  for (int j = 0; j < R; ++j) {
    if (b->logit_rows[j] < 0 || b->logit_rows[j] >= T) return fail(VD_ERR_OUT_OF_RANGE, "logit row out of range");
    h[d.logit_rows + j] = b->logit_rows[j];
  }
  // attention work classes: decode-shaped requests (one warp of rows) and the rest
  d.pre_tc = m->prefill_kernel == 0 && attn_tc_supported(c.head_dim);
  const int pre_rows = d.pre_tc ? 128 : 64;  // rows per prefill-class CTA
  int nd = 0, npre = 0, ipre = 0;
  std::vector<int>& dec = m->scratch_dec;
  dec.clear();
  for (int s = 0; s < B; ++s) {
    const int ql = b->cu_q[s + 1] - b->cu_q[s], kv = b->cached_len[s] + ql;
    if (ql * m->G <= 16) {
      dec.push_back(s);
      ++nd;
    } else {
      h[d.pre_seq + npre] = s;
      h[d.pre_start + npre] = ipre;
      ipre += attn_items(ql, kv, m->G, c.n_kv_heads, pre_rows);
      ++npre;
    }
  }
  // Fold mode (one CTA per request and KV head, folding its splits itself)
  // only on request: on this GPU it never beat split mode (a fold CTA walks
  // its splits one after another, so a long request sets the launch's
  // critical path, and its merged state costs registers).  In fold mode the
  // longest requests go first.  Neither mode changes a row's arithmetic.
  d.fold = nd > 0 && c.head_dim <= 128 && m->fold_mode == 1;
  if (d.fold)
    std::stable_sort(dec.begin(), dec.end(), [&](int x, int y) {
      return b->cached_len[x] + b->cu_q[x + 1] - b->cu_q[x] > b->cached_len[y] + b->cu_q[y + 1] - b->cu_q[y];
    });
  int idec = 0;
  for (int k = 0; k < nd; ++k) {
    const int s = dec[k], ql = b->cu_q[s + 1] - b->cu_q[s], kv = b->cached_len[s] + ql;
    h[d.dec_seq + k] = s;
    h[d.dec_start + k] = idec;
    idec += d.fold ? c.n_kv_heads : attn_items(ql, kv, m->G, c.n_kv_heads, 16);
  }
  h[d.dec_start + nd] = idec;
  h[d.pre_start + npre] = ipre;
  d.n_dec = nd;
  d.n_pre = npre;
  d.items_dec = idec;
  d.items_pre = ipre;
  d.grid_dec = graph_shape ? bucket_items(idec) : idec;
  d.grid_pre = graph_shape ? bucket_items(ipre) : ipre;
  // tokens the merge kernel folds: all of them, or only the prefill class's
  d.n_merge = T;
  if (d.fold) {
    d.n_merge = 0;
    for (int k = 0; k < npre; ++k) {
      const int s = h[d.pre_seq + k];
      for (int t = b->cu_q[s]; t < b->cu_q[s + 1]; ++t) h[d.merge_tok + d.n_merge++] = t;
    }
  }
  return VD_OK;
}

int upload_desc(vd_model* m, vd_kv_pool* pool, const vd_batch* b, bool need_tokens, Desc& d, cudaStream_t s,
                bool graph_shape = false, const int32_t* feed_index = nullptr) {
  const int slot = m->desc_slot;
  m->desc_slot ^= 1;
  VD_CUDA_TRY(cudaEventSynchronize(m->desc_ev[slot]));  // previous upload from this staging slot is done
  int* h = m->h_desc[slot];
  int rc = build_desc(m, pool, b, need_tokens, d, h, graph_shape, feed_index);
  if (rc || d.T == 0) return rc;
  VD_CUDA_TRY(cudaMemcpyAsync(m->d_desc, h, static_cast<size_t>(d.total) * 4, cudaMemcpyHostToDevice, s));
  VD_CUDA_TRY(cudaEventRecord(m->desc_ev[slot], s));
  return VD_OK;
}

int run_attention(vd_model* m, vd_kv_pool* pool, int layer, const Desc& d, const __nv_bfloat16* q,
                  __nv_bfloat16* out, cudaStream_t s) {
  const vd_model_config& c = m->cfg;
  const int hd = c.head_dim;
  const int window = layer_is_local(c, layer) ? c.sliding_window : 0;
  AttnArgs a{};
  a.q = q;
  a.part_o = m->part_o;
  a.part_ml = m->part_ml;
  a.cu_q = m->d_desc + d.cu_q;
  a.cached_len = m->d_desc + d.cached;
  a.page_table = m->d_desc + d.page_table;
  a.pt_stride = d.stride;
  a.Hq = c.n_heads;
  a.Hkv = c.n_kv_heads;
  a.layer_row0 = static_cast<int>(static_cast<long long>(layer) * pool->num_pages * 2 * c.n_kv_heads * 16);
  a.pool_rows = static_cast<int>(pool->rows);
  a.window = window;
  a.split = m->split;
  a.max_splits = m->max_splits;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(hd)));
  a.status = m->status;
  int rc;
  if (d.n_dec) {
    Prof p(m, K_ATTN, s);
    a.cls_seq = m->d_desc + d.dec_seq;
    a.cls_start = m->d_desc + d.dec_start;
    a.n_cls = d.n_dec;
    a.fold = d.fold;
    a.out = out;
    if ((rc = launch_attention(pool->map, a, hd, false, d.grid_dec, s))) return rc;
    a.fold = 0;
  }
  if (d.n_pre) {
    Prof p(m, K_ATTN, s);
    a.cls_seq = m->d_desc + d.pre_seq;
    a.cls_start = m->d_desc + d.pre_start;
    a.n_cls = d.n_pre;
    if ((rc = d.pre_tc ? launch_attention_tc(pool->map_tc, a, hd, d.grid_pre, s)
                        : launch_attention(pool->map, a, hd, true, d.grid_pre, s)))
      return rc;
  }
  if (d.n_merge == 0) return VD_OK;  // every row was folded inside the attention kernel
  MergeArgs g{};
  g.part_o = m->part_o;
  g.part_ml = m->part_ml;
  g.out = out;
  g.positions = m->d_desc + d.positions;
  g.tokens = d.fold ? m->d_desc + d.merge_tok : nullptr;
  g.T = d.n_merge;
  g.Hq = c.n_heads;
  g.window = window;
  g.split = m->split;
  g.max_splits = m->max_splits;
  Prof p(m, K_MERGE, s);
  return launch_merge(g, hd, s);
}

int run_rope(vd_model* m, vd_kv_pool* pool, int layer, const Desc& d, const __nv_bfloat16* qkv,
             __nv_bfloat16* q_out, cudaStream_t s) {
  const vd_model_config& c = m->cfg;
  const bool local = layer_is_local(c, layer);
  RopeArgs r{};
  r.qkv = qkv;
  r.q_out = q_out;
  r.pool = static_cast<__nv_bfloat16*>(pool->data);
  r.positions = m->d_desc + d.positions;
  r.slot_page = m->d_desc + d.slot_page;
  r.cos_t = local ? m->cos_l : m->cos_g;
  r.sin_t = local ? m->sin_l : m->sin_g;
  r.q_norm = c.qk_norm ? static_cast<const __nv_bfloat16*>(m->layers[layer].q_norm) : nullptr;
  r.k_norm = c.qk_norm ? static_cast<const __nv_bfloat16*>(m->layers[layer].k_norm) : nullptr;
  r.eps = c.rms_eps;
  r.gain_offset = m->gain_offset;
  r.T = d.T;
  r.Hq = c.n_heads;
  r.Hkv = c.n_kv_heads;
  r.hd = c.head_dim;
  r.layer_elem0 = static_cast<long long>(layer) * pool->num_pages * 2 * c.n_kv_heads * 16 * c.head_dim;
  Prof p(m, K_ROPE, s);
  return launch_rope_kv(r, s);
}

// vd_op_attention with the split partials in caller-independent static
// scratch (part_o / part_ml, row stride `splits`) instead of the workspace.
int run_attention_static(vd_model* m, vd_kv_pool* pool, int layer, const Desc& d, const __nv_bfloat16* q,
                         __nv_bfloat16* out, float* part_o, float* part_ml, int splits, cudaStream_t s) {
  const vd_model_config& c = m->cfg;
  const int hd = c.head_dim;
  const int window = layer_is_local(c, layer) ? c.sliding_window : 0;
  AttnArgs a{};
  a.q = q;
  a.part_o = part_o;
  a.part_ml = part_ml;
  a.cu_q = m->d_desc + d.cu_q;
  a.cached_len = m->d_desc + d.cached;
  a.page_table = m->d_desc + d.page_table;
  a.pt_stride = d.stride;
  a.Hq = c.n_heads;
  a.Hkv = c.n_kv_heads;
  a.layer_row0 = static_cast<int>(static_cast<long long>(layer) * pool->num_pages * 2 * c.n_kv_heads * 16);
  a.pool_rows = static_cast<int>(pool->rows);
  a.window = window;
  a.split = m->split;
  a.max_splits = splits;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(hd)));
  a.status = m->status;
  int rc;
  if (d.n_dec) {
    a.cls_seq = m->d_desc + d.dec_seq;
    a.cls_start = m->d_desc + d.dec_start;
    a.n_cls = d.n_dec;
    a.fold = d.fold;
    a.out = out;
    if ((rc = launch_attention(pool->map, a, hd, false, d.items_dec, s))) return rc;
    a.fold = 0;
  }
  if (d.n_pre) {
    a.cls_seq = m->d_desc + d.pre_seq;
    a.cls_start = m->d_desc + d.pre_start;
    a.n_cls = d.n_pre;
    if ((rc = d.pre_tc ? launch_attention_tc(pool->map_tc, a, hd, d.items_pre, s)
                        : launch_attention(pool->map, a, hd, true, d.items_pre, s)))
      return rc;
  }
  if (d.n_merge == 0) return VD_OK;
  MergeArgs g{};
  g.part_o = part_o;
  g.part_ml = part_ml;
  g.out = out;
  g.positions = m->d_desc + d.positions;
  g.tokens = d.fold ? m->d_desc + d.merge_tok : nullptr;
  g.T = d.n_merge;
  g.Hq = c.n_heads;
  g.window = window;
  g.split = m->split;
  g.max_splits = splits;
  return launch_merge(g, hd, s);
}

// Status word for the single-kernel ops (they have no model): one int per
// device, allocated on first use and never freed, so a failed bounded wait
// in an op makes its remaining CTAs skip their work.
int* op_status() {
  static std::mutex mu;
  static int* words[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!words[dev] && cudaMalloc(reinterpret_cast<void**>(&words[dev]), 256) == cudaSuccess)
    cudaMemset(words[dev], 0, 256);
  return words[dev];
}

int check_model(const vd_model* m) { return m ? VD_OK : fail(VD_ERR_INVALID_ARG, "null model"); }

// Fast path only: tokens per step up to which narrow GEMMs split K.
constexpr int kFastMaxTokens = 256;

// K splits of a GEMM on the fast path: enough tiles for every SM, at most 8,
// at least two K blocks per split; 1 (no split) on the invariant path.
int fast_splits(const vd_model* m, int T, int n_wtiles, int K) {
  if (!m->fast || T > kFastMaxTokens) return 1;
  const int ntt = (T + kGemmBN - 1) / kGemmBN;
  const int ks = std::min({8, m->n_sm / (ntt * n_wtiles), K / kGemmBK / 2});
  return ks >= 2 ? ks : 1;
}

// One GEMM of the step.  The invariant path fuses the epilogue; the fast
// path may split K (fp32 partials, then a reduction kernel applying the same
// epilogue), which is not batch-invariant.
int gemm_step(vd_model* m, const WeightMaps& w, const ActBuf& xb, int T, int ldo, void* out, const void* residual,
              int epi, int glu_up_row, Prof& p, cudaStream_t s) {
  GemmArgs g{};
  g.status = m->status;
  g.T = T;
  g.K = w.K;
  g.ldo = ldo;
  g.out = out;
  g.residual = residual;
  g.glu_up_row = glu_up_row;
  const bool glu = epi == EPI_SWIGLU || epi == EPI_GEGLU;
  const int ks = fast_splits(m, T, w.rows / kGemmBM, w.K);
  const int np = glu ? 2 * glu_up_row : ldo;  // width of the partial sums
  if (ks == 1 || static_cast<size_t>(ks) * T * np > m->splitk_cap) return launch_gemm(w, xb.view(T), g, epi, s);
  g.out = m->splitk_part;
  g.ldo = np;
  g.residual = nullptr;
  g.k_splits = ks;
  g.glu = glu;
  int rc;
  if ((rc = launch_gemm(w, xb.view(T), g, EPI_PARTIAL, s))) return rc;
  p.kernels = 2;
  return launch_splitk_reduce(m->splitk_part, ks, T, np, epi, out, residual, s);
}

// The kernel sequence of one step (descriptor already uploaded).
int enqueue_step(vd_model* m, vd_kv_pool* pool, const Desc& d, float* logits_out, int* tokens_out, cudaStream_t s) {
  int rc;
  const vd_model_config& c = m->cfg;
  const int T = d.T, dm = c.d_model, hd = c.head_dim, F = c.ffn_dim;
  const int qkv_dim = (c.n_heads + 2 * c.n_kv_heads) * hd;
  const float off = m->gain_offset;
  const bool sandwich = c.sandwich_norm != 0;
  {
    Prof p(m, K_EMBED, s);
    if ((rc = launch_embed(m->embed, m->d_desc + d.tokens, d.feed, c.vocab, m->status, m->embed_scale, m->x, T, dm,
                           s)))
      return rc;
  }
  for (int l = 0; l < c.n_layers; ++l) {
    const vd_layer_weights& L = m->layers[l];
    if (l == 0 || !sandwich) {  // with sandwich norms the previous layer's last kernel produced it
      Prof p(m, K_RMSNORM, s);
      if ((rc = launch_rmsnorm(m->x, nullptr, L.attn_norm, m->a.ptr, T, dm, c.rms_eps, off, s))) return rc;
    }
    {
      Prof p(m, K_GEMM_QKV, s);
      if ((rc = gemm_step(m, m->m_qkv[l], m->a, T, qkv_dim, m->qkv, nullptr, EPI_BF16, 0, p, s)))
        return rc;
    }
    if ((rc = run_rope(m, pool, l, d, m->qkv, m->q, s))) return rc;
    if ((rc = run_attention(m, pool, l, d, m->q, m->o.ptr, s))) return rc;
    if (sandwich) {
      // h = bf16(o Wo^T); x = bf16(x + rms_post(h)); a = rms_ffn(x)
      {
        Prof p(m, K_GEMM_O, s);
        if ((rc = gemm_step(m, m->m_o[l], m->o, T, dm, m->hsub, nullptr, EPI_BF16, 0, p, s)))
          return rc;
      }
      Prof p(m, K_RMSNORM, s);
      if ((rc = launch_postnorm_residual(m->hsub, m->x, L.post_attn_norm, L.ffn_norm, m->a.ptr, T, dm, c.rms_eps,
                                         off, s)))
        return rc;
    } else {
      {
        Prof p(m, K_GEMM_O, s);
        if ((rc = gemm_step(m, m->m_o[l], m->o, T, dm, m->x, m->x, EPI_RESIDUAL, 0, p, s)))
          return rc;
      }
      Prof p(m, K_RMSNORM, s);
      if ((rc = launch_rmsnorm(m->x, nullptr, L.ffn_norm, m->a.ptr, T, dm, c.rms_eps, off, s))) return rc;
    }
    {
      Prof p(m, K_GEMM_GU, s);
      if ((rc = gemm_step(m, m->m_gu[l], m->a, T, F, m->z.ptr, nullptr,
                          c.act == VD_ACT_GEGLU ? EPI_GEGLU : EPI_SWIGLU, F, p, s)))
        return rc;
    }
    if (sandwich) {
      // h = bf16(z Wd^T); x = bf16(x + rms_post(h)); a = rms_attn of the next layer (none after the last)
      {
        Prof p(m, K_GEMM_DOWN, s);
        if ((rc = gemm_step(m, m->m_down[l], m->z, T, dm, m->hsub, nullptr, EPI_BF16, 0, p, s)))
          return rc;
      }
      const void* next_norm = l + 1 < c.n_layers ? m->layers[l + 1].attn_norm : nullptr;
      Prof p(m, K_RMSNORM, s);
      if ((rc = launch_postnorm_residual(m->hsub, m->x, L.post_ffn_norm, next_norm, m->a.ptr, T, dm, c.rms_eps, off,
                                         s)))
        return rc;
    } else {
      Prof p(m, K_GEMM_DOWN, s);
      if ((rc = gemm_step(m, m->m_down[l], m->z, T, dm, m->x, m->x, EPI_RESIDUAL, 0, p, s))) return rc;
    }
  }
  if (d.R > 0) {
    {
      Prof p(m, K_FINAL_NORM, s);
      if ((rc = launch_rmsnorm(m->x, m->d_desc + d.logit_rows, m->final_norm, m->ar.ptr, d.R, dm, c.rms_eps, off, s)))
        return rc;
    }
    {
      Prof p(m, K_GEMM_LM, s);
      GemmArgs h{};
      h.status = m->status;
      h.T = d.R;
      h.out = logits_out;
      h.K = dm;
      h.ldo = c.vocab;
      if (tokens_out) {
        h.samp = m->d_samp;
        h.part_v = m->fused_part_v;
        h.part_i = m->fused_part_i;
        h.part_stride = c.vocab / 32;
      }
      if ((rc = launch_gemm(m->m_lm, m->ar.view(d.R), h, tokens_out ? EPI_F32_SAMPLE : EPI_F32,
                            s)))
        return rc;
    }
    if (tokens_out) {
      Prof p(m, K_SAMPLE, s);
      if ((rc = launch_sample_final(m->fused_part_v, m->fused_part_i, d.R, c.vocab / 32, tokens_out, s))) return rc;
    }
  }
  return VD_OK;
}

// Replays the graph captured for d's key.  A key seen for the first time
// runs eagerly and is remembered; the second time it is captured, so one-off
// shapes (continuous batching with requests joining and leaving) never pay
// for a capture.  Capture runs on a private stream (the legacy default
// stream cannot be captured); the replay is launched on s, after the
// descriptor upload.
int replay_step(vd_model* m, vd_kv_pool* pool, const Desc& d, float* logits_out, int* tokens_out, cudaStream_t s) {
  GraphKey k;
  k.pool_id = pool->id;
  k.logits = logits_out;
  k.tokens = tokens_out;
  k.feed = d.feed;
  k.T = d.T;
  k.B = d.B;
  k.R = d.R;
  k.stride = d.stride;
  k.n_dec = d.n_dec;
  k.n_pre = d.n_pre;
  k.grid_dec = d.grid_dec;
  k.grid_pre = d.grid_pre;
  k.fold = d.fold;
  k.pre_tc = d.pre_tc;
  k.n_merge = d.n_merge;
  k.fast = m->fast;
  k.plan_epoch = gemm_plan_epoch();
  GraphEntry* seen = nullptr;
  for (GraphEntry& e : m->graphs)
    if (e.key == k) {
      e.used = ++m->graph_clock;
      if (e.exec) {
        ++m->graph_replays;
        VD_CUDA_TRY(cudaGraphLaunch(e.exec, s));
        return VD_OK;
      }
      seen = &e;
      break;
    }
  if (!seen) {  // first sight: remember the key, run eagerly
    if (static_cast<int>(m->graphs.size()) >= m->graph_max) {
      auto lru = std::min_element(m->graphs.begin(), m->graphs.end(),
                                  [](const GraphEntry& a, const GraphEntry& b) { return a.used < b.used; });
      if (lru->exec) cudaGraphExecDestroy(lru->exec);  // freed after any launch still in flight
      m->graphs.erase(lru);
    }
    m->graphs.push_back({k, nullptr, ++m->graph_clock});
    ++m->graph_eager;
    return enqueue_step(m, pool, d, logits_out, tokens_out, s);
  }
  if (!m->cap_stream) VD_CUDA_TRY(cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking));
  VD_CUDA_TRY(cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeRelaxed));
  const int rc = enqueue_step(m, pool, d, logits_out, tokens_out, m->cap_stream);
  cudaGraph_t g = nullptr;
  const cudaError_t ce = cudaStreamEndCapture(m->cap_stream, &g);
  if (rc || ce != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return rc ? rc : fail(VD_ERR_CUDA, std::string("step capture: ") + cudaGetErrorString(ce));
  }
  cudaGraphExec_t x = nullptr;
  const cudaError_t ie = cudaGraphInstantiate(&x, g, 0);
  cudaGraphDestroy(g);
  if (ie != cudaSuccess) return fail(VD_ERR_CUDA, std::string("graph instantiate: ") + cudaGetErrorString(ie));
  seen->exec = x;
  ++m->graph_captures;
  VD_CUDA_TRY(cudaGraphLaunch(x, s));
  return VD_OK;
}

void drop_graphs(vd_model* m) {
  for (GraphEntry& e : m->graphs)
    if (e.exec) cudaGraphExecDestroy(e.exec);
  m->graphs.clear();
}


}  // namespace

// ====================================================================== API
extern "C" {

const char* vd_last_error(void) { return g_err.c_str(); }
const char* vd_version(void) { return "vd 0.1 (sm_103a)"; }

int vd_create_model(const vd_model_config* cfg, const vd_weight_ptrs* w, vd_model** out) {
  if (!cfg || !w || !out) return fail(VD_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  const vd_model_config& c = *cfg;
  if (c.n_layers < 1 || c.d_model < 1 || c.n_heads < 1 || c.n_kv_heads < 1 || c.ffn_dim < 1 || c.vocab < 1 ||
      c.max_tokens < 1 || c.max_seqs < 1 || c.max_logit_rows < 1 || c.max_context < 1)
    return fail(VD_ERR_INVALID_ARG, "non-positive dimension or capacity");
  if (c.n_heads % c.n_kv_heads) return fail(VD_ERR_INVALID_ARG, "n_heads must be a multiple of n_kv_heads");
  if (c.page_size != 16) return fail(VD_ERR_UNSUPPORTED, "page_size must be 16");
  if (c.head_dim != 64 && c.head_dim != 128 && c.head_dim != 256)
    return fail(VD_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
  if (c.d_model % kGemmBM || c.vocab % kGemmBM || c.ffn_dim % 64 || c.ffn_dim % kGemmBK ||
      ((c.n_heads + 2 * c.n_kv_heads) * c.head_dim) % kGemmBM || (c.n_heads * c.head_dim) % kGemmBK ||
      c.d_model % kGemmBK)
    return fail(VD_ERR_UNSUPPORTED, "no fixed GEMM tiling: d, V, (Hq+2Hkv)hd must be multiples of 128; F, Hq*hd multiples of 64");
  if (c.n_heads / c.n_kv_heads > 16) return fail(VD_ERR_UNSUPPORTED, "GQA group larger than 16");
  if (c.act != VD_ACT_SWIGLU && c.act != VD_ACT_GEGLU) return fail(VD_ERR_INVALID_ARG, "unknown activation");
  if (c.sliding_window < 0 || c.local_global_period < 0) return fail(VD_ERR_INVALID_ARG, "negative window");
  if (!w->embed || !w->final_norm || !w->lm_head || !w->layers) return fail(VD_ERR_INVALID_ARG, "null weight");
  for (int i = 0; i < c.n_layers; ++i) {
    const vd_layer_weights& L = w->layers[i];
    if (!L.attn_norm || !L.wqkv || !L.wo || !L.ffn_norm || !L.w_gate_up || !L.w_down ||
        (c.qk_norm && (!L.q_norm || !L.k_norm)) || (c.sandwich_norm && (!L.post_attn_norm || !L.post_ffn_norm)))
      return fail(VD_ERR_INVALID_ARG, "null layer weight");
    if (c.sandwich_norm && (!aligned16(L.post_attn_norm) || !aligned16(L.post_ffn_norm)))
      return fail(VD_ERR_INVALID_ARG, "weights must be 16-byte aligned");
    if (!aligned16(L.wqkv) || !aligned16(L.wo) || !aligned16(L.w_gate_up) || !aligned16(L.w_down) ||
        !aligned16(L.attn_norm) || !aligned16(L.ffn_norm))
      return fail(VD_ERR_INVALID_ARG, "weights must be 16-byte aligned");
  }
  if (!aligned16(w->embed) || !aligned16(w->lm_head) || !aligned16(w->final_norm))
    return fail(VD_ERR_INVALID_ARG, "weights must be 16-byte aligned");

  vd_model* m = new vd_model();
  m->cfg = c;
  cudaGetDevice(&m->device);
  m->embed = static_cast<const __nv_bfloat16*>(w->embed);
  m->final_norm = static_cast<const __nv_bfloat16*>(w->final_norm);
  m->lm_head = static_cast<const __nv_bfloat16*>(w->lm_head);
  m->layers.assign(w->layers, w->layers + c.n_layers);
  m->G = c.n_heads / c.n_kv_heads;
  if (c.embed_scale)  // the scale itself rounded to bf16, as a bf16 model multiplies by it
    m->embed_scale = __bfloat162float(__float2bfloat16_rn(static_cast<float>(sqrt(static_cast<double>(c.d_model)))));
  m->gain_offset = c.norm_offset ? 1.0f : 0.0f;
  if (cudaDeviceGetAttribute(&m->n_sm, cudaDevAttrMultiProcessorCount, m->device) != cudaSuccess || m->n_sm <= 0)
    m->n_sm = 148;
  m->key_tile = attn_key_tile(c.head_dim);
  m->split = kSplitKeys;
  m->max_splits = (c.max_context - 1) / m->split + 1;
  const int d = c.d_model, hd = c.head_dim, F = c.ffn_dim, V = c.vocab;
  const int qkv_dim = (c.n_heads + 2 * c.n_kv_heads) * hd, attn_dim = c.n_heads * hd;
  int rc = VD_OK;
  auto bail = [&](int r) {
    vd_destroy_model(m);
    return r;
  };
  for (int i = 0; i < c.n_layers; ++i) {
    WeightMaps mp;
    const vd_layer_weights& L = m->layers[i];
    if ((rc = make_weight_maps(&mp, L.wqkv, qkv_dim, d, false))) return bail(rc);
    m->m_qkv.push_back(mp);
    if ((rc = make_weight_maps(&mp, L.wo, d, attn_dim, false))) return bail(rc);
    m->m_o.push_back(mp);
    if ((rc = make_weight_maps(&mp, L.w_gate_up, 2 * static_cast<uint64_t>(F), d, true))) return bail(rc);
    m->m_gu.push_back(mp);
    if ((rc = make_weight_maps(&mp, L.w_down, d, F, false))) return bail(rc);
    m->m_down.push_back(mp);
  }
  if ((rc = make_weight_maps(&m->m_lm, w->lm_head, V, d, false))) return bail(rc);
  const int TM = c.max_tokens;
  if ((rc = make_act(m, m->a, TM, d))) return bail(rc);
  if ((rc = make_act(m, m->o, TM, attn_dim))) return bail(rc);
  if ((rc = make_act(m, m->z, TM, F))) return bail(rc);
  if ((rc = make_act(m, m->ar, c.max_logit_rows, d))) return bail(rc);
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(&m->x), static_cast<size_t>(TM) * d * 2))) return bail(rc);
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(&m->qkv), static_cast<size_t>(TM) * qkv_dim * 2))) return bail(rc);
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(&m->q), static_cast<size_t>(TM) * attn_dim * 2))) return bail(rc);
  if (c.sandwich_norm &&
      (rc = dev_alloc(m, reinterpret_cast<void**>(&m->hsub), static_cast<size_t>(TM) * d * 2)))
    return bail(rc);
  const size_t np = static_cast<size_t>(TM) * c.n_heads * m->max_splits;
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(&m->part_o), np * hd * 4))) return bail(rc);
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(&m->part_ml), np * 2 * 4))) return bail(rc);
  if ((rc = rope_table(m, c.rope_theta, hd, &m->cos_g, &m->sin_g))) return bail(rc);
  if ((rc = rope_table(m, c.rope_theta_local, hd, &m->cos_l, &m->sin_l))) return bail(rc);
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(&m->status), 256))) return bail(rc);
  const int max_pages = (c.max_context + 15) / 16;
  m->desc_cap = 4 * static_cast<size_t>(TM) + 6 * static_cast<size_t>(c.max_seqs) + 8 +
                static_cast<size_t>(c.max_seqs) * max_pages + c.max_logit_rows;
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(&m->d_desc), m->desc_cap * 4))) return bail(rc);
  for (int k = 0; k < 2; ++k) {
    if (cudaMallocHost(reinterpret_cast<void**>(&m->h_desc[k]), m->desc_cap * 4) != cudaSuccess ||
        cudaEventCreateWithFlags(&m->desc_ev[k], cudaEventDisableTiming) != cudaSuccess)
      return bail(fail(VD_ERR_CUDA, "pinned descriptor buffer"));
  }
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(&m->d_samp), sizeof(vd_sampler) * c.max_logit_rows))) return bail(rc);
  const size_t nsp = static_cast<size_t>(c.max_logit_rows) * sample_chunks(c.vocab);
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(&m->samp_part_v), nsp * 4))) return bail(rc);
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(&m->samp_part_i), nsp * 4))) return bail(rc);
  const size_t nfp = static_cast<size_t>(c.max_logit_rows) * (c.vocab / 32);
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(&m->fused_part_v), nfp * 4))) return bail(rc);
  if ((rc = dev_alloc(m, reinterpret_cast<void**>(&m->fused_part_i), nfp * 4))) return bail(rc);
  if (cudaMallocHost(reinterpret_cast<void**>(&m->h_samp), sizeof(vd_sampler) * c.max_logit_rows) != cudaSuccess ||
      cudaEventCreateWithFlags(&m->samp_ev, cudaEventDisableTiming) != cudaSuccess)
    return bail(fail(VD_ERR_CUDA, "pinned sampler buffer"));
  VD_CUDA_TRY(cudaDeviceSynchronize());
  int shapes_ok = 0;
  if ((rc = gemm_shapes_self_check(&shapes_ok))) return bail(rc);
  *out = m;
  return VD_OK;
}

void vd_destroy_model(vd_model* m) {
  if (!m) return;
  cudaDeviceSynchronize();
  drop_graphs(m);
  if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
  for (void* p : m->dev_allocs) cudaFree(p);
  for (int k = 0; k < 2; ++k) {
    if (m->h_desc[k]) cudaFreeHost(m->h_desc[k]);
    if (m->desc_ev[k]) cudaEventDestroy(m->desc_ev[k]);
  }
  if (m->h_samp) cudaFreeHost(m->h_samp);
  if (m->samp_ev) cudaEventDestroy(m->samp_ev);
  for (auto& r : m->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : m->ev_pool) cudaEventDestroy(e);
  delete m;
}

size_t vd_kv_pool_bytes(const vd_model* m, int32_t num_pages) {
  if (!m || num_pages < 0) return 0;
  const vd_model_config& c = m->cfg;
  return static_cast<size_t>(c.n_layers) * num_pages * 2 * c.n_kv_heads * 16 * c.head_dim * 2;
}

int vd_kv_pool_alloc(vd_model* m, int32_t num_pages, void* dev_mem, size_t bytes, vd_kv_pool** out) {
  if (check_model(m) || !out) return fail(VD_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  if (num_pages < 1) return fail(VD_ERR_INVALID_ARG, "num_pages must be >= 1");
  const size_t need = vd_kv_pool_bytes(m, num_pages);
  const vd_model_config& c = m->cfg;
  const long long rows = static_cast<long long>(c.n_layers) * num_pages * 2 * c.n_kv_heads * 16;
  if (rows + 16 > 0x7fffffffLL) return fail(VD_ERR_CAPACITY, "pool too large for 32-bit TMA row coordinates");
  static std::atomic<unsigned long long> next_id{1};
  vd_kv_pool* p = new vd_kv_pool();
  p->m = m;
  p->id = next_id++;
  p->num_pages = num_pages;
  p->rows = rows;
  if (dev_mem) {
    if (bytes < need) {
      delete p;
      return fail(VD_ERR_CAPACITY, "dev_mem smaller than vd_kv_pool_bytes()");
    }
    if (reinterpret_cast<uintptr_t>(dev_mem) & 255) {
      delete p;
      return fail(VD_ERR_INVALID_ARG, "dev_mem must be 256-byte aligned");
    }
    p->data = dev_mem;
  } else {
    if (cudaMalloc(&p->data, need) != cudaSuccess) {
      delete p;
      return fail(VD_ERR_CUDA, "cudaMalloc(pool) failed");
    }
    p->owned = true;
  }
  if (cudaMemset(p->data, 0, need) != cudaSuccess) {
    vd_destroy_kv_pool(p);
    return fail(VD_ERR_CUDA, "cudaMemset(pool) failed");
  }
  int rc = make_map_kv(&p->map, p->data, static_cast<uint64_t>(rows), c.head_dim, c.head_dim / 64);
  if (!rc) rc = make_map_kv(&p->map_tc, p->data, static_cast<uint64_t>(rows), c.head_dim, 1);
  if (rc) {
    vd_destroy_kv_pool(p);
    return rc;
  }
  cudaDeviceSynchronize();
  *out = p;
  return VD_OK;
}

void vd_destroy_kv_pool(vd_kv_pool* p) {
  if (!p) return;
  if (p->owned && p->data) {
    cudaDeviceSynchronize();
    cudaFree(p->data);
  }
  delete p;
}

void* vd_kv_pool_data(vd_kv_pool* p) { return p ? p->data : nullptr; }

int vd_step(vd_model* m, vd_kv_pool* pool, const vd_batch* b, float* logits_out, void* stream) {
  if (check_model(m) || !pool || pool->m != m) return fail(VD_ERR_INVALID_ARG, "null or foreign model/pool");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (b && b->num_logit_rows > 0 && !logits_out) return fail(VD_ERR_INVALID_ARG, "null logits_out");
  const bool graph = m->graph_max > 0 && !m->profiling;
  Desc d;
  int rc = upload_desc(m, pool, b, true, d, s, graph);
  if (rc || d.T == 0) return rc;
  return graph ? replay_step(m, pool, d, logits_out, nullptr, s) : enqueue_step(m, pool, d, logits_out, nullptr, s);
}

namespace {
int step_sample_impl(vd_model* m, vd_kv_pool* pool, const vd_batch* b, const int32_t* feed_index,
                     const int32_t* feed_tokens, const vd_sampler* per_row, float* logits_out, int32_t* tokens_out,
                     void* stream) {
  if (check_model(m) || !pool || pool->m != m) return fail(VD_ERR_INVALID_ARG, "null or foreign model/pool");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int R = b ? b->num_logit_rows : 0;
  if (R > 0 && (!per_row || !tokens_out)) return fail(VD_ERR_INVALID_ARG, "null per_row or tokens_out");
  if (R > m->cfg.max_logit_rows) return fail(VD_ERR_CAPACITY, "step exceeds max_logit_rows");
  if (feed_index && !feed_tokens && b)
    for (int t = 0; t < b->num_tokens; ++t)
      if (feed_index[t] >= 0) return fail(VD_ERR_INVALID_ARG, "feed_index without feed_tokens");
  const bool graph = m->graph_max > 0 && !m->profiling;
  Desc d;
  int rc = upload_desc(m, pool, b, true, d, s, graph, feed_index);
  if (rc || d.T == 0) return rc;
  d.feed = feed_index ? feed_tokens : nullptr;
  if (d.R > 0) {
    VD_CUDA_TRY(cudaEventSynchronize(m->samp_ev));  // the staging buffer's previous copy is done
    memcpy(m->h_samp, per_row, sizeof(vd_sampler) * d.R);
    VD_CUDA_TRY(cudaMemcpyAsync(m->d_samp, m->h_samp, sizeof(vd_sampler) * d.R, cudaMemcpyHostToDevice, s));
    VD_CUDA_TRY(cudaEventRecord(m->samp_ev, s));
  }
  int* tok = d.R > 0 ? tokens_out : nullptr;
  return graph ? replay_step(m, pool, d, logits_out, tok, s) : enqueue_step(m, pool, d, logits_out, tok, s);
}
}  // namespace

int vd_step_sample(vd_model* m, vd_kv_pool* pool, const vd_batch* b, const vd_sampler* per_row, float* logits_out,
                   int32_t* tokens_out, void* stream) {
  return step_sample_impl(m, pool, b, nullptr, nullptr, per_row, logits_out, tokens_out, stream);
}

int vd_step_sample_fed(vd_model* m, vd_kv_pool* pool, const vd_batch* b, const int32_t* feed_index,
                       const int32_t* feed_tokens, const vd_sampler* per_row, float* logits_out, int32_t* tokens_out,
                       void* stream) {
  if (!feed_index) return fail(VD_ERR_INVALID_ARG, "null feed_index");
  return step_sample_impl(m, pool, b, feed_index, feed_tokens, per_row, logits_out, tokens_out, stream);
}

int vd_set_reduction_mode(vd_model* m, int32_t mode) {
  if (check_model(m)) return VD_ERR_INVALID_ARG;
  if (mode != 0 && mode != 1) return fail(VD_ERR_INVALID_ARG, "mode must be 0 (invariant) or 1 (fast)");
  if (mode == 1 && !m->splitk_part) {  // partial sums of the largest split GEMM at kFastMaxTokens
    const vd_model_config& c = m->cfg;
    const int T = std::min(kFastMaxTokens, c.max_tokens), dm = c.d_model, F = c.ffn_dim;
    const int qkv_dim = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
    m->fast = 1;
    size_t cap = 0;
    cap = std::max(cap, static_cast<size_t>(fast_splits(m, T, qkv_dim / kGemmBM, dm)) * T * qkv_dim);
    cap = std::max(cap, static_cast<size_t>(fast_splits(m, T, dm / kGemmBM, c.n_heads * c.head_dim)) * T * dm);
    cap = std::max(cap, static_cast<size_t>(fast_splits(m, T, F / 64, dm)) * T * 2 * F);
    cap = std::max(cap, static_cast<size_t>(fast_splits(m, T, dm / kGemmBM, F)) * T * dm);
    m->fast = 0;
    int rc;
    if ((rc = dev_alloc(m, reinterpret_cast<void**>(&m->splitk_part), cap * 4))) return rc;
    m->splitk_cap = cap;
  }
  m->fast = mode;
  return VD_OK;
}

int vd_set_attention_fold(vd_model* m, int32_t mode) {
  if (check_model(m)) return VD_ERR_INVALID_ARG;
  if (mode < 0 || mode > 2) return fail(VD_ERR_INVALID_ARG, "mode must be 0 (auto), 1 (always) or 2 (never)");
  m->fold_mode = mode;
  return VD_OK;
}

int vd_set_attention_prefill(vd_model* m, int32_t kernel) {
  if (check_model(m)) return VD_ERR_INVALID_ARG;
  if (kernel < 0 || kernel > 1) return fail(VD_ERR_INVALID_ARG, "kernel must be 0 (tcgen05 where supported) or 1 (mma.sync)");
  m->prefill_kernel = kernel;
  return VD_OK;
}

int vd_set_graph_mode(vd_model* m, int32_t max_graphs) {
  if (check_model(m)) return VD_ERR_INVALID_ARG;
  if (max_graphs < 0) return fail(VD_ERR_INVALID_ARG, "max_graphs must be >= 0");
  m->graph_max = max_graphs;
  while (static_cast<int>(m->graphs.size()) > max_graphs) {
    if (m->graphs.front().exec) cudaGraphExecDestroy(m->graphs.front().exec);
    m->graphs.erase(m->graphs.begin());
  }
  return VD_OK;
}

int vd_graph_stats(const vd_model* m, int64_t* out4) {
  if (check_model(m) || !out4) return fail(VD_ERR_INVALID_ARG, "null argument");
  out4[0] = m->graph_captures;
  out4[1] = m->graph_replays;
  int64_t cached = 0;
  for (const GraphEntry& e : m->graphs) cached += e.exec != nullptr;
  out4[2] = cached;
  out4[3] = m->graph_eager;
  return VD_OK;
}

int vd_sample(vd_model* m, const float* logits, int32_t R, const vd_sampler* per_row, int32_t* tokens_out,
              void* stream) {
  if (check_model(m)) return VD_ERR_INVALID_ARG;
  if (R < 0 || R > m->cfg.max_logit_rows) return fail(VD_ERR_CAPACITY, "R exceeds max_logit_rows");
  if (R == 0) return VD_OK;
  if (!logits || !per_row || !tokens_out) return fail(VD_ERR_INVALID_ARG, "null argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  VD_CUDA_TRY(cudaEventSynchronize(m->samp_ev));
  memcpy(m->h_samp, per_row, sizeof(vd_sampler) * R);
  VD_CUDA_TRY(cudaMemcpyAsync(m->d_samp, m->h_samp, sizeof(vd_sampler) * R, cudaMemcpyHostToDevice, s));
  VD_CUDA_TRY(cudaEventRecord(m->samp_ev, s));
  if (reinterpret_cast<uintptr_t>(logits) & 15) return fail(VD_ERR_INVALID_ARG, "logits must be 16-byte aligned");
  Prof p(m, K_SAMPLE, s);
  p.kernels = 2;
  return launch_sample(logits, R, m->cfg.vocab, m->d_samp, m->samp_part_v, m->samp_part_i, tokens_out, s);
}

int vd_copy_kv(vd_model* m, vd_kv_pool* pool, int32_t layer, const int32_t* page_table, int32_t n_tokens,
               void* out_k, void* out_v, void* stream) {
  if (check_model(m) || !pool || pool->m != m) return fail(VD_ERR_INVALID_ARG, "null or foreign model/pool");
  const vd_model_config& c = m->cfg;
  if (layer < 0 || layer >= c.n_layers) return fail(VD_ERR_OUT_OF_RANGE, "layer out of range");
  if (n_tokens < 0) return fail(VD_ERR_INVALID_ARG, "negative n_tokens");
  if (n_tokens == 0) return VD_OK;
  if (!page_table || !out_k || !out_v) return fail(VD_ERR_INVALID_ARG, "null argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int np = (n_tokens + 15) / 16;
  for (int i = 0; i < np; ++i)
    if (page_table[i] < 0 || page_table[i] >= pool->num_pages) return fail(VD_ERR_OUT_OF_RANGE, "page id out of range");
  const size_t row = static_cast<size_t>(c.head_dim) * 2;
  const __nv_bfloat16* base = static_cast<const __nv_bfloat16*>(pool->data) +
                              static_cast<size_t>(layer) * pool->num_pages * 2 * c.n_kv_heads * 16 * c.head_dim;
  // one strided copy per (page, K/V): 16 slots x Hkv heads -> [pos][head][hd]
  for (int i = 0; i < np; ++i) {
    const int nt = std::min(16, n_tokens - i * 16);
    for (int kv = 0; kv < 2; ++kv) {
      const __nv_bfloat16* src = base + (static_cast<size_t>(page_table[i]) * 2 + kv) * c.n_kv_heads * 16 * c.head_dim;
      char* dst = static_cast<char*>(kv ? out_v : out_k) + static_cast<size_t>(i) * 16 * c.n_kv_heads * row;
      for (int h = 0; h < c.n_kv_heads; ++h)
        VD_CUDA_TRY(cudaMemcpy2DAsync(dst + h * row, c.n_kv_heads * row, src + static_cast<size_t>(h) * 16 * c.head_dim,
                                      row, row, nt, cudaMemcpyDeviceToDevice, s));
    }
  }
  return VD_OK;
}

int vd_device_status(vd_model* m) {
  if (check_model(m)) return VD_ERR_INVALID_ARG;
  int v = 0;
  VD_CUDA_TRY(cudaDeviceSynchronize());
  VD_CUDA_TRY(cudaMemcpy(&v, m->status, 4, cudaMemcpyDeviceToHost));
  VD_CUDA_TRY(cudaMemset(m->status, 0, 4));
  if (v == VD_ERR_OUT_OF_RANGE) return fail(VD_ERR_OUT_OF_RANGE, "a token read on the device was outside the vocabulary");
  if (v) return fail(VD_ERR_TIMEOUT, "a bounded on-device wait gave up");
  return VD_OK;
}

int vd_profile_enable(vd_model* m, int32_t on) {
  if (check_model(m)) return VD_ERR_INVALID_ARG;
  m->profiling = on != 0;
  return VD_OK;
}

int vd_profile_collect(vd_model* m, vd_kernel_stat* out, int32_t max_out) {
  if (check_model(m)) return VD_ERR_INVALID_ARG;
  for (auto& r : m->recs) {
    VD_CUDA_TRY(cudaEventSynchronize(r.b));
    float ms = 0.f;
    cudaEventElapsedTime(&ms, r.a, r.b);
    m->prof_ms[r.cls] += ms;
    m->prof_n[r.cls] += 1;
    m->prof_k[r.cls] += r.kernels;
    m->ev_pool.push_back(r.a);
    m->ev_pool.push_back(r.b);
  }
  m->recs.clear();
  int n = 0;
  for (int k = 0; k < K_COUNT && n < max_out; ++k) {
    if (!m->prof_n[k]) continue;
    if (out) {
      memset(&out[n], 0, sizeof(vd_kernel_stat));
      strncpy(out[n].name, kKernelNames[k], sizeof(out[n].name) - 1);
      out[n].launches = m->prof_n[k];
      out[n].kernels = m->prof_k[k];
      out[n].total_ms = m->prof_ms[k];
    }
    ++n;
  }
  for (int k = 0; k < K_COUNT; ++k) {
    m->prof_ms[k] = 0;
    m->prof_n[k] = 0;
    m->prof_k[k] = 0;
  }
  return n;
}

// ---------------------------------------------------------------- single ops
int vd_op_gemm(const void* A, const void* W, void* C, int32_t T, int32_t N, int32_t K, int32_t epilogue,
               const void* residual, void* stream) {
  if (!A || !W || !C) return fail(VD_ERR_INVALID_ARG, "null pointer");
  if (T < 1 || N < 1 || K < 1) return fail(VD_ERR_INVALID_ARG, "non-positive size");
  const bool glu = epilogue == VD_EPI_SWIGLU || epilogue == VD_EPI_GEGLU;
  if (epilogue < 0 || epilogue > VD_EPI_GEGLU) return fail(VD_ERR_INVALID_ARG, "unknown epilogue");
  if (K % kGemmBK || (glu ? N % 64 : N % kGemmBM)) return fail(VD_ERR_UNSUPPORTED, "N or K not a multiple of the tile");
  if (epilogue == VD_EPI_RESIDUAL && !residual) return fail(VD_ERR_INVALID_ARG, "residual required");
  if (!aligned16(A) || !aligned16(W) || !aligned16(C) || (residual && !aligned16(residual)))
    return fail(VD_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  WeightMaps wm;
  std::array<CUtensorMap, kNumBn> xm;
  int rc;
  if ((rc = make_weight_maps(&wm, W, glu ? 2 * static_cast<uint64_t>(N) : N, K, glu))) return rc;
  for (int i = 0; i < kNumBn; ++i)
    if ((rc = make_map_2d(&xm[i], A, T, K, std::min<int>(T, 16 << i)))) return rc;
  ActMaps xv;
  xv.maps = xm.data();
  xv.rows = T;
  GemmArgs g{};
  g.out = C;
  g.residual = residual;
  g.T = T;
  g.K = K;
  g.ldo = N;
  g.glu_up_row = N;
  g.status = op_status();
  return launch_gemm(wm, xv, g, epilogue, static_cast<cudaStream_t>(stream));
}

int vd_gemm_shape_check(void) {
  int dev = 0, r = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (gemm_shapes_self_check(&r) != VD_OK) return -1;
  return r;
}

int vd_gemm_plan_query(int32_t T, int32_t N, int32_t K, int32_t epilogue, int32_t out[3]) {
  if (!out) return fail(VD_ERR_INVALID_ARG, "null pointer");
  if (T < 1 || N < 1 || K < 1 || K % kGemmBK) return fail(VD_ERR_INVALID_ARG, "sizes");
  if (epilogue < 0 || epilogue > EPI_F32_SAMPLE) return fail(VD_ERR_INVALID_ARG, "unknown epilogue");
  const bool glu = epilogue == EPI_SWIGLU || epilogue == EPI_GEGLU;
  WeightMaps w;  // shapes only: no map is encoded
  w.rows = glu ? 2 * N : N;
  w.K = K;
  w.glu = glu;
  const GemmPlan p = gemm_plan(w, T, epilogue, 1);
  out[0] = p.bm;
  out[1] = p.bn;
  out[2] = p.kpo;
  return VD_OK;
}

int vd_set_gemm_plan(int32_t bm, int32_t bn, int32_t kpo) {
  GemmPlan p;
  p.bm = bm;
  p.bn = bn;
  p.kpo = kpo;
  return set_forced_gemm_plan(p);
}

int vd_op_rmsnorm(const void* x, const void* w, void* y, int32_t rows, int32_t d, float eps, void* stream) {
  if (!x || !w || !y) return fail(VD_ERR_INVALID_ARG, "null pointer");
  if (rows < 0 || d < 8 || d % 8) return fail(VD_ERR_INVALID_ARG, "d must be a positive multiple of 8");
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return fail(VD_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  return launch_rmsnorm(x, nullptr, w, y, rows, d, eps, 0.f, static_cast<cudaStream_t>(stream));
}

int vd_op_attention(vd_model* m, vd_kv_pool* p, int32_t layer, const vd_batch* b, const void* q, void* out,
                    void* stream) {
  if (check_model(m) || !p || p->m != m || !q || !out) return fail(VD_ERR_INVALID_ARG, "null argument");
  if (layer < 0 || layer >= m->cfg.n_layers) return fail(VD_ERR_OUT_OF_RANGE, "layer out of range");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Desc d;
  int rc = upload_desc(m, p, b, false, d, s);
  if (rc || d.T == 0) return rc;
  return run_attention(m, p, layer, d, static_cast<const __nv_bfloat16*>(q), static_cast<__nv_bfloat16*>(out), s);
}

int vd_op_attention_static(vd_model* m, vd_kv_pool* p, int32_t layer, const vd_batch* b, const void* q,
                           void* out, void* stream) {
  if (check_model(m) || !p || p->m != m || !q || !out) return fail(VD_ERR_INVALID_ARG, "null argument");
  if (layer < 0 || layer >= m->cfg.n_layers) return fail(VD_ERR_OUT_OF_RANGE, "layer out of range");
  // The descriptor is validated (and uploaded) exactly as vd_op_attention
  // does it, so both entries give the same error for the same batch; only
  // then is the scratch the call needs checked against the array.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Desc d;
  int rc = upload_desc(m, p, b, false, d, s);
  if (rc || d.T == 0) return rc;
  // Splits per row stride: the largest split count of any request of the call.
  int splits = 1;
  for (int i = 0; i < b->num_seqs; ++i) {
    const long long kv = static_cast<long long>(b->cached_len[i]) + b->cu_q[i + 1] - b->cu_q[i];
    splits = std::max(splits, static_cast<int>((kv - 1) / m->split + 1));
  }
  const size_t rows = static_cast<size_t>(b->num_tokens) * m->cfg.n_heads * splits;
  const size_t need = rows * (m->cfg.head_dim + 2) * sizeof(float);
  if (need > kAttnStaticScratchBytes)
    return fail(VD_ERR_CAPACITY, "call needs " + std::to_string(need) + " bytes of split scratch; the static buffer holds " +
                                     std::to_string(kAttnStaticScratchBytes) + " (fewer tokens or shorter contexts per call)");
  void* scratch = nullptr;
  if ((rc = attn_static_scratch(&scratch))) return rc;
  float* part_o = static_cast<float*>(scratch);
  float* part_ml = part_o + rows * m->cfg.head_dim;
  return run_attention_static(m, p, layer, d, static_cast<const __nv_bfloat16*>(q),
                              static_cast<__nv_bfloat16*>(out), part_o, part_ml, splits, s);
}

int vd_op_rope_kv(vd_model* m, vd_kv_pool* p, int32_t layer, const vd_batch* b, const void* qkv, void* q_out,
                  void* stream) {
  if (check_model(m) || !p || p->m != m || !qkv || !q_out) return fail(VD_ERR_INVALID_ARG, "null argument");
  if (layer < 0 || layer >= m->cfg.n_layers) return fail(VD_ERR_OUT_OF_RANGE, "layer out of range");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Desc d;
  int rc = upload_desc(m, p, b, false, d, s);
  if (rc || d.T == 0) return rc;
  return run_rope(m, p, layer, d, static_cast<const __nv_bfloat16*>(qkv), static_cast<__nv_bfloat16*>(q_out), s);
}

int vd_op_tma_stream(const void* w, int64_t rows, int64_t K, const void* x, int64_t x_rows, int32_t box_rows,
                     int32_t kpo, int32_t x_box_rows, int32_t k_parts, int32_t ctas, void* stream) {
  if (!w || (x_box_rows > 0 && !x)) return fail(VD_ERR_INVALID_ARG, "null pointer");
  if (rows < 1 || K < kGemmBK || K % kGemmBK || rows > (1ll << 31) || K > (1ll << 31))
    return fail(VD_ERR_INVALID_ARG, "rows >= 1, K a positive multiple of 64");
  if ((box_rows != 64 && box_rows != 128 && box_rows != 256) || rows % box_rows)
    return fail(VD_ERR_INVALID_ARG, "box_rows in {64, 128, 256}, dividing rows");
  if ((kpo != 1 && kpo != 2 && kpo != 4) || (K / kGemmBK) % kpo || (box_rows == 256 && kpo != 1))
    return fail(VD_ERR_INVALID_ARG, "kpo in {1, 2, 4} dividing the K blocks (1 for 256-row boxes)");
  if (x_box_rows < 0 || x_box_rows > kGemmBN || (x_box_rows > 0 && (x_rows < x_box_rows)))
    return fail(VD_ERR_INVALID_ARG, "x_box_rows in [0, 256] and at most x_rows");
  if (ctas < 0) return fail(VD_ERR_INVALID_ARG, "ctas >= 0");
  if (k_parts < 1 || (K / kGemmBK) % (static_cast<int64_t>(kpo) * k_parts))
    return fail(VD_ERR_INVALID_ARG, "k_parts >= 1 with kpo * k_parts dividing the K blocks");
  if (!aligned16(w) || (x_box_rows > 0 && !aligned16(x))) return fail(VD_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  WeightMaps wm;
  int rc;
  if ((rc = make_weight_maps(&wm, w, static_cast<uint64_t>(rows), static_cast<uint64_t>(K), false))) return rc;
  CUtensorMap xm{};
  if (x_box_rows > 0 && (rc = make_map_2d(&xm, x, x_rows, K, x_box_rows))) return rc;
  const int ki = kpo == 1 ? 0 : kpo == 2 ? 1 : 2;
  const CUtensorMap& m = wm.m[box_rows == 128 ? 0 : box_rows == 64 ? 1 : 2][ki];
  return launch_tma_stream(m, xm, static_cast<int>(rows), static_cast<int>(K), box_rows, kpo, x_box_rows, k_parts,
                           ctas, op_status(), static_cast<cudaStream_t>(stream));
}

int vd_op_mma_issue_probe(int32_t M, int32_t N, int32_t n_mma, int32_t wait, int64_t* out, void* stream) {
  if (!out || (reinterpret_cast<uintptr_t>(out) & 7)) return fail(VD_ERR_INVALID_ARG, "out: 8-byte aligned dev int64 [2]");
  if ((M != 64 && M != 128) || N < 16 || N > 256 || N % 16 || n_mma < 16 || n_mma > 65536 || n_mma % 16 ||
      wait < 0 || wait > 3)
    return fail(VD_ERR_INVALID_ARG, "M in {64, 128}; N a multiple of 16 in [16, 256]; n_mma a multiple of 16 in "
                                    "[16, 65536]; wait in {0, 1, 2, 3}");
  return launch_mma_issue_probe(M, N, n_mma, wait, reinterpret_cast<long long*>(out), op_status(),
                                static_cast<cudaStream_t>(stream));
}

int vd_op_wait_probe(vd_model* m, int32_t limit_us, int32_t* out, void* stream) {
  if (check_model(m)) return fail(VD_ERR_INVALID_ARG, "null model");
  if (limit_us < 1 || limit_us > 2000000) return fail(VD_ERR_INVALID_ARG, "limit_us must be in [1, 2000000]");
  if (out && !aligned16(out)) return fail(VD_ERR_INVALID_ARG, "out must be 16-byte aligned");
  return launch_wait_probe(m->status, static_cast<uint64_t>(limit_us) * 1000u, out, static_cast<cudaStream_t>(stream));
}

int vd_op_philox(uint64_t seed, uint64_t step, int32_t n, uint32_t* out, void* stream) {
  if (n < 0) return fail(VD_ERR_INVALID_ARG, "negative n");
  if (n > 0 && !out) return fail(VD_ERR_INVALID_ARG, "null out");
  return launch_philox(seed, step, n, out, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
