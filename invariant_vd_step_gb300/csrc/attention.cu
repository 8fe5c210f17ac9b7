// Unified prefill/decode paged attention with a fixed KV split size.
//
// Rows.  For request b and KV head g the rows are (token i, query head of
// the group) pairs, token-major.  A CTA owns a block of rows of one
// (request, KV head) and one KV split.  Decode-shaped requests (q_len *
// Hq/Hkv <= 16, one block of 16 rows) run with two warps that share the rows
// and split the head dimension of the P V product; longer chunks run four
// warps of 16 rows each, sharing every K/V tile.  A decode launch of at most
// one CTA per SM (small batches) runs the scores-first CTA instead (head
// dims 64 and 128; see attn_sf_kernel), whose warps score the split's tiles
// first and then fold P V in rounds.  Each value goes through the same step
// functions in the same order per row in every variant (the `tile_*` steps
// that `attn_tile` strings together), so a row's result does not depend on
// which of them ran it.
//
// Traversal (深入解析 Vosti §六 6.2, causal prefix equivalence and the
// sliding-window traversal; "Deterministic and bit-exact inference",
// technical section: fixed split *size*).  Keys are cut into splits of
// S_kv keys and tiles of B_N keys, both aligned to absolute key positions.
// A row at position p with window lower bound lo = max(0, p-w+1) (lo = 0 for
// global layers) sees keys [lo, p].  Inside one split it folds the tiles
// that intersect [lo, p] in ascending order into an online-softmax state
// (m, l, o); tiles of the CTA's range that hold no visible key for the row
// leave its state bit-for-bit unchanged (the masking rules of §六 6.2: a
// masked score is -inf, its weight exactly 0, and a fully masked row keeps
// its incoming state).  Split partials go to the workspace; the merge
// kernel folds the splits of each row left to right, always in the same
// order, with one merge routine, then normalises.  The tile size, split
// size and fold order depend only on the head dimension (fixed at model
// creation), never on the batch, q_len, page table or split placement.
//
// Numerics: S = Q K^T and O += P V on mma.sync m16n8k16 (bf16 in, fp32
// accumulate), scores scaled by log2(e)/sqrt(hd), exp2 by ex2.approx.ftz,
// P split into bf16 hi + lo terms for the P V product (fp32 for the row
// sum), every other float operation an explicitly rounded intrinsic.
#include <math.h>

#include "vd_device.cuh"
#include "vd_internal.h"

namespace vd {
namespace {

template <int HD>
struct AttnCfg {
  static constexpr int BNK = 32;                     // keys per tile
  static constexpr int PAGES = BNK / 16;             // 16-token pages per tile
  static constexpr int PAGE_BYTES = 16 * HD * 2;     // one page of one KV head
  static constexpr int TILE_BYTES = BNK * HD * 2;
  static constexpr int MAX_STAGES = 8;
  static constexpr int PIDS = 64;  // page ids a decode CTA stages: every page of its split
  static constexpr int STATIC_SMEM = PIDS * 4 + 16;
  // K + V tiles of `stages` pipeline stages, their barriers, the abort flag
  static constexpr int smem(int stages) { return 1024 + stages * 2 * TILE_BYTES + MAX_STAGES * 8 + 16; }
};

// Byte offset of (key, 16-byte chunk along hd) inside a K or V tile staged
// by the 3-D TMA box (64, hd/64, 16) with the 128-byte swizzle.
template <int HD>
__device__ __forceinline__ uint32_t kv_off(int key, int chunk) {
  const int pg = key >> 4, slot = key & 15;
  const int lr = slot * (HD / 64) + (chunk >> 3);
  return pg * AttnCfg<HD>::PAGE_BYTES + lr * 128 + (((chunk & 7) ^ (lr & 7)) << 4);
}

template <int ND>
struct RowState {
  float m[2], l[2];     // rows g and g+8 of the warp
  float o[ND / 8][4];   // mma C fragments of the ND output dims this warp owns
};

// The steps of one key tile for the 16 rows of a warp (rows g and g + 8 of
// lane (g, t4)).  `attn_tile` runs them back to back, one tile at a time;
// the scores-first decode kernel runs the same steps over a whole split in
// three phases.  Either way every row's values pass through the same
// operations in the same order.  LOWER8: rows 8..15 of the warp are known
// to hold no row (a decode CTA of at most 8 rows), so their masking,
// softmax and rescale are skipped: their weights are exactly 0 either way,
// and the other rows' instructions are unchanged.

// S = Q K^T of a 32-key tile: per 8-key block, HD/16 K = 16 steps from zero.
template <int HD, int BNK>
__device__ __forceinline__ void tile_scores(float (&s)[BNK / 8][4], const uint32_t (&qf)[HD / 16][4], uint32_t kbase,
                                            int lane) {
  const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
  for (int j = 0; j < BNK / 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
    for (int jp = 0; jp < BNK / 16; ++jp) {
      uint32_t b[4];
      ldmatrix_x4(b, kbase + kv_off<HD>(jp * 16 + (mi >> 1) * 8 + r8, kk * 2 + (mi & 1)));
      mma_bf16_16816(s[2 * jp], qf[kk], b);
      mma_bf16_16816(s[2 * jp + 1], qf[kk], b + 2);
    }
  }
}

// Scores to the log2 domain, -inf outside each row's keys [lo, pos]; the
// tile's maximum of rows g and g + 8 over the lane quad.
template <int BNK, bool LOWER8>
__device__ __forceinline__ void tile_mask_max(float (&s)[BNK / 8][4], float (&mx)[2], int key0, const int (&pos)[2],
                                              const int (&lo)[2], float scale_log2, int lane) {
  const int t4 = lane & 3;
  mx[0] = mx[1] = -INFINITY;
#pragma unroll
  for (int j = 0; j < BNK / 8; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = e >> 1;
      if (LOWER8 && r == 1) {
        s[j][e] = -INFINITY;
        continue;
      }
      const int key = key0 + j * 8 + t4 * 2 + (e & 1);
      const bool vis = key >= lo[r] && key <= pos[r];
      const float v = vis ? __fmul_rn(s[j][e], scale_log2) : -INFINITY;
      s[j][e] = v;
      mx[r] = fmaxf(mx[r], v);
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (LOWER8 && r == 1) continue;  // stays -inf: the row keeps its state
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
  }
}

// The running maximum after a tile with row maximum mx, the factor that
// rescales the state before it, and whether the row saw a key in it (a row
// that saw none keeps its state bit for bit: alpha = 1, m unchanged).
__device__ __forceinline__ void tile_running_max(float m, float mx, float& mnew, float& alpha, bool& rv) {
  rv = mx != -INFINITY;
  mnew = rv ? fmaxf(m, mx) : m;
  alpha = rv ? ex2(__fsub_rn(m, mnew)) : 1.0f;
}

// P = 2^(s - m_new) as the A fragments of the P V product, and the fp32 row
// sums over the quad.  P enters the product as two bf16 terms, hi = bf16(p)
// and lo = bf16(p - hi) (p - hi is exact in fp32), so the weights carry
// about 16 significant bits; the row sum uses the fp32 weights.
template <int BNK, bool LOWER8>
__device__ __forceinline__ void tile_probs(const float (&s)[BNK / 8][4], const float (&mnew)[2],
                                           uint32_t (&pa)[BNK / 16][4], uint32_t (&pl)[BNK / 16][4], float (&rs)[2]) {
  rs[0] = rs[1] = 0.f;
#pragma unroll
  for (int j = 0; j < BNK / 8; ++j) {
    float p[4], h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = e >> 1;
      if (LOWER8 && r == 1) {
        p[e] = h[e] = l[e] = 0.f;
        continue;
      }
      p[e] = (s[j][e] == -INFINITY) ? 0.f : ex2(__fsub_rn(s[j][e], mnew[r]));
      h[e] = bf16_round(p[e]);
      l[e] = __fsub_rn(p[e], h[e]);
    }
    rs[0] = __fadd_rn(__fadd_rn(rs[0], p[0]), p[1]);
    rs[1] = __fadd_rn(__fadd_rn(rs[1], p[2]), p[3]);
    pa[j >> 1][(j & 1) * 2 + 0] = pack_bf16x2(h[0], h[1]);
    pa[j >> 1][(j & 1) * 2 + 1] = pack_bf16x2(h[2], h[3]);
    pl[j >> 1][(j & 1) * 2 + 0] = pack_bf16x2(l[0], l[1]);
    pl[j >> 1][(j & 1) * 2 + 1] = pack_bf16x2(l[2], l[3]);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (LOWER8 && r == 1) continue;
    rs[r] = __fadd_rn(rs[r], __shfl_xor_sync(0xffffffffu, rs[r], 1));
    rs[r] = __fadd_rn(rs[r], __shfl_xor_sync(0xffffffffu, rs[r], 2));
  }
}

// l <- l alpha + (the tile's row sum) for a row that saw a key of the tile.
__device__ __forceinline__ void tile_update_l(float& l, float alpha, float rs, bool rv) {
  l = rv ? __fadd_rn(__fmul_rn(l, alpha), rs) : l;
}

// O <- O alpha (with LOWER8 rows 8..15 have alpha 1 and are never stored).
template <int ND, bool LOWER8>
__device__ __forceinline__ void tile_rescale(float (&o)[ND / 8][4], const float (&alpha)[2]) {
#pragma unroll
  for (int n = 0; n < ND / 8; ++n) {
    o[n][0] = __fmul_rn(o[n][0], alpha[0]);
    o[n][1] = __fmul_rn(o[n][1], alpha[0]);
    if (!LOWER8) {
      o[n][2] = __fmul_rn(o[n][2], alpha[1]);
      o[n][3] = __fmul_rn(o[n][3], alpha[1]);
    }
  }
}

// O += P_hi V, P_lo V over the tile's two 16-key steps, for the output dims
// [dim0, dim0 + ND); per 8-dim block the order is hi, lo, hi, lo.  Each V
// fragment is loaded right before its products (the tile-at-a-time order).
template <int HD, int BNK, int ND>
__device__ __forceinline__ void tile_pv(float (&o)[ND / 8][4], const uint32_t (&pa)[BNK / 16][4],
                                        const uint32_t (&pl)[BNK / 16][4], uint32_t vbase, int lane, int dim0) {
  const int mi = lane >> 3, r8 = lane & 7;
  const int np0 = dim0 / 16;
#pragma unroll
  for (int ks = 0; ks < BNK / 16; ++ks) {
#pragma unroll
    for (int np = 0; np < ND / 16; ++np) {
      uint32_t b[4];
      ldmatrix_x4_trans(b, vbase + kv_off<HD>(ks * 16 + (mi & 1) * 8 + r8, (np0 + np) * 2 + (mi >> 1)));
      mma_bf16_16816(o[2 * np], pa[ks], b);
      mma_bf16_16816(o[2 * np], pl[ks], b);
      mma_bf16_16816(o[2 * np + 1], pa[ks], b + 2);
      mma_bf16_16816(o[2 * np + 1], pl[ks], b + 2);
    }
  }
}

// The same products in two steps, so that a tile's V fragments can be
// loaded while the previous tile's products run: the fragments for the
// output dims [dim0, dim0 + ND) per 16-key step and 16-dim block ...
template <int HD, int BNK, int ND>
__device__ __forceinline__ void tile_v_frags(uint32_t (&vb)[BNK / 16][ND / 16][4], uint32_t vbase, int lane,
                                             int dim0) {
  const int mi = lane >> 3, r8 = lane & 7;
  const int np0 = dim0 / 16;
#pragma unroll
  for (int ks = 0; ks < BNK / 16; ++ks)
#pragma unroll
    for (int np = 0; np < ND / 16; ++np)
      ldmatrix_x4_trans(vb[ks][np], vbase + kv_off<HD>(ks * 16 + (mi & 1) * 8 + r8, (np0 + np) * 2 + (mi >> 1)));
}

// ... then the products, in tile_pv's order.
template <int BNK, int ND>
__device__ __forceinline__ void tile_pv_mma(float (&o)[ND / 8][4], const uint32_t (&pa)[BNK / 16][4],
                                            const uint32_t (&pl)[BNK / 16][4],
                                            const uint32_t (&vb)[BNK / 16][ND / 16][4]) {
#pragma unroll
  for (int ks = 0; ks < BNK / 16; ++ks) {
#pragma unroll
    for (int np = 0; np < ND / 16; ++np) {
      mma_bf16_16816(o[2 * np], pa[ks], vb[ks][np]);
      mma_bf16_16816(o[2 * np], pl[ks], vb[ks][np]);
      mma_bf16_16816(o[2 * np + 1], pa[ks], vb[ks][np] + 2);
      mma_bf16_16816(o[2 * np + 1], pl[ks], vb[ks][np] + 2);
    }
  }
}

// One key tile for the 16 rows of a warp, which accumulates output dims
// [dim0, dim0 + ND).  S and the softmax state are computed over the full
// head either way, so every output element gets the same instruction chain
// whether one warp owns all dims or several warps share them.
template <int HD, int BNK, int ND, bool LOWER8>
__device__ __forceinline__ void attn_tile(RowState<ND>& st, const uint32_t (&qf)[HD / 16][4], uint32_t kbase,
                                          uint32_t vbase, int key0, const int (&pos)[2], const int (&lo)[2],
                                          float scale_log2, int lane, int dim0) {
  float s[BNK / 8][4], mx[2], mnew[2], alpha[2], rs[2];
  bool rv[2];
  uint32_t pa[BNK / 16][4], pl[BNK / 16][4];
  tile_scores<HD, BNK>(s, qf, kbase, lane);
  tile_mask_max<BNK, LOWER8>(s, mx, key0, pos, lo, scale_log2, lane);
#pragma unroll
  for (int r = 0; r < 2; ++r) tile_running_max(st.m[r], mx[r], mnew[r], alpha[r], rv[r]);
  tile_probs<BNK, LOWER8>(s, mnew, pa, pl, rs);
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    tile_update_l(st.l[r], alpha[r], rs[r], rv[r]);
    st.m[r] = mnew[r];
  }
  tile_rescale<ND, LOWER8>(st.o, alpha);
  tile_pv<HD, BNK, ND>(st.o, pa, pl, vbase, lane, dim0);
}

// NW warps per CTA; groups of DS warps own the same 16 rows and split the
// head dimension between them (DS = 2 for decode-shaped CTAs, which have one
// row block only; DS = 1 for prefill CTAs).  PROD: one more warp issues the
// K/V copies, and each warp releases a stage on its own as soon as it is done
// with it, instead of all warps meeting at a barrier after every tile (a
// launch with one CTA per SM has no other CTA to hide that barrier and the
// copy issue behind).
template <int HD, int NW, int DS, bool FOLD, bool PROD = false>
__global__ void __launch_bounds__((NW + PROD) * 32)
    attn_kernel(const __grid_constant__ CUtensorMap kvmap, AttnArgs a) {
  using C = AttnCfg<HD>;
  constexpr int RB = 16 * NW / DS;  // rows per CTA
  constexpr int ND = HD / DS;       // output dims per warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int NS = a.stages;  // tiles in flight; changes when copies are issued, never the fold order
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * 2 * C::TILE_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + C::MAX_STAGES);
  __shared__ int pid_s[C::PIDS];
  __shared__ uint64_t empty_s[PROD ? C::MAX_STAGES : 1];  // PROD: the NW warps are done with a stage

  // Up to the wait for the previous kernel this CTA reads only the status
  // word and the step's description (sequence classes, lengths, page table),
  // written before the step's first kernel, so that those round trips hide
  // behind the wait; Q and the K/V pages are read after it.  Once any
  // bounded wait has given up, later CTAs skip their work (a failure of the
  // kernel right before this one is seen by the next kernel).
  {
    __shared__ int skip;  // one read for the whole CTA keeps the exit uniform
    if (threadIdx.x == 0) skip = a.status ? *reinterpret_cast<volatile int*>(a.status) : 0;
    __syncthreads();
    if (skip) return;
  }
  // ---- work item -> (request, row block, KV head, split)
  const int item = blockIdx.x;
  if (item >= a.cls_start[a.n_cls]) return;  // grid rounded up past the class's items
  int lo_i = 0, hi_i = a.n_cls - 1;
  while (lo_i < hi_i) {  // last j with cls_start[j] <= item
    const int mid = (lo_i + hi_i + 1) >> 1;
    if (a.cls_start[mid] <= item) lo_i = mid; else hi_i = mid - 1;
  }
  const int b = a.cls_seq[lo_i];
  int local = item - a.cls_start[lo_i];
  const int q0 = a.cu_q[b], qlen = a.cu_q[b + 1] - q0, cached = a.cached_len[b];
  const int kv_len = cached + qlen;
  const int G = a.Hq / a.Hkv;
  // Split mode: one CTA per split.  Fold mode: one CTA walks every split of
  // its rows (the same tiles, split by split) and folds the split states
  // itself, with the merge kernel's arithmetic and order.
  const int nsplit = FOLD ? 1 : (kv_len - 1) / a.split + 1;
  const int sidx = local % nsplit;
  local /= nsplit;
  const int kvh = local % a.Hkv;
  const int rb = local / a.Hkv;
  const int rows = qlen * G;
  const int r0 = rb * RB;
  const int r_end = min(rows, r0 + RB);
  const int p_min = cached + r0 / G, p_max = cached + (r_end - 1) / G;
  const int lo_min = a.window > 0 ? max(0, p_min - a.window + 1) : 0;
  const int key_lo = FOLD ? lo_min : max(sidx * a.split, lo_min);
  const int key_hi = FOLD ? p_max : min((sidx + 1) * a.split - 1, p_max);
  if (key_lo > key_hi) return;  // no visible key of these rows in this split
  const int tile_lo = key_lo / C::BNK;
  const int ntiles = key_hi / C::BNK - tile_lo + 1;
  // Decode-shaped split CTAs (few CTAs per SM, so each copy's issue latency
  // shows): the physical ids of the (at most PIDS) pages this CTA streams,
  // read by one warp in one round trip, so that the copies are issued
  // without a dependent page-table load each.  Fold CTAs walk the whole
  // context and prefill CTAs run several per SM: they look ids up as they go.
  constexpr bool kStagePids = DS > 1 && !FOLD;
  const int lp_first = (tile_lo * C::BNK) >> 4;
  if (kStagePids && threadIdx.x < 32)
    for (int j = threadIdx.x; j < C::PIDS; j += 32) {
      const int lp = lp_first + j;
      pid_s[j] = (j < ntiles * C::PAGES && lp * 16 < kv_len)
                     ? a.page_table[static_cast<size_t>(b) * a.pt_stride + lp] : -1;
    }

  if (threadIdx.x == 0) {
    for (int k = 0; k < NS; ++k) mbar_init(&full[k], 1);
    if constexpr (PROD)
      for (int k = 0; k < NS; ++k) mbar_init(&empty_s[k], NW);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  auto issue = [&](int it, int stg) {
    uint8_t* sk = smem + stg * 2 * C::TILE_BYTES;
    uint8_t* sv = sk + C::TILE_BYTES;
    mbar_arrive_expect_tx(&full[stg], 2 * C::TILE_BYTES);
    const int lp0 = ((tile_lo + it) * C::BNK) >> 4;
#pragma unroll
    for (int pg = 0; pg < C::PAGES; ++pg) {
      const int lp = lp0 + pg;
      int rk = a.pool_rows, rvw = a.pool_rows;  // outside the pool: zero fill
      if constexpr (kStagePids) {
        const int phys = pid_s[it * C::PAGES + pg];  // -1 past the context
        if (phys >= 0) {
          rk = a.layer_row0 + ((phys * 2) * a.Hkv + kvh) * 16;
          rvw = rk + a.Hkv * 16;
        }
      } else if (lp * 16 < kv_len) {
        const int phys = a.page_table[static_cast<size_t>(b) * a.pt_stride + lp];
        rk = a.layer_row0 + ((phys * 2) * a.Hkv + kvh) * 16;
        rvw = rk + a.Hkv * 16;
      }
      tma_load_3d(sk + pg * C::PAGE_BYTES, &kvmap, &full[stg], 0, 0, rk);
      tma_load_3d(sv + pg * C::PAGE_BYTES, &kvmap, &full[stg], 0, 0, rvw);
    }
  };
  int issued = 0;
  if (!PROD && threadIdx.x == 0) {
    issued = min(NS, ntiles);
    for (int k = 0; k < issued; ++k) issue(k, k);
  }

  // ---- this warp's rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if constexpr (PROD) {
    if (warp == NW) {  // the copy warp: a stage is refilled once every warp has released it
      if (lane == 0) {
        for (int g = 0; g < ntiles && !*abort_flag; ++g) {
          const int s = g % NS;
          if (g >= NS && !mbar_wait(&empty_s[s], ((g / NS) - 1) & 1, abort_flag, a.status)) break;
          issue(g, s);
          issued = g + 1;
        }
        // every copy lands before this warp leaves (the last use of each stage)
        for (int k = max(0, issued - NS); k < issued; ++k) drain_wait(&full[k % NS], (k / NS) & 1);
      }
      return;
    }
  }
  const int gq = lane >> 2, t4 = lane & 3;
  const int dim0 = (warp % DS) * ND;
  int pos[2], lo[2], tok[2], hq[2];
  bool valid[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = r0 + (warp / DS) * 16 + gq + 8 * r;
    valid[r] = row < rows;
    tok[r] = row / G;
    hq[r] = kvh * G + row % G;
    pos[r] = valid[r] ? cached + tok[r] : -1;
    lo[r] = valid[r] ? (a.window > 0 ? max(0, pos[r] - a.window + 1) : 0) : 1;
  }
  uint32_t qf[HD / 16][4];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const __nv_bfloat16* qr = a.q + (static_cast<size_t>(q0 + tok[r]) * a.Hq + hq[r]) * HD;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      qf[kk][r] = valid[r] ? *reinterpret_cast<const uint32_t*>(qr + kk * 16 + t4 * 2) : 0u;
      qf[kk][2 + r] = valid[r] ? *reinterpret_cast<const uint32_t*>(qr + kk * 16 + 8 + t4 * 2) : 0u;
    }
  }
  RowState<ND> st;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    st.m[r] = -INFINITY;
    st.l[r] = 0.f;
  }
#pragma unroll
  for (int n = 0; n < ND / 8; ++n) st.o[n][0] = st.o[n][1] = st.o[n][2] = st.o[n][3] = 0.f;

  // fold mode: the merged state of the splits seen so far (rows g, g+8)
  float fm[2] = {-INFINITY, -INFINITY}, fl[2] = {0.f, 0.f};
  float fo[FOLD ? ND / 8 : 1][4];
  if constexpr (FOLD) {
#pragma unroll
    for (int n = 0; n < ND / 8; ++n) fo[n][0] = fo[n][1] = fo[n][2] = fo[n][3] = 0.f;
  }
  // A decode CTA (one block of 16 rows) with at most 8 rows: its warps'
  // rows 8..15 are empty (the same for every warp, so the branch is uniform).
  const bool lower8 = DS > 1 && rows - r0 <= 8;
  bool ok = true;
  int it = 0, stg = 0;
  uint32_t ph = 0;  // tile it sits in stage it % NS, round it / NS
  for (; it < ntiles; ++it) {
    if constexpr (PROD) {  // the warp's lanes agree, then the warp leaves or goes on
      if (!__all_sync(0xffffffffu, mbar_wait(&full[stg], ph, abort_flag, a.status))) break;
    } else if (!mbar_wait(&full[stg], ph, abort_flag, a.status)) {
      ok = false;
    }
    const int key0 = (tile_lo + it) * C::BNK;
    bool mine = false;  // any row of this warp sees a key of this tile
#pragma unroll
    for (int r = 0; r < 2; ++r) mine |= max(lo[r], key0) <= min(pos[r], key0 + C::BNK - 1);
    mine = __any_sync(0xffffffffu, mine);
    if (ok && mine) {
      const uint32_t kb = smem_u32(smem + stg * 2 * C::TILE_BYTES);
      if (DS > 1 && lower8)
        attn_tile<HD, C::BNK, ND, DS != 1>(st, qf, kb, kb + C::TILE_BYTES, key0, pos, lo, a.scale_log2, lane, dim0);
      else
        attn_tile<HD, C::BNK, ND, false>(st, qf, kb, kb + C::TILE_BYTES, key0, pos, lo, a.scale_log2, lane, dim0);
    }
    if (FOLD && ((key0 + C::BNK) % a.split == 0 || it == ntiles - 1)) {
      // end of a split: fold it into the merged state of every row that saw a
      // key in it (merge order: splits left to right, the first one taken as is)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (st.m[r] != -INFINITY) {
          if (fm[r] == -INFINITY) {
            fm[r] = st.m[r];
            fl[r] = st.l[r];
#pragma unroll
            for (int n = 0; n < ND / 8; ++n) {
              fo[n][2 * r] = st.o[n][2 * r];
              fo[n][2 * r + 1] = st.o[n][2 * r + 1];
            }
          } else {
            const float mn = fmaxf(fm[r], st.m[r]);
            const float ca = ex2(__fsub_rn(fm[r], mn)), cb = ex2(__fsub_rn(st.m[r], mn));
            fl[r] = __fadd_rn(__fmul_rn(fl[r], ca), __fmul_rn(st.l[r], cb));
#pragma unroll
            for (int n = 0; n < ND / 8; ++n) {
              fo[n][2 * r] = __fadd_rn(__fmul_rn(fo[n][2 * r], ca), __fmul_rn(st.o[n][2 * r], cb));
              fo[n][2 * r + 1] = __fadd_rn(__fmul_rn(fo[n][2 * r + 1], ca), __fmul_rn(st.o[n][2 * r + 1], cb));
            }
            fm[r] = mn;
          }
        }
        st.m[r] = -INFINITY;
        st.l[r] = 0.f;
      }
#pragma unroll
      for (int n = 0; n < ND / 8; ++n) st.o[n][0] = st.o[n][1] = st.o[n][2] = st.o[n][3] = 0.f;
    }
    if constexpr (PROD) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_s[stg]);
    } else {
      if (__syncthreads_or(!ok)) break;
      if (threadIdx.x == 0 && it + NS < ntiles) {
        issue(it + NS, stg);
        issued = it + NS + 1;
      }
    }
    if (++stg == NS) {
      stg = 0;
      ph ^= 1u;
    }
  }
  if (it < ntiles) {  // gave up: let copies in flight land before leaving (PROD: the copy warp does)
    if (!PROD && threadIdx.x == 0)
      for (int k = it; k < issued; ++k) drain_wait(&full[k % NS], (k / NS) & 1);
    return;
  }

  if constexpr (FOLD) {  // o / l of every row -> bf16, as the merge kernel writes it
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (!valid[r] || fm[r] == -INFINITY) continue;
      __nv_bfloat16* out = a.out + (static_cast<size_t>(q0 + tok[r]) * a.Hq + hq[r]) * HD + dim0;
#pragma unroll
      for (int n = 0; n < ND / 8; ++n)
        *reinterpret_cast<uint32_t*>(out + n * 8 + t4 * 2) =
            pack_bf16x2(__fdiv_rn(fo[n][2 * r], fl[r]), __fdiv_rn(fo[n][2 * r + 1], fl[r]));
    }
    return;
  }
  // ---- split partial of every row that saw a key here
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (!valid[r] || st.m[r] == -INFINITY) continue;
    const size_t base = (static_cast<size_t>(q0 + tok[r]) * a.Hq + hq[r]) * a.max_splits + sidx;
    if (t4 == 0 && dim0 == 0) {
      a.part_ml[base * 2] = st.m[r];
      a.part_ml[base * 2 + 1] = st.l[r];
    }
    float* po = a.part_o + base * HD + dim0;
#pragma unroll
    for (int n = 0; n < ND / 8; ++n)
      *reinterpret_cast<float2*>(po + n * 8 + t4 * 2) = make_float2(st.o[n][2 * r], st.o[n][2 * r + 1]);
  }
}

// Scores-first decode CTA, for launches of at most one CTA per SM (small
// batches) at head dims 64 and 128.  There the tile-at-a-time kernel's time
// is one chain of dependent steps over the split's 16 tiles, each waiting
// for its copies.  One block of at most 16 rows, one split of at most
// kSfTiles tiles.  Warp 4 issues the copies, one tile per lane: every K
// tile into a slot of its own, the first V_OWN V tiles into slots of their
// own (one barrier for all of them), the remaining V tiles into K slots as
// the warps that scored those K tiles release them (one barrier again).
// Warps 0..3:
//   1. scores: warp w takes S, the mask and the row maxima of tiles
//      w, w + 4, ... as they land, keeps S in registers and posts the
//      maxima;
//   2. every warp runs the running maximum over all the tiles' maxima,
//      keeping each tile's rescale factor;
//   3. rounds of four tiles: each warp turns S of its tile of the round
//      into P (the bf16 hi/lo A fragments, posted to shared memory) and row
//      sums; after a named barrier every warp folds the round's tiles in
//      order into its quarter of the head dimension (l and O rescaled,
//      then the P V steps), with each tile's fragments loaded while the
//      previous tile's products run.
// Each value is computed by the same step functions as in `attn_tile`,
// from the same inputs, so every row's partial is bit for bit the one the
// tile-at-a-time kernels write; what changes is that only O's rescale and
// P V remain a chain from tile to tile, and that no step waits for a copy
// once the scores are in.
constexpr int kSfTiles = 16;  // tiles of a 512-key split
constexpr int kSfWarps = 4;

template <int HD>
struct SfCfg {
  using C = AttnCfg<HD>;
  static constexpr int P_BYTES = kSfTiles * 4 * 32 * 16;  // [tile][hi0, hi1, lo0, lo1][lane]: 16 B each
  static constexpr int STATIC_SMEM = C::PIDS * 4 + 2 * kSfTiles * 16 * 4 + 16;
  static constexpr int BAR_BYTES = (2 * kSfTiles + 2) * 8 + 16;
  static constexpr int FIXED = 1024 + P_BYTES + kSfTiles * C::TILE_BYTES + BAR_BYTES + STATIC_SMEM;
  static constexpr int V_FIT = (227 * 1024 - FIXED) / C::TILE_BYTES;
  static constexpr int V_OWN = V_FIT < kSfTiles ? V_FIT : kSfTiles;  // V tiles with slots of their own
  static constexpr int SMEM = 1024 + P_BYTES + (kSfTiles + V_OWN) * C::TILE_BYTES + BAR_BYTES;
  static_assert(V_OWN >= 1 && kSfTiles - V_OWN <= 32, "one lane per reused slot");
};

template <int HD>
struct SfShared {
  uint8_t* kslot;  // K tile t in slot t; V tile V_OWN + j later in slot j
  uint8_t* vslot;  // V tiles 0 .. V_OWN - 1
  uint4* pbuf;
  uint64_t* kfull;   // [kSfTiles] K tile t landed
  uint64_t* kempty;  // [kSfTiles] K tile t scored (its slot is free)
  uint64_t* vfull;   // [2] the V tiles in slots of their own / in K slots landed
  volatile int* abort_flag;
  float (*tmax)[16];  // [tile][row] row maxima of the tile's scores
  float (*rsum)[16];  // [tile][row] row sums of the tile's weights
  __device__ uint32_t vaddr(int t) const {
    return smem_u32(t < SfCfg<HD>::V_OWN ? vslot + t * AttnCfg<HD>::TILE_BYTES
                                         : kslot + (t - SfCfg<HD>::V_OWN) * AttnCfg<HD>::TILE_BYTES);
  }
};

// FULL: the split has all kSfTiles tiles (every split but a context's last
// and, under a window, its first), so that every loop has a fixed trip count
// and each round is straight-line code.
template <int HD, bool LOWER8, bool FULL>
__device__ __forceinline__ void sf_rows(const AttnArgs& a, const SfShared<HD>& sh, int ntiles, int tile_lo,
                                        const uint32_t (&qf)[HD / 16][4], const int (&pos)[2], const int (&lo)[2],
                                        const bool (&valid)[2], size_t base0, size_t base1, int warp, int lane) {
  using C = AttnCfg<HD>;
  constexpr int ND = HD / kSfWarps, KS = C::BNK / 16, NP = ND / 16;
  constexpr int V_OWN = SfCfg<HD>::V_OWN;
  constexpr int ROUNDS = kSfTiles / kSfWarps;
  const int nt = FULL ? kSfTiles : ntiles;
  const int gq = lane >> 2, t4 = lane & 3;
  const int dim0 = warp * ND;
  bool ok = true;
  auto wait = [&](uint64_t* bar) {
    ok = ok && __all_sync(0xffffffffu, mbar_wait(bar, 0, sh.abort_flag, a.status));
  };

  // ---- 1. scores of this warp's tiles.  Every tile of the CTA's key range
  // holds a key that some row sees (the rows' ranges [lo, pos] belong to
  // consecutive positions, so they overlap, and the CTA's range lies in
  // their union): no tile is skipped, as none is in the tile-at-a-time
  // kernels.  Tiles past the range post -inf maxima, which leave every
  // row's state as it is.
  float s[ROUNDS][C::BNK / 8][4];
#pragma unroll
  for (int i = 0; i < ROUNDS; ++i) {
    const int t = warp + kSfWarps * i;
    float mx[2] = {-INFINITY, -INFINITY};
    if (t < nt) {
      wait(&sh.kfull[t]);
      if (ok) {
        tile_scores<HD, C::BNK>(s[i], qf, smem_u32(sh.kslot + t * C::TILE_BYTES), lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.kempty[t]);
        tile_mask_max<C::BNK, LOWER8>(s[i], mx, (tile_lo + t) * C::BNK, pos, lo, a.scale_log2, lane);
      }
    }
    if (t4 == 0) {
      sh.tmax[t][gq] = mx[0];
      sh.tmax[t][gq + 8] = mx[1];
    }
  }
  bar_sync_named(1, kSfWarps * 32);

  // ---- 2. the running maximum over all tiles, with each tile's rescale factor
  float m[2] = {-INFINITY, -INFINITY};
  float alpha[kSfTiles][2], mown[ROUNDS][2];
#pragma unroll
  for (int t = 0; t < kSfTiles; ++t) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mn;
      bool rv;
      tile_running_max(m[r], sh.tmax[t][gq + 8 * r], mn, alpha[t][r], rv);
      m[r] = mn;
      if (t % kSfWarps == warp) mown[t / kSfWarps][r] = mn;
    }
  }
  // P of this warp's tile of round i (bf16 hi/lo fragments) and its row sums
  auto post_p = [&](int i) {
    const int t = warp + kSfWarps * i;
    if (t >= nt) return;
    uint32_t pa[KS][4], pl[KS][4];
    float rs[2];
    tile_probs<C::BNK, LOWER8>(s[i], mown[i], pa, pl, rs);
    uint4* dst = sh.pbuf + t * 4 * 32 + lane;
    dst[0] = make_uint4(pa[0][0], pa[0][1], pa[0][2], pa[0][3]);
    dst[32] = make_uint4(pa[1][0], pa[1][1], pa[1][2], pa[1][3]);
    dst[64] = make_uint4(pl[0][0], pl[0][1], pl[0][2], pl[0][3]);
    dst[96] = make_uint4(pl[1][0], pl[1][1], pl[1][2], pl[1][3]);
    if (t4 == 0) {
      sh.rsum[t][gq] = rs[0];
      sh.rsum[t][gq + 8] = rs[1];
    }
  };

  // ---- 3. rounds of 4 tiles: every warp's P of the round posted, then
  // P V of the round's tiles in order (each tile's fragments loaded while
  // the previous tile's products run), then this warp's P of the next round
  float l[2] = {0.f, 0.f};
  float o[ND / 8][4];
#pragma unroll
  for (int n = 0; n < ND / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  uint32_t fa[2][KS][4], fl[2][KS][4], vb[2][KS][NP][4];
  auto load = [&](int t, int buf) {
    const uint4* src = sh.pbuf + t * 4 * 32 + lane;
    const uint4 h0 = src[0], h1 = src[32], l0 = src[64], l1 = src[96];
    fa[buf][0][0] = h0.x; fa[buf][0][1] = h0.y; fa[buf][0][2] = h0.z; fa[buf][0][3] = h0.w;
    fa[buf][1][0] = h1.x; fa[buf][1][1] = h1.y; fa[buf][1][2] = h1.z; fa[buf][1][3] = h1.w;
    fl[buf][0][0] = l0.x; fl[buf][0][1] = l0.y; fl[buf][0][2] = l0.z; fl[buf][0][3] = l0.w;
    fl[buf][1][0] = l1.x; fl[buf][1][1] = l1.y; fl[buf][1][2] = l1.z; fl[buf][1][3] = l1.w;
    tile_v_frags<HD, C::BNK, ND>(vb[buf], sh.vaddr(t), lane, dim0);
  };
  if (ok) post_p(0);
#pragma unroll
  for (int i = 0; i < ROUNDS; ++i) {
    bar_sync_named(1, kSfWarps * 32);
    const int t0 = kSfWarps * i;
    if (t0 < nt) {
      if (t0 == 0) wait(&sh.vfull[0]);
      if (t0 == V_OWN) wait(&sh.vfull[1]);
      load(t0, 0);
#pragma unroll
      for (int j = 0; j < kSfWarps; ++j) {
        const int t = t0 + j, u = t + 1;
        if (t >= nt) break;
        if (j + 1 < kSfWarps && u < nt) {
          if (u == V_OWN) wait(&sh.vfull[1]);
          load(u, (j + 1) & 1);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int row = gq + 8 * r;
          tile_update_l(l[r], alpha[t][r], sh.rsum[t][row], sh.tmax[t][row] != -INFINITY);
        }
        tile_rescale<ND, LOWER8>(o, alpha[t]);
        tile_pv_mma<C::BNK, ND>(o, fa[j & 1], fl[j & 1], vb[j & 1]);
      }
    }
    if (i + 1 < ROUNDS && ok) post_p(i + 1);
  }
  if (!ok) return;  // a wait gave up: the data of some tiles may not have landed

  // ---- split partial of every row that saw a key here
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (!valid[r] || m[r] == -INFINITY) continue;
    const size_t base = r ? base1 : base0;
    if (t4 == 0 && dim0 == 0) {
      a.part_ml[base * 2] = m[r];
      a.part_ml[base * 2 + 1] = l[r];
    }
    float* po = a.part_o + base * HD + dim0;
#pragma unroll
    for (int n = 0; n < ND / 8; ++n)
      *reinterpret_cast<float2*>(po + n * 8 + t4 * 2) = make_float2(o[n][2 * r], o[n][2 * r + 1]);
  }
}

template <int HD>
__global__ void __launch_bounds__((kSfWarps + 1) * 32, 1)
    attn_sf_kernel(const __grid_constant__ CUtensorMap kvmap, AttnArgs a) {
  using C = AttnCfg<HD>;
  using SC = SfCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ int pid_s[C::PIDS];
  __shared__ float tmax[kSfTiles][16], rsum[kSfTiles][16];
  SfShared<HD> sh;
  sh.pbuf = reinterpret_cast<uint4*>(smem);
  sh.kslot = smem + SC::P_BYTES;
  sh.vslot = sh.kslot + kSfTiles * C::TILE_BYTES;
  sh.kfull = reinterpret_cast<uint64_t*>(sh.vslot + SC::V_OWN * C::TILE_BYTES);
  sh.kempty = sh.kfull + kSfTiles;
  sh.vfull = sh.kempty + kSfTiles;
  sh.abort_flag = reinterpret_cast<volatile int*>(sh.vfull + 2);
  sh.tmax = tmax;
  sh.rsum = rsum;

  // Up to the wait for the previous kernel this CTA reads only the status
  // word and the step's description (sequence classes, lengths, page table),
  // which are written before the step's first kernel, so that their round
  // trips hide behind that wait; the Q rows and K/V pages the previous
  // kernels write are read after it.  (A failure of the kernel right before
  // this one is then seen by the next kernel instead.)
  {
    __shared__ int skip;  // once any bounded wait has given up, later CTAs skip their work
    if (threadIdx.x == 0) skip = a.status ? *reinterpret_cast<volatile int*>(a.status) : 0;
    __syncthreads();
    if (skip) return;
  }
  // ---- work item -> (request, KV head, split); one block of 16 rows
  const int item = blockIdx.x;
  if (item >= a.cls_start[a.n_cls]) return;
  int lo_i = 0, hi_i = a.n_cls - 1;
  while (lo_i < hi_i) {
    const int mid = (lo_i + hi_i + 1) >> 1;
    if (a.cls_start[mid] <= item) lo_i = mid; else hi_i = mid - 1;
  }
  const int b = a.cls_seq[lo_i];
  int local = item - a.cls_start[lo_i];
  const int q0 = a.cu_q[b], qlen = a.cu_q[b + 1] - q0, cached = a.cached_len[b];
  const int kv_len = cached + qlen;
  const int G = a.Hq / a.Hkv;
  const int nsplit = (kv_len - 1) / a.split + 1;
  const int sidx = local % nsplit;
  local /= nsplit;
  const int kvh = local % a.Hkv;
  const int r0 = (local / a.Hkv) * 16;
  const int rows = qlen * G;
  const int r_end = min(rows, r0 + 16);
  const int p_min = cached + r0 / G, p_max = cached + (r_end - 1) / G;
  const int lo_min = a.window > 0 ? max(0, p_min - a.window + 1) : 0;
  const int key_lo = max(sidx * a.split, lo_min);
  const int key_hi = min((sidx + 1) * a.split - 1, p_max);
  if (key_lo > key_hi) return;
  const int tile_lo = key_lo / C::BNK;
  const int ntiles = key_hi / C::BNK - tile_lo + 1;  // <= kSfTiles (checked at launch)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kSfWarps) {  // the copy warp reads the page ids it needs
    const int lp_first = (tile_lo * C::BNK) >> 4;
    for (int j = lane; j < C::PIDS; j += 32) {
      const int lp = lp_first + j;
      pid_s[j] = (j < ntiles * C::PAGES && lp * 16 < kv_len)
                     ? a.page_table[static_cast<size_t>(b) * a.pt_stride + lp] : -1;
    }
  }
  if (threadIdx.x == 0) {
    for (int k = 0; k < kSfTiles; ++k) {
      mbar_init(&sh.kfull[k], 1);
      mbar_init(&sh.kempty[k], 1);
    }
    mbar_init(&sh.vfull[0], 1);
    mbar_init(&sh.vfull[1], 1);
    *sh.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  if (warp == kSfWarps) {
    // One tile per lane: K tile `lane`, V tile `lane - 16` into its own slot,
    // then V tile V_OWN + `lane` into the slot of K tile `lane` once scored.
    auto copy_tile = [&](int t, bool is_v, uint8_t* dst, uint64_t* bar) {
#pragma unroll
      for (int pg = 0; pg < C::PAGES; ++pg) {
        const int phys = pid_s[t * C::PAGES + pg];  // -1 past the context: zero fill
        const int row = phys >= 0 ? a.layer_row0 + ((phys * 2 + (is_v ? 1 : 0)) * a.Hkv + kvh) * 16 : a.pool_rows;
        tma_load_3d(dst + pg * C::PAGE_BYTES, &kvmap, bar, 0, 0, row);
      }
    };
    const int nv0 = min(ntiles, SC::V_OWN), nv1 = ntiles - nv0;
    if (lane == 0) {
      mbar_arrive_expect_tx(&sh.vfull[0], nv0 * C::TILE_BYTES);
      if (nv1 > 0) mbar_arrive_expect_tx(&sh.vfull[1], nv1 * C::TILE_BYTES);
    }
    __syncwarp();
    if (lane < ntiles) {
      mbar_arrive_expect_tx(&sh.kfull[lane], C::TILE_BYTES);
      copy_tile(lane, false, sh.kslot + lane * C::TILE_BYTES, &sh.kfull[lane]);
    }
    if (lane >= 16 && lane - 16 < nv0) copy_tile(lane - 16, true, sh.vslot + (lane - 16) * C::TILE_BYTES, &sh.vfull[0]);
    if (lane < nv1 && mbar_wait(&sh.kempty[lane], 0, sh.abort_flag, a.status))
      copy_tile(SC::V_OWN + lane, true, sh.kslot + lane * C::TILE_BYTES, &sh.vfull[1]);
    __syncwarp();
    if (lane == 0) {  // every copy lands before the CTA leaves, also when a wait gave up
      for (int t = 0; t < ntiles; ++t) drain_wait(&sh.kfull[t], 0);
      drain_wait(&sh.vfull[0], 0);
      if (nv1 > 0) drain_wait(&sh.vfull[1], 0);
    }
    return;
  }

  // ---- the block's rows (every compute warp holds all 16 and a quarter of the head)
  const int gq = lane >> 2, t4 = lane & 3;
  int pos[2], lo[2], tok[2], hq[2];
  bool valid[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = r0 + gq + 8 * r;
    valid[r] = row < rows;
    tok[r] = row / G;
    hq[r] = kvh * G + row % G;
    pos[r] = valid[r] ? cached + tok[r] : -1;
    lo[r] = valid[r] ? (a.window > 0 ? max(0, pos[r] - a.window + 1) : 0) : 1;
  }
  uint32_t qf[HD / 16][4];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const __nv_bfloat16* qr = a.q + (static_cast<size_t>(q0 + tok[r]) * a.Hq + hq[r]) * HD;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      qf[kk][r] = valid[r] ? *reinterpret_cast<const uint32_t*>(qr + kk * 16 + t4 * 2) : 0u;
      qf[kk][2 + r] = valid[r] ? *reinterpret_cast<const uint32_t*>(qr + kk * 16 + 8 + t4 * 2) : 0u;
    }
  }
  const size_t base0 = (static_cast<size_t>(q0 + tok[0]) * a.Hq + hq[0]) * a.max_splits + sidx;
  const size_t base1 = (static_cast<size_t>(q0 + tok[1]) * a.Hq + hq[1]) * a.max_splits + sidx;
  const bool lower8 = rows - r0 <= 8, full = ntiles == kSfTiles;
  if (lower8 && full)
    sf_rows<HD, true, true>(a, sh, ntiles, tile_lo, qf, pos, lo, valid, base0, base1, warp, lane);
  else if (lower8)
    sf_rows<HD, true, false>(a, sh, ntiles, tile_lo, qf, pos, lo, valid, base0, base1, warp, lane);
  else if (full)
    sf_rows<HD, false, true>(a, sh, ntiles, tile_lo, qf, pos, lo, valid, base0, base1, warp, lane);
  else
    sf_rows<HD, false, false>(a, sh, ntiles, tile_lo, qf, pos, lo, valid, base0, base1, warp, lane);
}

// Left-to-right fold of a row's split partials, then o / l -> bf16.  The
// loop is unrolled so that the loads of later splits are in flight while
// earlier ones are folded; the fold itself stays strictly left to right.
template <int PER>
__device__ __forceinline__ void load_part(const float* p, float* o) {
  if constexpr (PER % 4 == 0) {
#pragma unroll
    for (int i = 0; i < PER; i += 4) {
      const float4 v = *reinterpret_cast<const float4*>(p + i);
      o[i] = v.x;
      o[i + 1] = v.y;
      o[i + 2] = v.z;
      o[i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < PER; i += 2) {
      const float2 v = *reinterpret_cast<const float2*>(p + i);
      o[i] = v.x;
      o[i + 1] = v.y;
    }
  }
}

template <int HD, int kBatch>
__global__ void __launch_bounds__(128) merge_kernel(MergeArgs a) {
  constexpr int PER = HD / 32;
  // The row's token and position come from the step's description (written
  // before the step's first kernel): read before the wait for the attention
  // kernel, whose partials are read after it.
  const int w = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const bool row = w < a.T * a.Hq;
  const int tok = !row ? 0 : a.tokens ? a.tokens[w / a.Hq] : w / a.Hq, h = w % a.Hq;
  const int p = row ? a.positions[tok] : 0;
  pdl_wait();
  pdl_trigger();
  if (!row) return;
  const int lo = a.window > 0 ? max(0, p - a.window + 1) : 0;
  const int s0 = lo / a.split, s1 = p / a.split;
  const size_t base = (static_cast<size_t>(tok) * a.Hq + h) * a.max_splits;
  float M = a.part_ml[(base + s0) * 2], L = a.part_ml[(base + s0) * 2 + 1];
  float O[PER];
  load_part<PER>(a.part_o + (base + s0) * HD + lane * PER, O);
  // The partials of up to kBatch splits are loaded together (one memory
  // round trip per batch instead of one per split), then folded one by one
  // in ascending split order exactly as before.  Launches of many rows take
  // four at a time, which keeps the registers low enough for ten CTAs per SM
  // (eight at a time held 75 registers and six CTAs: the kernel waits on
  // memory and needs the warps); launches of at most one CTA per SM take all
  // the splits of a context in one round trip.
  for (int sb = s0 + 1; sb <= s1; sb += kBatch) {
    float2 ml[kBatch];
    float P[kBatch][PER];
#pragma unroll
    for (int c = 0; c < kBatch; ++c)
      if (sb + c <= s1) {
        ml[c] = *reinterpret_cast<const float2*>(a.part_ml + (base + sb + c) * 2);
        load_part<PER>(a.part_o + (base + sb + c) * HD + lane * PER, P[c]);
      }
#pragma unroll
    for (int c = 0; c < kBatch; ++c)
      if (sb + c <= s1) {
        const float mn = fmaxf(M, ml[c].x);
        const float ca = ex2(__fsub_rn(M, mn)), cb = ex2(__fsub_rn(ml[c].x, mn));
        L = __fadd_rn(__fmul_rn(L, ca), __fmul_rn(ml[c].y, cb));
#pragma unroll
        for (int i = 0; i < PER; ++i) O[i] = __fadd_rn(__fmul_rn(O[i], ca), __fmul_rn(P[c][i], cb));
        M = mn;
      }
  }
  __nv_bfloat16* out = a.out + (static_cast<size_t>(tok) * a.Hq + h) * HD + lane * PER;
#pragma unroll
  for (int i = 0; i < PER; i += 2)
    *reinterpret_cast<uint32_t*>(out + i) = pack_bf16x2(__fdiv_rn(O[i], L), __fdiv_rn(O[i + 1], L));
}

constexpr int kMergeWide = 16;  // splits of an 8192-key context

int sm_count_attn() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  }
  return n;
}

// Pipeline depth of one launch: the deepest (up to 8 stages) whose CTAs all
// fit on the GPU at once, so that few work items (small batches) keep as many
// key tiles in flight per SM as a full wave of 2-stage CTAs does.
template <int HD>
int attn_stages(int n_items, int static_smem) {
  using C = AttnCfg<HD>;
  constexpr int kSmemPerSM = 228 * 1024, kSmemPerCTA = 227 * 1024;
  for (int ns = C::MAX_STAGES; ns > 2; --ns) {
    if (C::smem(ns) + static_smem > kSmemPerCTA) continue;
    const long long slots =
        static_cast<long long>(sm_count_attn()) * (kSmemPerSM / (C::smem(ns) + static_smem + 1024));
    if (slots >= n_items) return ns;
  }
  return 2;
}

template <int HD, int NW, int DS, bool FOLD, bool PROD = false>
int launch_attn_t(const CUtensorMap& kvmap, const AttnArgs& a0, int n_items, cudaStream_t s) {
  using C = AttnCfg<HD>;
  constexpr int kStatic = C::STATIC_SMEM + (PROD ? C::MAX_STAGES * 8 : 0);  // + the release barriers
  static bool configured = false;
  if (!configured) {
    int max_ns = C::MAX_STAGES;
    while (C::smem(max_ns) + kStatic > 227 * 1024) --max_ns;
    VD_CUDA_TRY(cudaFuncSetAttribute(attn_kernel<HD, NW, DS, FOLD, PROD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::smem(max_ns)));
    configured = true;
  }
  AttnArgs a = a0;
  a.stages = attn_stages<HD>(n_items, kStatic);
  VD_CUDA_TRY(
      launch_k(attn_kernel<HD, NW, DS, FOLD, PROD>, dim3(n_items), dim3((NW + PROD) * 32), C::smem(a.stages), s, kvmap,
               a));
  return VD_OK;
}

template <int HD>
int launch_attn_sf(const CUtensorMap& kvmap, const AttnArgs& a, int n_items, cudaStream_t s) {
  using SC = SfCfg<HD>;
  static_assert(kSfTiles * AttnCfg<HD>::PAGES <= AttnCfg<HD>::PIDS, "page ids of a split");
  static_assert(SC::SMEM + SC::STATIC_SMEM <= 227 * 1024, "shared memory");
  static bool configured = false;
  if (!configured) {
    VD_CUDA_TRY(cudaFuncSetAttribute(attn_sf_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, SC::SMEM));
    configured = true;
  }
  VD_CUDA_TRY(launch_k(attn_sf_kernel<HD>, dim3(n_items), dim3((kSfWarps + 1) * 32), SC::SMEM, s, kvmap, a));
  return VD_OK;
}

// One CTA per SM: the scores-first CTA where a split's K tiles fit in shared
// memory at once (head dims 64 and 128), else the copy-warp CTA.
template <int HD>
int launch_attn_wide(const CUtensorMap& kvmap, const AttnArgs& a, int n_items, bool sf, cudaStream_t s) {
  if constexpr (HD <= 128)
    if (sf) return launch_attn_sf<HD>(kvmap, a, n_items, s);
  return launch_attn_t<HD, 4, 4, false, true>(kvmap, a, n_items, s);
}

}  // namespace

// Scratch for vd_op_attention_static: the split partials (o, then m/l) of
// one call.  It is a fixed device array so that the call needs no
// allocation; every device that loads the library holds it until exit.
static __device__ __align__(256) float g_attn_static_scratch[kAttnStaticScratchBytes / sizeof(float)];

int attn_static_scratch(void** ptr) {
  // Device address of the array on the current device.  Host code cannot
  // take the address of a __device__ symbol; the lookup allocates nothing
  // and is made on every call, so a context re-created on the same device
  // never gets an address cached from the old one.
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_static_scratch);
  if (e != cudaSuccess)
    return fail(VD_ERR_CUDA, std::string("cudaGetSymbolAddress(static attention scratch): ") + cudaGetErrorString(e));
  *ptr = p;
  return VD_OK;
}

int attn_key_tile(int hd) { return hd >= 256 ? AttnCfg<256>::BNK : AttnCfg<128>::BNK; }
static_assert(512 % AttnCfg<64>::BNK == 0 && 512 % AttnCfg<256>::BNK == 0, "splits must hold whole key tiles");

int launch_attention(const CUtensorMap& kvmap, const AttnArgs& a, int hd, bool prefill_class, int n_items,
                     cudaStream_t s) {
  if (n_items <= 0) return VD_OK;
  if (prefill_class && a.fold) return fail(VD_ERR_INVALID_ARG, "split folding is for decode-class CTAs");
  if (a.split > AttnCfg<64>::PIDS * 16)  // a split CTA stages the ids of every page it streams
    return fail(VD_ERR_INVALID_ARG, "KV split larger than the staged page ids");
  // Decode CTAs split the head dimension of P V over 2 warps; a launch of at
  // most one CTA per SM (small batches) runs the scores-first CTA, whose 4
  // warps share the split's scores and a quarter of P V each.  Every output
  // element keeps the same instruction chain either way.
  const bool wide = !prefill_class && !a.fold && n_items <= sm_count_attn();
  const bool sf = wide && a.split <= kSfTiles * AttnCfg<64>::BNK;
#define VD_ATTN_LAUNCH(HD_)                                                                     \
  if (hd == HD_)                                                                              \
    return prefill_class ? launch_attn_t<HD_, 4, 1, false>(kvmap, a, n_items, s)               \
           : a.fold      ? launch_attn_t<HD_, 2, 2, true>(kvmap, a, n_items, s)                \
           : wide        ? launch_attn_wide<HD_>(kvmap, a, n_items, sf, s)                     \
                         : launch_attn_t<HD_, 2, 2, false>(kvmap, a, n_items, s);
  VD_ATTN_LAUNCH(64)
  VD_ATTN_LAUNCH(128)
  VD_ATTN_LAUNCH(256)
#undef VD_ATTN_LAUNCH
  return fail(VD_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
}

int launch_merge(const MergeArgs& a, int hd, cudaStream_t s) {
  const int warps = a.T * a.Hq;
  if (warps <= 0) return VD_OK;
  const int blocks = (warps + 3) / 4;
  const bool few = blocks <= sm_count_attn();
  auto k = hd == 64    ? (few ? merge_kernel<64, kMergeWide> : merge_kernel<64, 4>)
           : hd == 128 ? (few ? merge_kernel<128, kMergeWide> : merge_kernel<128, 4>)
           : hd == 256 ? (few ? merge_kernel<256, kMergeWide> : merge_kernel<256, 4>)
                       : nullptr;
  if (!k) return fail(VD_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
  VD_CUDA_TRY(launch_k(k, dim3(blocks), dim3(128), 0, s, a));
  return VD_OK;
}

}  // namespace vd
