// Unified prefill/decode paged attention with a fixed KV split size.
//
// Rows.  For request b and KV head g the rows are (token i, query head of
// the group) pairs, token-major.  A CTA owns a block of rows of one
// (request, KV head) and one KV split.  Decode-shaped requests (q_len *
// Hq/Hkv <= 16, one block of 16 rows) run with two warps that share the rows
// and split the head dimension of the P V product; longer chunks run four
// warps of 16 rows each, sharing every K/V tile.  The per-element instruction
// sequence is the same in both instantiations (the same `attn_tile` body),
// so a row's result does not depend on which of them ran it.
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

// One key tile for the 16 rows of a warp, which accumulates output dims
// [dim0, dim0 + ND).  S and the softmax state are computed over the full
// head either way, so every output element gets the same instruction chain
// whether one warp owns all dims or several warps share them.  LOWER8: rows
// 8..15 of the warp are known to hold no row (a decode CTA of at most 8
// rows), so their masking, softmax and rescale are skipped: their weights
// are exactly 0 either way, and the other rows' instructions are unchanged.
template <int HD, int BNK, int ND, bool LOWER8>
__device__ __forceinline__ void attn_tile(RowState<ND>& st, const uint32_t (&qf)[HD / 16][4], uint32_t kbase,
                                          uint32_t vbase, int key0, const int (&pos)[2], const int (&lo)[2],
                                          float scale_log2, int lane, int dim0) {
  const int t4 = lane & 3, mi = lane >> 3, r8 = lane & 7;
  float s[BNK / 8][4];
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
  float mx[2] = {-INFINITY, -INFINITY};
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
  float mnew[2], alpha[2];
  bool rv[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (LOWER8 && r == 1) {  // no row: the state stays as it is, as a fully masked row's does
      rv[r] = false;
      mnew[r] = st.m[r];
      alpha[r] = 1.0f;
      continue;
    }
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    rv[r] = mx[r] != -INFINITY;
    mnew[r] = rv[r] ? fmaxf(st.m[r], mx[r]) : st.m[r];
    alpha[r] = rv[r] ? ex2(__fsub_rn(st.m[r], mnew[r])) : 1.0f;
  }
  // P enters the P V product as two bf16 terms, hi = bf16(p) and
  // lo = bf16(p - hi) (p - hi is exact in fp32), so the weights carry about
  // 16 significant bits; the row sum uses the fp32 weights.
  uint32_t pa[BNK / 16][4], pl[BNK / 16][4];
  float rs[2] = {0.f, 0.f};
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
    st.l[r] = rv[r] ? __fadd_rn(__fmul_rn(st.l[r], alpha[r]), rs[r]) : st.l[r];
    st.m[r] = mnew[r];
  }
#pragma unroll
  for (int n = 0; n < ND / 8; ++n) {
    st.o[n][0] = __fmul_rn(st.o[n][0], alpha[0]);
    st.o[n][1] = __fmul_rn(st.o[n][1], alpha[0]);
    if (!LOWER8) {  // rows 8..15 (with LOWER8 their alpha is 1, and their sums are never stored)
      st.o[n][2] = __fmul_rn(st.o[n][2], alpha[1]);
      st.o[n][3] = __fmul_rn(st.o[n][3], alpha[1]);
    }
  }
  const int np0 = dim0 / 16;
#pragma unroll
  for (int ks = 0; ks < BNK / 16; ++ks) {
#pragma unroll
    for (int np = 0; np < ND / 16; ++np) {
      uint32_t b[4];
      ldmatrix_x4_trans(b, vbase + kv_off<HD>(ks * 16 + (mi & 1) * 8 + r8, (np0 + np) * 2 + (mi >> 1)));
      mma_bf16_16816(st.o[2 * np], pa[ks], b);
      mma_bf16_16816(st.o[2 * np], pl[ks], b);
      mma_bf16_16816(st.o[2 * np + 1], pa[ks], b + 2);
      mma_bf16_16816(st.o[2 * np + 1], pl[ks], b + 2);
    }
  }
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

  pdl_wait();
  pdl_trigger();
  // Once any bounded wait has given up, later CTAs skip their work.
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

template <int HD>
__global__ void __launch_bounds__(128) merge_kernel(MergeArgs a) {
  constexpr int PER = HD / 32;
  pdl_wait();
  pdl_trigger();
  const int w = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= a.T * a.Hq) return;
  const int tok = a.tokens ? a.tokens[w / a.Hq] : w / a.Hq, h = w % a.Hq;
  const int p = a.positions[tok];
  const int lo = a.window > 0 ? max(0, p - a.window + 1) : 0;
  const int s0 = lo / a.split, s1 = p / a.split;
  const size_t base = (static_cast<size_t>(tok) * a.Hq + h) * a.max_splits;
  float M = a.part_ml[(base + s0) * 2], L = a.part_ml[(base + s0) * 2 + 1];
  float O[PER];
  load_part<PER>(a.part_o + (base + s0) * HD + lane * PER, O);
  // The partials of up to kBatch splits are loaded together (one memory
  // round trip per batch instead of one per split), then folded one by one
  // in ascending split order exactly as before.  Four at a time keeps the
  // registers low enough for ten CTAs per SM (eight at a time held 75
  // registers and six CTAs: the kernel waits on memory and needs the warps).
  constexpr int kBatch = 4;
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
  // Decode CTAs split the head dimension of P V over 2 warps, or over 4 when
  // the launch has at most one CTA per SM (small batches); every
  // output element keeps the same instruction chain either way.
  const bool wide = !prefill_class && !a.fold && n_items <= sm_count_attn();
#define VD_ATTN_LAUNCH(HD_)                                                                     \
  if (hd == HD_)                                                                              \
    return prefill_class ? launch_attn_t<HD_, 4, 1, false>(kvmap, a, n_items, s)               \
           : a.fold      ? launch_attn_t<HD_, 2, 2, true>(kvmap, a, n_items, s)                \
           : wide        ? launch_attn_t<HD_, 4, 4, false, true>(kvmap, a, n_items, s)         \
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
  auto k = hd == 64 ? merge_kernel<64> : hd == 128 ? merge_kernel<128> : hd == 256 ? merge_kernel<256> : nullptr;
  if (!k) return fail(VD_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
  VD_CUDA_TRY(launch_k(k, dim3(blocks), dim3(128), 0, s, a));
  return VD_OK;
}

}  // namespace vd
