// Prefill-class paged attention on 5th-generation tensor cores (tcgen05),
// head dimensions 64, 128 and 256.
//
// Same rows, tiles, splits and per-row arithmetic as the mma.sync kernel of
// attention.cu (深入解析 Vosti §六 6.2: causal prefix equivalence, the
// sliding-window traversal and the masking rules; "Deterministic and
// bit-exact inference", technical section: fixed split size).  A CTA owns
// 128 rows (the MMA's M) of one (request, KV head) and one KV split and folds
// the split's 32-key tiles in ascending order.  Per tile and row:
//
//   S     = Q K^T, one chain of hd/16 K = 16 steps from zero;
//   v     = visible ? S * log2(e)/sqrt(hd) : -inf;   mx = max v
//   m'    = mx > -inf ? max(m, mx) : m;   alpha = mx > -inf ? 2^(m - m') : 1
//   p     = v > -inf ? 2^(v - m') : 0;   hi = bf16(p), lo = bf16(p - hi)
//   l     = mx > -inf ? l * alpha + rowsum(p) : l
//   O     = O * alpha, then O += hi[0:16] V[0:16], lo[0:16] V[0:16],
//           hi[16:32] V[16:32], lo[16:32] V[16:32]   (four K = 16 steps)
//
// with rowsum(p) summed in the mma.sync kernel's order: four partial sums
// s_t over keys {2t, 2t+1, 8+2t, 9+2t, 16+2t, 17+2t, 24+2t, 25+2t} in that
// order, then (s_0 + s_1) + (s_2 + s_3).  A tcgen05.mma K = 16 step gives the
// same fp32 result as an mma.sync m16n8k16 step for the same operands and
// accumulator, bit for bit (measured on this GPU over 37.7 M elements:
// chains of 1, 2 and 8 steps, from zero and onto given accumulators), so a
// row run here equals the same row run by the mma.sync decode or prefill
// kernel; the attention tests check that bitwise.
//
// Roles (320 threads; 576 at hd 256): warp 0 allocates TMEM, reads the
// split's page ids and one lane issues the K/V page copies (3-D TMA boxes of
// one page and 64 head dims, so that the K or V of a stage, two tiles, is [hd
// block][64 keys][64] with the 128-byte swizzle, the canonical operand
// layout); warp 1, one lane, issues the MMAs; the softmax warps (8, or 16 at
// hd 256, two for each 16 rows) each hold 16 rows, read from TMEM in the
// layout of an mma.sync C fragment (two rows and eight keys per thread), and
// run the softmax, the O rescale and the epilogue with the mma.sync kernel's
// per-row code.  S of a stage's two tiles is one chain of N = 64
// MMAs (an MMA's N does not change an element) into 64 TMEM columns, issued
// once the softmax has read the previous stage's scores.  P (hi and lo bf16,
// two per 32-bit column) goes to one of two TMEM buffers and is the A operand
// of P V, straight from TMEM; V is the MN-major B operand; O takes hd TMEM
// columns.  Every wait is bounded.
#include <math.h>

#include "vd_device.cuh"
#include "vd_internal.h"

namespace vd {
namespace {

// x[0] *= y, x[1] *= y (or -= y) in one instruction: each element rounded to
// nearest exactly as mul.rn.f32 / sub.rn.f32 round it.
__device__ __forceinline__ void mul2_rn(float& x0, float& x1, float y) {
  uint64_t v, w;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(x0), "f"(x1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(w) : "f"(y));
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(v) : "l"(w));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(v));
}
__device__ __forceinline__ void sub2_rn(float& x0, float& x1, float y) {
  uint64_t v, w;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(x0), "f"(x1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(w) : "f"(y));
  asm("sub.rn.f32x2 %0, %0, %1;" : "+l"(v) : "l"(w));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(v));
}

template <int HD>
struct TcAttnCfg {
  static constexpr int ROWS = 128;                 // rows per CTA (MMA M)
  static constexpr int BNK = 32;                   // keys per tile: the softmax step of every attention kernel
  static constexpr int SK = 2 * BNK;               // keys per K/V stage (two tiles share one S MMA chain)
  static constexpr int KB = HD / 64;               // 64-wide head-dim blocks
  static constexpr int Q_BYTES = KB * ROWS * 128;  // [hd block][row][64]
  static constexpr int HB = SK * 128;              // one hd block of a stage's K or V: [key][64]
  static constexpr int KV_BYTES = KB * HB;         // K or V of a stage: [hd block][key][64]
  static constexpr int STAGES = HD == 64 ? 4 : 2;  // K/V stages in flight (two tiles each)
  // Softmax warps: eight hold 16 rows each; at hd 256 two warps share each 16
  // rows (both run the same softmax; each owns 128 of O's columns)
  static constexpr int NSW = HD == 256 ? 16 : 8;
  static constexpr int NS = 32 * NSW;  // softmax threads
  static constexpr int THREADS = 64 + NS;
  static constexpr int OW = HD / (NSW / 8);  // O columns per softmax warp
  // TMEM: the scores of a stage's two tiles (SK columns), O (hd columns),
  // then two P buffers of BNK columns (hi and lo bf16 of a row's BNK keys,
  // two per column)
  static constexpr int O_COL = SK;
  static constexpr int P_COL = O_COL + HD;
  static constexpr int TMEM_COLS = HD == 256 ? 512 : 256;
  static_assert(P_COL + 2 * BNK <= TMEM_COLS, "TMEM columns per CTA");
  static constexpr int PIDS = 64;  // page ids of a split (at most 32 pages of 16 keys)
  static constexpr int SMEM = 1024 + Q_BYTES + STAGES * 2 * KV_BYTES + 256 + PIDS * 4;
  // At most 512 / TMEM_COLS CTAs may share an SM (a CTA that found too few
  // TMEM columns would wait in tcgen05.alloc); shared memory bounds it.
  static constexpr int CTAS_PER_SM = (228 * 1024) / (SMEM + 1024);
  static_assert(CTAS_PER_SM * TMEM_COLS <= 512, "TMEM columns per SM");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

template <int HD>
__global__ void __launch_bounds__(TcAttnCfg<HD>::THREADS, HD == 256 ? 1 : 2)
    attn_tc_kernel(const __grid_constant__ CUtensorMap kvmap, AttnArgs a) {
  using C = TcAttnCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sq = smem;
  uint8_t* skv = sq + C::Q_BYTES;  // stage s: K at skv + s * 2 * KV_BYTES, V right after
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(skv + C::STAGES * 2 * C::KV_BYTES);
  uint64_t* kv_empty = kv_full + C::STAGES;
  uint64_t* s_full = kv_empty + C::STAGES;  // the scores of a stage's tiles are in TMEM
  uint64_t* s_free = s_full + 1;            // the softmax threads have read them
  uint64_t* p_full = s_free + 1;            // P of a tile written and O rescaled
  uint64_t* pv_done = p_full + 1;           // the tile's P V steps completed
  uint64_t* q_full = pv_done + 1;           // Q rows in shared memory
  uint64_t* mma_done = q_full + 1;          // every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* pid_s = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(kv_full) + 256);  // [PIDS]

  pdl_wait();
  pdl_trigger();
  {
    __shared__ int skip;  // one read for the whole CTA keeps the exit uniform
    if (threadIdx.x == 0) skip = a.status ? *reinterpret_cast<volatile int*>(a.status) : 0;
    __syncthreads();
    if (skip) return;
  }
  // ---- work item -> (request, row block, KV head, split), as in attention.cu
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
  const int rb = local / a.Hkv;
  const int rows = qlen * G;
  const int r0 = rb * C::ROWS;
  const int r_end = min(rows, r0 + C::ROWS);
  const int p_min = cached + r0 / G, p_max = cached + (r_end - 1) / G;
  const int lo_min = a.window > 0 ? max(0, p_min - a.window + 1) : 0;
  const int key_lo = max(sidx * a.split, lo_min);
  const int key_hi = min((sidx + 1) * a.split - 1, p_max);
  if (key_lo > key_hi) return;  // no visible key of these rows in this split
  const int tile_lo = key_lo / C::BNK;
  const int ntiles = key_hi / C::BNK - tile_lo + 1;
  const int nstage = (ntiles + 1) >> 1;  // K/V stages: tiles 2 g and 2 g + 1 (the latter may be past the end)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The physical ids of the split's pages (-1 past its tiles or the
  // context), read by one warp in one round trip, so that no copy waits for a
  // page-table load.
  const int lp_first = (tile_lo * C::BNK) >> 4;
  if (warp == 0)
    for (int j = lane; j < C::PIDS; j += 32) {
      const int lp = lp_first + j;
      pid_s[j] = (j < ntiles * (C::BNK / 16) && lp * 16 < kv_len)
                     ? a.page_table[static_cast<size_t>(b) * a.pt_stride + lp] : -1;
    }
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, C::NS);
    mbar_init(p_full, C::NS);
    mbar_init(pv_done, 1);
    mbar_init(q_full, C::NS);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int issued = 0;  // producer: stages whose copies were issued
  if (warp == 0) {
    if (lane == 0) {
      for (int g = 0; g < nstage && !*abort_flag; ++g) {
        const int s = g % C::STAGES;
        if (g >= C::STAGES && !mbar_wait(&kv_empty[s], ((g / C::STAGES) - 1) & 1, abort_flag, a.status)) break;
        uint8_t* sk = skv + s * 2 * C::KV_BYTES;
        uint8_t* sv = sk + C::KV_BYTES;
        mbar_arrive_expect_tx(&kv_full[s], 2 * C::KV_BYTES);
#pragma unroll
        for (int pg = 0; pg < C::SK / 16; ++pg) {
          const int phys = pid_s[g * (C::SK / 16) + pg];
          int rk = a.pool_rows, rvw = a.pool_rows;  // outside the pool (past the tiles or the context): zero fill
          if (phys >= 0) {
            rk = a.layer_row0 + ((phys * 2) * a.Hkv + kvh) * 16;
            rvw = rk + a.Hkv * 16;
          }
#pragma unroll
          for (int c = 0; c < C::KB; ++c) {
            tma_load_3d(sk + c * C::HB + pg * 2048, &kvmap, &kv_full[s], 0, c, rk);
            tma_load_3d(sv + c * C::HB + pg * 2048, &kvmap, &kv_full[s], 0, c, rvw);
          }
        }
        issued = g + 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = umma_idesc_bf16(C::ROWS, C::SK);
      const uint32_t id_pv = umma_idesc_bf16(C::ROWS, HD) | (1u << 16);  // B (V) MN-major
      const uint32_t q_lo = sw128_desc_lo(smem_u32(sq));
      // S of stage g's two tiles, one chain of hd/16 K = 16 steps per element
      auto issue_s = [&](int g) -> bool {
        const int s = g % C::STAGES;
        if (!mbar_wait(&kv_full[s], (g / C::STAGES) & 1, abort_flag, a.status)) return false;
        tc_fence_after();
        const uint32_t k_lo = sw128_desc_lo(smem_u32(skv + s * 2 * C::KV_BYTES));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16_lo(tmem, q_lo + (kk >> 2) * (C::ROWS * 128 >> 4) + 2 * (kk & 3),
                       k_lo + (kk >> 2) * (C::HB >> 4) + 2 * (kk & 3), id_s, kk ? 1u : 0u);
        umma_commit(s_full);
        return true;
      };
      // O += P V of tile t: hi then lo per 16 keys, onto the rescaled O; P
      // from TMEM buffer t & 1, V from the tile's half of its stage
      auto issue_pv = [&](int t) -> bool {
        if (!mbar_wait(p_full, t & 1, abort_flag, a.status)) return false;
        tc_fence_after();
        const int s = (t >> 1) % C::STAGES;
        const uint32_t pt = tmem + C::P_COL + (t & 1) * C::BNK;  // hi: keys 2j, 2j + 1 in column j; lo BNK / 2 on
        const uint32_t v_lo = sw128_desc_lo_mn(
            smem_u32(skv + s * 2 * C::KV_BYTES + C::KV_BYTES + (t & 1) * C::BNK * 128), C::HB);
#pragma unroll
        for (int ks = 0; ks < C::BNK / 16; ++ks) {
          const uint32_t vk = v_lo + ks * (16 * 128 >> 4);
          umma_bf16_ta(tmem + C::O_COL, pt + 8 * ks, vk, id_pv, 1u);
          umma_bf16_ta(tmem + C::O_COL, pt + C::BNK / 2 + 8 * ks, vk, id_pv, 1u);
        }
        umma_commit(pv_done);
        if ((t & 1) || t == ntiles - 1) umma_commit(&kv_empty[s]);  // the stage's last reader
        return true;
      };
      if (mbar_wait(q_full, 0, abort_flag, a.status) && issue_s(0)) {
        for (int t = 0; t < ntiles; ++t) {
          if (!issue_pv(t)) break;
          // once the softmax threads have read this stage's second scores,
          // the next stage's S goes into the score columns
          if (!(t & 1) && (t >> 1) + 1 < nstage) {
            if (!mbar_wait(s_free, (t >> 1) & 1, abort_flag, a.status) || !issue_s((t >> 1) + 1)) break;
          }
        }
      }
      umma_commit(mma_done);
    }
  } else {
    // ---- softmax warps 2 .. NSW + 1: warp w holds CTA rows (TMEM lanes) 32 (w % 4) + 16 h .. + 15,
    // h = ((w - 2) / 4) % 2, and O's columns 128 hs .. + 127, hs = (w - 2) / 8, as an mma.sync m16n8 C
    // fragment: thread (g, t4) has rows g and g + 8, keys 8 j + 2 t4 + {0, 1}
    const int st = threadIdx.x - 64;  // 0 .. NS - 1
    {  // Q -> [hd block][row][64], 128-byte swizzle; zeros for rows past the block
      constexpr int CH = HD / 8;  // 16-byte chunks of a row
#pragma unroll
      for (int i = 0; i < C::ROWS * CH / C::NS; ++i) {
        const int idx = st + i * C::NS, qr = idx / CH, c16 = idx % CH;
        const int row = r0 + qr;
        const bool valid = row < rows;
        const int tok = row / G, hq = kvh * G + row % G;
        const uint4* qs = reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(q0 + tok) * a.Hq + hq) * HD);
        const uint4 v = valid ? qs[c16] : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sq + (c16 >> 3) * (C::ROWS * 128) + qr * 128 + (((c16 & 7) ^ (qr & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    const int lrow0 = 32 * (warp & 3) + 16 * (((warp - 2) >> 2) & 1);  // first CTA row of this warp
    const int ocol = C::O_COL + 128 * ((warp - 2) >> 3);             // first O column of this warp
    const bool writes_p = warp - 2 < 8;                              // one warp of a pair writes P and m, l
    const uint32_t frag = tmem + (static_cast<uint32_t>(lrow0) << 16);
    const int gq = lane >> 2, t4 = lane & 3;
    int pos[2], lo[2], tok[2], hq[2];
    bool valid[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = r0 + lrow0 + gq + 8 * r;
      valid[r] = row < rows;
      tok[r] = row / G;
      hq[r] = kvh * G + row % G;
      pos[r] = valid[r] ? cached + tok[r] : -1;
      lo[r] = valid[r] ? (a.window > 0 ? max(0, pos[r] - a.window + 1) : 0) : 1;
    }
    {  // O = +0, as the mma.sync kernel's accumulators start
      float z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0.f;
#pragma unroll
      for (int c = 0; c < C::OW / 32; ++c) tmem_st16x4(frag + ocol + 32 * c, z);
      tmem_wait_st();
    }
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    // A wait's outcome is made uniform over the warp before the warp-wide
    // TMEM accesses that follow it, so that a timeout never splits a warp.
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, a.status));
    };
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      if (!(t & 1)) {  // a new stage's scores
        if (!warp_wait(s_full, (t >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      float sv[16];  // s[j][e] = sv[4 j + e]
      tmem_ld16x4(frag + (t & 1) * C::BNK, sv);
      if ((t & 1) || t == ntiles - 1) {  // the stage's scores are all read
        tc_fence_before();
        mbar_arrive(s_free);
      }
      const int key0 = (tile_lo + t) * C::BNK;
      // every row of the warp sees every key of the tile: no masking (the
      // same values the masked path computes for visible keys)
      const bool full = __all_sync(0xffffffffu, lo[0] <= key0 && key0 + C::BNK - 1 <= pos[0] &&
                                                    lo[1] <= key0 && key0 + C::BNK - 1 <= pos[1]);
      float mx[2] = {-INFINITY, -INFINITY};
      if (full) {
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          mul2_rn(sv[i], sv[i + 1], a.scale_log2);
          mx[(i >> 1) & 1] = fmaxf(fmaxf(mx[(i >> 1) & 1], sv[i]), sv[i + 1]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = (i >> 1) & 1;
          const int key = key0 + (i >> 2) * 8 + t4 * 2 + (i & 1);
          sv[i] = (key >= lo[r] && key <= pos[r]) ? __fmul_rn(sv[i], a.scale_log2) : -INFINITY;
          mx[r] = fmaxf(mx[r], sv[i]);
        }
      }
      float mnew[2], alpha[2];
      bool rv[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        rv[r] = mx[r] != -INFINITY;
        mnew[r] = rv[r] ? fmaxf(m[r], mx[r]) : m[r];
        alpha[r] = rv[r] ? ex2(__fsub_rn(m[r], mnew[r])) : 1.0f;
      }
      // weights: hi = bf16(p), lo = bf16(p - hi) as bf16 pairs of keys (8 j + 2 t4, + 1); fp32 row sums
      uint32_t ph[4][2], pl[4][2];  // [j][row]
      float rs[2] = {0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float s0 = sv[4 * j + 2 * r], s1 = sv[4 * j + 2 * r + 1];
          float p0, p1;
          if (full) {  // every score finite, m' finite
            sub2_rn(s0, s1, mnew[r]);
            p0 = ex2(s0);
            p1 = ex2(s1);
          } else {
            p0 = s0 != -INFINITY ? ex2(__fsub_rn(s0, mnew[r])) : 0.f;
            p1 = s1 != -INFINITY ? ex2(__fsub_rn(s1, mnew[r])) : 0.f;
          }
          const uint32_t h = pack_bf16x2(p0, p1);
          ph[j][r] = h;
          pl[j][r] = pack_bf16x2(__fsub_rn(p0, bf16_lo(h)), __fsub_rn(p1, bf16_hi(h)));
          rs[r] = __fadd_rn(__fadd_rn(rs[r], p0), p1);
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        rs[r] = __fadd_rn(rs[r], __shfl_xor_sync(0xffffffffu, rs[r], 1));
        rs[r] = __fadd_rn(rs[r], __shfl_xor_sync(0xffffffffu, rs[r], 2));
        l[r] = rv[r] ? __fadd_rn(__fmul_rn(l[r], alpha[r]), rs[r]) : l[r];
        m[r] = mnew[r];
      }
      // P of this tile into TMEM buffer t & 1 (16x128b: thread (g, t4) column
      // 4x + t4, rows g and g + 8: hi pairs of keys 8x + 2 t4 in x < 4, lo pairs
      // after them).  The buffer's last reader, P V of tile t - 2, completed
      // before the previous tile's wait below.
      {
        uint32_t pw[16];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          pw[2 * x] = ph[x][0];
          pw[2 * x + 1] = ph[x][1];
          pw[8 + 2 * x] = pl[x][0];
          pw[8 + 2 * x + 1] = pl[x][1];
        }
        if (writes_p) tmem_st16x128x8(frag + C::P_COL + (t & 1) * C::BNK, pw);
      }
      if (t > 0) {  // P V of the previous tile has completed: O is free
        if (!warp_wait(pv_done, (t - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // O * alpha; alpha = 1 leaves O's bits as they are
        if (!__all_sync(0xffffffffu, alpha[0] == 1.0f && alpha[1] == 1.0f)) {
#pragma unroll
          for (int c = 0; c < C::OW / 32; ++c) {
            float o[16];
            tmem_ld16x4(frag + ocol + 32 * c, o);
#pragma unroll
            for (int i = 0; i < 16; i += 2) mul2_rn(o[i], o[i + 1], alpha[(i >> 1) & 1]);
            tmem_st16x4(frag + ocol + 32 * c, o);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok && warp_wait(pv_done, (ntiles - 1) & 1)) {
      tc_fence_after();
      // ---- split partial of every row that saw a key here
      float* po[2] = {nullptr, nullptr};  // this thread's columns of each stored row
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (!valid[r] || m[r] == -INFINITY) continue;
        const size_t base = (static_cast<size_t>(q0 + tok[r]) * a.Hq + hq[r]) * a.max_splits + sidx;
        if (t4 == 0 && writes_p) {
          a.part_ml[base * 2] = m[r];
          a.part_ml[base * 2 + 1] = l[r];
        }
        po[r] = a.part_o + base * HD + (ocol - C::O_COL) + 2 * t4;
      }
#pragma unroll
      for (int c = 0; c < C::OW / 32; ++c) {
        float o[16];
        tmem_ld16x4(frag + ocol + 32 * c, o);
#pragma unroll
        for (int r = 0; r < 2; ++r)
          if (po[r]) {
#pragma unroll
            for (int x = 0; x < 4; ++x)
              *reinterpret_cast<float2*>(po[r] + 32 * c + 8 * x) = make_float2(o[4 * x + 2 * r], o[4 * x + 2 * r + 1]);
          }
      }
    }
  }

  // Teardown: let in-flight copies land and issued MMAs finish, then free TMEM.
  if (warp == 0 && lane == 0 && *abort_flag)
    for (int g = max(0, issued - C::STAGES); g < issued; ++g) drain_wait(&kv_full[g % C::STAGES], (g / C::STAGES) & 1);
  if (warp == 1 && lane == 0) drain_wait(mma_done, 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int HD>
int launch_attn_tc_t(const CUtensorMap& kvmap, const AttnArgs& a, int n_items, cudaStream_t s) {
  using C = TcAttnCfg<HD>;
  static bool configured = false;
  if (!configured) {
    VD_CUDA_TRY(cudaFuncSetAttribute(attn_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
    configured = true;
  }
  VD_CUDA_TRY(launch_k(attn_tc_kernel<HD>, dim3(n_items), dim3(C::THREADS), C::SMEM, s, kvmap, a));
  return VD_OK;
}

}  // namespace

bool attn_tc_supported(int hd) { return hd == 64 || hd == 128 || hd == 256; }

int launch_attention_tc(const CUtensorMap& kvmap_tc, const AttnArgs& a, int hd, int n_items, cudaStream_t s) {
  if (n_items <= 0) return VD_OK;
  if (a.fold) return fail(VD_ERR_INVALID_ARG, "split folding is for decode-class CTAs");
  if (a.split > TcAttnCfg<128>::PIDS * 16)  // a CTA stages the ids of every page its split streams
    return fail(VD_ERR_INVALID_ARG, "KV split larger than the staged page ids");
  if (hd == 64) return launch_attn_tc_t<64>(kvmap_tc, a, n_items, s);
  if (hd == 128) return launch_attn_tc_t<128>(kvmap_tc, a, n_items, s);
  if (hd == 256) return launch_attn_tc_t<256>(kvmap_tc, a, n_items, s);
  return fail(VD_ERR_UNSUPPORTED, "the tcgen05 attention kernel takes head_dim 64, 128 or 256");
}

}  // namespace vd
