// Prefill-class paged attention on 5th-generation tensor cores (tcgen05),
// head dimensions 64 and 128.
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
// Roles (320 threads): warp 0 allocates TMEM and one lane issues the K/V
// page copies (3-D TMA boxes of one page and 64 head dims, so that a K or V
// tile is [hd block][32 keys][64] with the 128-byte swizzle, the canonical
// operand layout); warp 1, one lane, issues the MMAs; warps 2..9 each hold
// 16 rows, read from TMEM in the layout of an mma.sync C fragment (two rows
// and eight keys per thread), and run the softmax, the O rescale and the
// epilogue with the mma.sync kernel's per-row code.  TMEM: two 32-column score buffers, so that S of the next
// tile is computed while this tile's softmax runs, and hd columns of O.
// P (hi | lo, 128 bytes a row) goes through shared memory as the A operand
// of P V; V is the MN-major B operand.  Every wait is bounded.
#include <math.h>

#include "vd_device.cuh"
#include "vd_internal.h"

namespace vd {
namespace {

template <int HD>
struct TcAttnCfg {
  static constexpr int ROWS = 128;                 // rows per CTA (MMA M)
  static constexpr int BNK = 32;                   // keys per tile, as in every attention kernel
  static constexpr int KB = HD / 64;               // 64-wide head-dim blocks
  static constexpr int Q_BYTES = KB * ROWS * 128;  // [hd block][row][64]
  static constexpr int TILE_BYTES = BNK * HD * 2;  // K or V: [hd block][key][64]
  static constexpr int HALF_BYTES = BNK * 128;     // one hd block of a tile
  static constexpr int P_BYTES = ROWS * 128;       // [row][hi 32 | lo 32]
  static constexpr int STAGES = 3;
  static constexpr int O_COL = 2 * BNK;            // TMEM: S buffers at 0 and BNK, O after them
  static constexpr int TMEM_COLS = 2 * BNK + HD <= 128 ? 128 : 256;
  static constexpr int SMEM = 1024 + Q_BYTES + STAGES * 2 * TILE_BYTES + P_BYTES + 256;
  // At most 512 / TMEM_COLS CTAs may share an SM (a CTA that found too few
  // TMEM columns would wait in tcgen05.alloc); shared memory bounds it.
  static constexpr int CTAS_PER_SM = (228 * 1024) / (SMEM + 1024);
  static_assert(CTAS_PER_SM * TMEM_COLS <= 512, "TMEM columns per SM");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

template <int HD>
__global__ void __launch_bounds__(320, 2) attn_tc_kernel(const __grid_constant__ CUtensorMap kvmap, AttnArgs a) {
  using C = TcAttnCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sq = smem;
  uint8_t* skv = sq + C::Q_BYTES;  // stage s: K at skv + s * 2 * TILE_BYTES, V right after
  uint8_t* sp = skv + C::STAGES * 2 * C::TILE_BYTES;
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(sp + C::P_BYTES);
  uint64_t* kv_empty = kv_full + C::STAGES;
  uint64_t* s_full = kv_empty + C::STAGES;  // [2] S of a tile is in its buffer
  uint64_t* s_free = s_full + 2;            // [2] the softmax threads have read it
  uint64_t* p_full = s_free + 2;            // P written and O rescaled
  uint64_t* pv_done = p_full + 1;           // the tile's P V steps completed
  uint64_t* q_full = pv_done + 1;           // Q rows in shared memory
  uint64_t* mma_done = q_full + 1;          // every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

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

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 256);
    }
    mbar_init(p_full, 256);
    mbar_init(pv_done, 1);
    mbar_init(q_full, 256);
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

  int issued = 0;  // producer: tiles whose copies were issued
  if (warp == 0) {
    if (lane == 0) {
      for (int g = 0; g < ntiles && !*abort_flag; ++g) {
        const int s = g % C::STAGES;
        if (g >= C::STAGES && !mbar_wait(&kv_empty[s], ((g / C::STAGES) - 1) & 1, abort_flag, a.status)) break;
        uint8_t* sk = skv + s * 2 * C::TILE_BYTES;
        uint8_t* sv = sk + C::TILE_BYTES;
        mbar_arrive_expect_tx(&kv_full[s], 2 * C::TILE_BYTES);
        const int lp0 = ((tile_lo + g) * C::BNK) >> 4;
#pragma unroll
        for (int pg = 0; pg < C::BNK / 16; ++pg) {
          const int lp = lp0 + pg;
          int rk = a.pool_rows, rvw = a.pool_rows;  // outside the pool: zero fill
          if (lp * 16 < kv_len) {
            const int phys = a.page_table[static_cast<size_t>(b) * a.pt_stride + lp];
            rk = a.layer_row0 + ((phys * 2) * a.Hkv + kvh) * 16;
            rvw = rk + a.Hkv * 16;
          }
#pragma unroll
          for (int c = 0; c < C::KB; ++c) {
            tma_load_3d(sk + c * C::HALF_BYTES + pg * 2048, &kvmap, &kv_full[s], 0, c, rk);
            tma_load_3d(sv + c * C::HALF_BYTES + pg * 2048, &kvmap, &kv_full[s], 0, c, rvw);
          }
        }
        issued = g + 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = umma_idesc_bf16(C::ROWS, C::BNK);
      const uint32_t id_pv = umma_idesc_bf16(C::ROWS, HD) | (1u << 16);  // B (V) MN-major
      const uint32_t q_lo = sw128_desc_lo(smem_u32(sq));
      const uint32_t p_lo = sw128_desc_lo(smem_u32(sp));
      // S of tile t into score buffer t & 1
      auto issue_s = [&](int t) -> bool {
        const int s = t % C::STAGES, sb = t & 1;
        if (!mbar_wait(&kv_full[s], (t / C::STAGES) & 1, abort_flag, a.status)) return false;
        if (t >= 2 && !mbar_wait(&s_free[sb], ((t >> 1) - 1) & 1, abort_flag, a.status)) return false;
        tc_fence_after();
        const uint32_t k_lo = sw128_desc_lo(smem_u32(skv + s * 2 * C::TILE_BYTES));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16_lo(tmem + sb * C::BNK, q_lo + (kk >> 2) * (C::ROWS * 128 >> 4) + 2 * (kk & 3),
                       k_lo + (kk >> 2) * (C::HALF_BYTES >> 4) + 2 * (kk & 3), id_s, kk ? 1u : 0u);
        umma_commit(&s_full[sb]);
        return true;
      };
      // O += P V of tile t: hi then lo per 16 keys, onto the rescaled O
      auto issue_pv = [&](int t) -> bool {
        if (!mbar_wait(p_full, t & 1, abort_flag, a.status)) return false;
        tc_fence_after();
        const int s = t % C::STAGES;
        const uint32_t v_lo = sw128_desc_lo_mn(smem_u32(skv + s * 2 * C::TILE_BYTES + C::TILE_BYTES), C::HALF_BYTES);
#pragma unroll
        for (int ks = 0; ks < C::BNK / 16; ++ks) {
          const uint32_t vk = v_lo + ks * (16 * 128 >> 4);
          umma_bf16_lo(tmem + C::O_COL, p_lo + 2 * ks, vk, id_pv, 1u);
          umma_bf16_lo(tmem + C::O_COL, p_lo + 4 + 2 * ks, vk, id_pv, 1u);
        }
        umma_commit(&kv_empty[s]);
        umma_commit(pv_done);
        return true;
      };
      if (mbar_wait(q_full, 0, abort_flag, a.status) && issue_s(0)) {
        for (int t = 0; t < ntiles; ++t) {
          if (t + 1 < ntiles && !issue_s(t + 1)) break;
          if (!issue_pv(t)) break;
        }
      }
      umma_commit(mma_done);
    }
  } else {
    // ---- softmax warps 2..9: warp w holds CTA rows (TMEM lanes) 32 (w % 4) + 16 h .. + 15, h = (w - 2) / 4,
    // as an mma.sync m16n8 C fragment: thread (g, t4) has rows g and g + 8, keys 8 j + 2 t4 + {0, 1}
    const int st = threadIdx.x - 64;  // 0..255
    {  // Q -> [hd block][row][64], 128-byte swizzle; zeros for rows past the block.  Two threads a row.
      const int qr = st >> 1, half = st & 1;
      const int row = r0 + qr;
      const bool valid = row < rows;
      const int tok = row / G, hq = kvh * G + row % G;
      const uint4* qs = reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(q0 + tok) * a.Hq + hq) * HD);
#pragma unroll
      for (int i = 0; i < HD / 16; ++i) {
        const int c16 = half * (HD / 16) + i;
        const uint4 v = valid ? qs[c16] : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sq + (c16 >> 3) * (C::ROWS * 128) + qr * 128 + (((c16 & 7) ^ (qr & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    const int lrow0 = 32 * (warp & 3) + 16 * ((warp - 2) >> 2);  // first CTA row of this warp
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
      for (int c = 0; c < HD / 32; ++c) tmem_st16x4(frag + C::O_COL + 32 * c, z);
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
      const int sb = t & 1;
      if (!warp_wait(&s_full[sb], (t >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[16];  // s[j][e] = sv[4 j + e]
      tmem_ld16x4(frag + sb * C::BNK, sv);
      tc_fence_before();
      mbar_arrive(&s_free[sb]);
      const int key0 = (tile_lo + t) * C::BNK;
      // every row of the warp sees every key of the tile: no masking (the
      // same values the masked path computes for visible keys)
      const bool full = __all_sync(0xffffffffu, lo[0] <= key0 && key0 + C::BNK - 1 <= pos[0] &&
                                                    lo[1] <= key0 && key0 + C::BNK - 1 <= pos[1]);
      float mx[2] = {-INFINITY, -INFINITY};
      if (full) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          sv[i] = __fmul_rn(sv[i], a.scale_log2);
          mx[(i >> 1) & 1] = fmaxf(mx[(i >> 1) & 1], sv[i]);
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
          const float s0 = sv[4 * j + 2 * r], s1 = sv[4 * j + 2 * r + 1];
          const float p0 = (full || s0 != -INFINITY) ? ex2(__fsub_rn(s0, mnew[r])) : 0.f;
          const float p1 = (full || s1 != -INFINITY) ? ex2(__fsub_rn(s1, mnew[r])) : 0.f;
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
      if (t > 0) {  // P V of the previous tile has completed: O and the P buffer are free
        if (!warp_wait(pv_done, (t - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        uint8_t* prow = sp + (lrow0 + gq + 8 * r) * 128 + t4 * 4;  // row & 7 == gq
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          *reinterpret_cast<uint32_t*>(prow + ((j ^ gq) << 4)) = ph[j][r];
          *reinterpret_cast<uint32_t*>(prow + (((4 + j) ^ gq) << 4)) = pl[j][r];
        }
      }
      // O * alpha; alpha = 1 leaves O's bits as they are, and so does any
      // alpha on the first tile (O is +0)
      if (t > 0 && !__all_sync(0xffffffffu, alpha[0] == 1.0f && alpha[1] == 1.0f)) {
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          float o[16];
          tmem_ld16x4(frag + C::O_COL + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = __fmul_rn(o[i], alpha[(i >> 1) & 1]);
          tmem_st16x4(frag + C::O_COL + 32 * c, o);
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
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
        if (t4 == 0) {
          a.part_ml[base * 2] = m[r];
          a.part_ml[base * 2 + 1] = l[r];
        }
        po[r] = a.part_o + base * HD + 2 * t4;
      }
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        float o[16];
        tmem_ld16x4(frag + C::O_COL + 32 * c, o);
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
  VD_CUDA_TRY(launch_k(attn_tc_kernel<HD>, dim3(n_items), dim3(320), C::SMEM, s, kvmap, a));
  return VD_OK;
}

}  // namespace

bool attn_tc_supported(int hd) { return hd == 64 || hd == 128; }

int launch_attention_tc(const CUtensorMap& kvmap_tc, const AttnArgs& a, int hd, int n_items, cudaStream_t s) {
  if (n_items <= 0) return VD_OK;
  if (a.fold) return fail(VD_ERR_INVALID_ARG, "split folding is for decode-class CTAs");
  if (hd == 64) return launch_attn_tc_t<64>(kvmap_tc, a, n_items, s);
  if (hd == 128) return launch_attn_tc_t<128>(kvmap_tc, a, n_items, s);
  return fail(VD_ERR_UNSUPPORTED, "the tcgen05 attention kernel takes head_dim 64 or 128");
}

}  // namespace vd
