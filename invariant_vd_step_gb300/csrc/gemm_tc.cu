// Batch-invariant bf16 GEMM on 5th-generation tensor cores (tcgen05).
//
// acc[t][n] = sum_k X[t][k] * W[n][k], fp32 accumulation in TMEM.  The
// weight matrix is the MMA's A operand (BM = 64, 128 or 256 weight rows per
// tile, the last as two M = 128 instructions sharing each activation block)
// and the tokens are its N dimension (BN = 16 .. 256 per tile), so a decode
// batch streams each weight tile once per token tile.  Every output element
// is one chain of K = 16 MMA steps in ascending K order (4 per 64-wide K
// block, K blocks in order) into a zero-initialised accumulator, and no launch
// splits K: column t of D depends only on row t of X and on W, the matmul
// contract of 深入解析 Vosti §六 6.1 (row x of a batched run equals the singleton
// run bit for bit).  The tile shape is chosen per launch for speed; it sets
// the instruction's M and N, and tcgen05.mma computes each element of D the
// same way whatever M (64, 128) and N (16 .. 256) are, which the GPU tests
// check bitwise across all shapes.
//
// Warp roles (192 threads, one persistent CTA per SM): warp 0 issues TMA
// loads (one elected lane) and owns the TMEM allocation; warp 1 issues
// tcgen05.mma (one lane) into one of two TMEM accumulators; warps 2..5 read
// the other accumulator (warp w reaches lanes 32*(w%4)..+31; with BM = 64 the
// tile's rows sit in lanes 0..15 of each group of 32) and run the fused
// epilogue.  Every wait is bounded (see vd_device.cuh).
//
// A pipeline stage holds kpo K blocks: one weight copy of kpo x BM rows x 64
// (a 3-D or 4-D box, 8 to 64 KB; kpo = 1 for 256-row tiles) and kpo
// activation boxes of up to BN rows.
// Larger weight copies raise the rate at which one SM pulls a narrow matrix
// in; the ring (200 KB) holds as many stages as fit.  Rows of a B block past
// the activation box keep stale shared-memory contents, which only feed
// columns that are never stored (a column depends on its own row alone).
// The depth and the copy size change when copies are issued, never the MMA
// sequence.
#include <limits.h>
#include <math.h>

#include <cmath>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "vd_device.cuh"
#include "vd_internal.h"

namespace vd {
namespace {

constexpr int kMaxStages = 12;
constexpr int kThreads = 192;
constexpr int kRingBytes = 200 * 1024;
// Epilogue exchange: the sampling epilogue transposes each warp's 32 x 32
// block (4 x 32 x 33).
constexpr int kXchgFloats = 128 * 33;
constexpr int kSmemBytes = 1024 + kRingBytes + kXchgFloats * 4 + 256;
static_assert((2 * kMaxStages + 5) * 8 + 8 <= 256, "barrier block");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// bf16(a + b) of eight bf16 pairs (a, b exact in fp32; one rounding).
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
  return pack_bf16x2(__fadd_rn(bf16_lo(a), bf16_lo(b)), __fadd_rn(bf16_hi(a), bf16_hi(b)));
}
__device__ __forceinline__ uint4 add_bf16x8(uint4 a, uint4 b) {
  return make_uint4(add_bf16x2(a.x, b.x), add_bf16x2(a.y, b.y), add_bf16x2(a.z, b.z), add_bf16x2(a.w, b.w));
}

__device__ __forceinline__ float silu_f(float g) { return __fdiv_rn(g, __fadd_rn(1.0f, expf(-g))); }
__device__ __forceinline__ float gelu_tanh_f(float g) {
  const float g3 = __fmul_rn(__fmul_rn(g, g), g);
  const float inner = __fmul_rn(0.7978845608028654f, __fadd_rn(g, __fmul_rn(0.044715f, g3)));
  return __fmul_rn(__fmul_rn(0.5f, g), __fadd_rn(1.0f, tanhf(inner)));
}

// Epilogue of one tile: accumulator columns [c*32, c*32+32) are tokens
// t0.. of the tile.  TMEM lane 32*lg + i holds tile row lg*32 + i (BM = 128)
// or, for i < 16, tile row lg*16 + i (BM = 64).  A 256-row tile is two
// 128-row halves, the second one's accumulator BN columns further on.
template <int EPI>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& args, uint32_t tacc, int tile_t, int tile_n, int lg,
                                              int lane, float* xchg, int ksplit) {
  const int BM = args.bm, BN = args.bn;
  const int HM = BM > kGemmBM ? kGemmBM : BM;  // rows of one MMA half
  const int rpw = HM >> 2;            // tile rows per lane group and half
  const bool live = lane < rpw;       // lane holds a tile row
  for (int h = 0; h * HM < BM; ++h) {
    const int row = h * HM + lg * rpw + lane;  // tile row of this lane
    const uint32_t taddr = tacc + h * BN + (static_cast<uint32_t>(lg * 32) << 16);
    for (int c = 0; c * 32 < BN; ++c) {
      const int t0 = tile_t * BN + c * 32;
      if (t0 >= args.T) break;  // uniform over the four epilogue warps
      float v[32];
      tmem_ld32(taddr + c * 32, v);
      const int nt = min(min(32, BN - c * 32), args.T - t0);
      if (EPI == EPI_PARTIAL) {
        // fp32 partial of K split `ksplit`: part[ksplit][t][n], n the row of the
        // full output (gate rows then up rows for a GLU matrix)
        const int n = args.glu ? ((row & 1) ? args.glu_up_row : 0) + tile_n * (BM >> 1) + (row >> 1)
                               : tile_n * BM + row;
        float* out = static_cast<float*>(args.out) + (static_cast<size_t>(ksplit) * args.T) * args.ldo + n;
        if (live) {
  #pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nt) out[static_cast<size_t>(t0 + j) * args.ldo] = v[j];
        }
      } else if (EPI == EPI_F32) {
        float* out = static_cast<float*>(args.out) + tile_n * BM + row;
        if (live) {
  #pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nt) out[static_cast<size_t>(t0 + j) * args.ldo] = v[j];
        }
      } else if (EPI == EPI_F32_SAMPLE) {  // BM = 128 only
        if (args.out) {
          float* out = static_cast<float*>(args.out) + tile_n * BM + row;
  #pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nt) out[static_cast<size_t>(t0 + j) * args.ldo] = v[j];
        }
        // Transpose the warp's block (lane = vocabulary row, j = token) so that
        // lane j scans token t0 + j over the warp's 32 consecutive rows, one
        // Philox block per 4 rows, exactly as the standalone sampler does.
        float* xs = xchg + lg * 32 * 33;
  #pragma unroll
        for (int j = 0; j < 32; ++j) xs[lane * 33 + j] = v[j];
        __syncwarp();
        if (lane < nt) {
          const int t = t0 + lane;
          const vd_sampler sp = args.samp[t];
          const bool greedy = !(sp.temperature > 0.f);
          const int n0 = tile_n * BM + h * HM + lg * 32;
          float bv = -INFINITY;
          int bi = INT_MAX;
  #pragma unroll
          for (int r4 = 0; r4 < 32; r4 += 4) {
            float sc[4];
  #pragma unroll
            for (int q = 0; q < 4; ++q) sc[q] = xs[(r4 + q) * 33 + lane];
            if (!greedy) {
              const uint4 w = philox_block(sp.seed, sp.step, static_cast<uint32_t>((n0 + r4) >> 2));
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  #pragma unroll
              for (int q = 0; q < 4; ++q) sc[q] = gumbel_score(sc[q], ws[q], sp.temperature);
            }
  #pragma unroll
            for (int q = 0; q < 4; ++q)
              if (better(sc[q], n0 + r4 + q, bv, bi)) {
                bv = sc[q];
                bi = n0 + r4 + q;
              }
          }
          const size_t pi = static_cast<size_t>(t) * args.part_stride + tile_n * (BM / 32) + h * 4 + lg;
          args.part_v[pi] = bv;
          args.part_i[pi] = bi;
        }
        __syncwarp();
      } else if (EPI == EPI_BF16 || EPI == EPI_RESIDUAL) {
        // The warp's block (rpw feature rows x 32 tokens) is turned around in
        // shared memory so that each output row (one token's rpw features)
        // is written, and its residual read, as 16-byte vectors: a few wide
        // accesses instead of one 2-byte access per (feature, token).  The
        // staged value is bf16(acc) for EPI_BF16 and bf16_round(acc) for
        // EPI_RESIDUAL (exact in bf16), so each element's arithmetic is as
        // before: bf16(acc), or bf16(bf16_round(acc) + residual).
        __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(xchg) + lg * 32 * 32;  // [token][rpw]
        if (live) {
  #pragma unroll
          for (int j = 0; j < 32; ++j) xs[j * rpw + lane] = __float2bfloat16_rn(v[j]);
        }
        __syncwarp();
        const int lpr = rpw >> 3, tpp = 32 / lpr;  // lanes per output row, rows per pass
        const int f8 = (lane % lpr) * 8;
        const size_t col = static_cast<size_t>(tile_n) * BM + h * HM + lg * rpw + f8;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out) + col;
        uint4 val[4], rr[4];
  #pragma unroll
        for (int k = 0; k < 4; ++k) {  // tpp >= 8: at most four passes cover 32 tokens
          const int j = k * tpp + lane / lpr;
          if (j < nt) {
            val[k] = *reinterpret_cast<const uint4*>(xs + j * rpw + f8);
            if (EPI == EPI_RESIDUAL)  // the residual may alias the output: every load before any store
              rr[k] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(args.residual) + col +
                                                      static_cast<size_t>(t0 + j) * args.ldo);
          }
        }
  #pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = k * tpp + lane / lpr;
          if (j < nt) {
            if (EPI == EPI_RESIDUAL) val[k] = add_bf16x8(val[k], rr[k]);
            *reinterpret_cast<uint4*>(out + static_cast<size_t>(t0 + j) * args.ldo) = val[k];
          }
        }
        __syncwarp();  // the block's shared memory is rewritten by the next chunk
      } else {  // GLU: tile row 2f holds gate, 2f+1 up of feature f (the weight box interleaves them)
        // z = bf16(act(bf16(gate)) * bf16(up)) per (feature, token), staged
        // transposed in shared memory and written as 16-byte rows, as above.
        const bool gate_lane = live && (lane & 1) == 0;
        const int fpw = rpw >> 1;  // features per warp: 16 (128-row halves) or 8 (64-row tiles)
        __nv_bfloat16* zs = reinterpret_cast<__nv_bfloat16*>(xchg) + lg * 32 * 16;  // [token][fpw]
  #pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float u = __shfl_xor_sync(0xffffffffu, bf16_round(v[j]), 1);  // the neighbour's up value
          if (gate_lane && j < nt) {
            const float g = bf16_round(v[j]);
            const float a = (EPI == EPI_SWIGLU) ? silu_f(g) : gelu_tanh_f(g);
            zs[j * fpw + (lane >> 1)] = __float2bfloat16_rn(__fmul_rn(a, u));
          }
        }
        __syncwarp();
        const int lpr = fpw >> 3, tpp = 32 / lpr;  // lanes per output row, rows per pass
        const int f8 = (lane % lpr) * 8;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out) + tile_n * (BM >> 1) + h * (HM >> 1) +
                             lg * fpw + f8;
  #pragma unroll
        for (int k = 0; k < 2; ++k) {  // tpp >= 16: two passes cover 32 tokens
          const int j = k * tpp + lane / lpr;
          if (j < nt)
            *reinterpret_cast<uint4*>(out + static_cast<size_t>(t0 + j) * args.ldo) =
                *reinterpret_cast<const uint4*>(zs + j * fpw + f8);
        }
        __syncwarp();  // the block's shared memory is rewritten by the next chunk
      }
    }
  }  // halves
}

// What the MMA issuer needs from the kernel's set-up.
struct MmaLoop {
  uint8_t* ring;
  uint64_t *full, *empty, *acc_full, *acc_empty;
  volatile int* abort_flag;
  uint32_t tmem;
  int ntiles, nbuf, n_ops, KS;
  uint32_t idesc;
  int a_bytes, a_sub, b_sub;
};

// The MMA issuer (one thread).  For each of the CTA's tiles it takes an
// accumulator, then per stage waits for the stage's copies, issues its MMAs
// (KPO K blocks of four K = 16 steps; HALVES: both M = 128 halves of a
// 256-row tile per step) and releases the stage.  A stage is one straight
// run of MMAs whose descriptors advance by 32-bit adds: with few tokens per
// tile an MMA takes the tensor core about 45 cycles, so this thread's
// instructions between two MMAs, not the tensor core, would otherwise set
// the pace (vd_op_mma_issue_probe measures the instruction and the per-stage
// wait).  The MMAs, their operands and their order are those of the
// K-ascending chain described at the top of this file.
template <int KPO, bool HALVES>
__device__ __forceinline__ void mma_issuer(const GemmArgs& args, const MmaLoop& L) {
  const int S = args.stages, BN = args.bn;
  const uint32_t ring_lo = sw128_desc_lo(smem_u32(L.ring));
  const uint32_t st_step = static_cast<uint32_t>(args.stage_bytes) >> 4;  // one stage, 16-byte units
  const uint32_t b_off = static_cast<uint32_t>(L.a_bytes) >> 4;           // a stage's B blocks
  const uint32_t a_step = static_cast<uint32_t>(L.a_sub) >> 4, b_step = static_cast<uint32_t>(L.b_sub) >> 4;
  int i = 0, s = 0;
  uint32_t ph = 0, st_lo = ring_lo;
  for (int tile = blockIdx.x; tile < L.ntiles && !*L.abort_flag; tile += gridDim.x, ++i) {
    const int b = i % L.nbuf;
    if (i >= L.nbuf && !mbar_wait(&L.acc_empty[b], ((i / L.nbuf) - 1) & 1, L.abort_flag, args.status)) break;
    tc_fence_after();
    const uint32_t tacc = L.tmem + b * kGemmBN;
    const int split = tile % L.KS;
    const int op_end = (split + 1) * L.n_ops / L.KS;
    uint32_t acc = 0;  // the tile's first MMA starts from a zeroed accumulator
    for (int op = split * L.n_ops / L.KS; op < op_end; ++op) {
      if (!mbar_wait(&L.full[s], ph, L.abort_flag, args.status)) break;
      tc_fence_after();
      const uint32_t a_lo = st_lo, b_lo = st_lo + b_off;  // a K step of 16 elements: 32 bytes, 2 units
      if constexpr (HALVES) {  // rows 128..255 of the tile: A rows 16 KB on, accumulator BN columns on
#pragma unroll
        for (int kk = 0; kk < kGemmBK / 16; ++kk) {
          umma_bf16_lo(tacc, a_lo + 2 * kk, b_lo + 2 * kk, L.idesc, acc | kk);
          umma_bf16_lo(tacc + BN, a_lo + ((kGemmBM * 128) >> 4) + 2 * kk, b_lo + 2 * kk, L.idesc, acc | kk);
        }
      } else {
#pragma unroll
        for (int j = 0; j < KPO; ++j)
#pragma unroll
          for (int kk = 0; kk < kGemmBK / 16; ++kk)
            umma_bf16_lo(tacc, a_lo + j * a_step + 2 * kk, b_lo + j * b_step + 2 * kk, L.idesc, acc | j | kk);
      }
      acc = 1;
      umma_commit(&L.empty[s]);
      st_lo += st_step;
      if (++s == S) {
        s = 0;
        ph ^= 1u;
        st_lo = ring_lo;
      }
    }
    umma_commit(&L.acc_full[b]);
  }
}

// Persistent: CTA b handles tiles b, b + gridDim.x, ...; tile i = (token
// tile i % n_tok_tiles, weight tile i / n_tok_tiles), so CTAs working on the
// same weight tile at the same time share its reads through L2.  Two TMEM
// accumulators (2 x 256 columns) let the MMAs of one tile run while the
// epilogue warps drain the previous one; a tile that needs more than 256
// accumulator columns (256 rows x more than 128 tokens) has all 512 and the
// two overlap no longer.
template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap, GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int S = args.stages;
  uint8_t* ring = smem;
  float* xchg = reinterpret_cast<float*>(smem + kRingBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(xchg + kXchgFloats);
  uint64_t* empty = full + kMaxStages;
  uint64_t* acc_full = empty + kMaxStages;  // [2] MMAs of a tile done
  uint64_t* acc_empty = acc_full + 2;     // [2] epilogue finished reading
  uint64_t* mma_done = acc_empty + 2;     // every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // a GLU weight tile: gate and up rows of the same BM / 2 features, interleaved
  const bool kGlu = EPI == EPI_SWIGLU || EPI == EPI_GEGLU || (EPI == EPI_PARTIAL && args.glu);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BM = args.bm, BN = args.bn, kpo = args.kpo;
  const int nbuf = ((BM > kGemmBM ? 2 : 1) * BN <= kGemmBN) ? 2 : 1;  // accumulators that fit in TMEM
  const int n_ops = args.K / kGemmBK / kpo;  // stages per tile over the whole K
  const int ntt = (args.T + BN - 1) / BN;
  const int KS = args.k_splits;  // 1 on the invariant path
  const int ntiles = ntt * args.n_wtiles * KS;
  // tile -> (K split, token tile, weight tile); a split covers stages [op_lo, op_hi)
  auto op_lo = [&](int tile) { return (tile % KS) * n_ops / KS; };
  auto op_hi = [&](int tile) { return (tile % KS + 1) * n_ops / KS; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 128);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&xmap);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 2 * kGemmBN);
    tmem_relinquish();
  }
  // Once any bounded wait has given up, later CTAs skip their work instead
  // of each waiting out the limit (the status word reports the failure).  The
  // word is read before the wait for the previous kernel, so that its latency
  // hides behind that wait; a failure of the kernel right before this one is
  // then seen by the next kernel instead (every result after a failure is
  // discarded either way).
  __shared__ int skip;  // one read for the whole CTA keeps the exit uniform
  const int status_seen = (threadIdx.x == 0 && args.status) ? *reinterpret_cast<volatile int*>(args.status) : 0;
  // The prologue above touches no global memory but the status word; everything
  // below may read what the previous kernel of the stream writes.
  pdl_wait();
  if (threadIdx.x == 0) skip = status_seen;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();
  const uint32_t tmem = *tmem_slot;
  const int a_sub = BM * 128;            // one K block of A
  const int a_bytes = kpo * a_sub;       // B blocks follow the A blocks in a stage
  const int b_sub = args.b_sub;

  int issued = 0;  // producer: stages loaded so far (all tiles)
  if (skip) {
    // nothing issued: fall through to the teardown
  } else if (warp == 0) {
    if (lane == 0) {
      const uint32_t tx = static_cast<uint32_t>(kpo * (a_sub + args.b_box_rows * 128));
      int g = 0, s = 0;  // stage g lives in slot s = g % S, round g / S
      uint32_t ph = 0;     // parity of round g / S
      for (int tile = blockIdx.x; tile < ntiles && !*abort_flag; tile += gridDim.x) {
        const int tile_t = (tile / KS) % ntt, tile_n = (tile / KS) / ntt;
        for (int op = op_lo(tile); op < op_hi(tile); ++op, ++g) {
          if (g >= S && !mbar_wait(&empty[s], ph ^ 1u, abort_flag, args.status)) break;
          mbar_arrive_expect_tx(&full[s], tx);
          uint8_t* st = ring + s * args.stage_bytes;
          const int kb = op * kpo;
          if (kGlu)
            tma_load_4d(st, &wmap, &full[s], 0, 0, tile_n * (BM >> 1), kb);
          else
            tma_load_3d(st, &wmap, &full[s], 0, tile_n * BM, kb);
          for (int j = 0; j < kpo; ++j)
            tma_load_2d(st + a_bytes + j * b_sub, &xmap, &full[s], (kb + j) * kGemmBK, tile_t * BN);
          issued = g + 1;
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const int HM = BM > kGemmBM ? kGemmBM : BM;  // rows per MMA (a 256-row tile issues two)
      const MmaLoop L{ring, full, empty, acc_full, acc_empty, abort_flag, tmem, ntiles, nbuf, n_ops, KS,
                      umma_idesc_bf16(HM, BN), a_bytes, a_sub, b_sub};
      if (BM > kGemmBM)
        mma_issuer<1, true>(args, L);
      else if (kpo == 4)
        mma_issuer<4, false>(args, L);
      else if (kpo == 2)
        mma_issuer<2, false>(args, L);
      else
        mma_issuer<1, false>(args, L);
      umma_commit(mma_done);  // fires once every issued MMA has completed
    }
  } else {
    const int lg = warp & 3;  // TMEM lane group reachable by this warp
    int i = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
      const int b = i % nbuf;
      if (!mbar_wait(&acc_full[b], (i / nbuf) & 1, abort_flag, args.status)) break;
      tc_fence_after();
      epilogue_tile<EPI>(args, tmem + b * kGemmBN, (tile / KS) % ntt, (tile / KS) / ntt, lg, lane, xchg, tile % KS);
      tc_fence_before();
      mbar_arrive(&acc_empty[b]);
    }
  }

  // Teardown: let in-flight TMA copies land and issued MMAs finish, then
  // release TMEM.  On the normal path these waits return at once.
  if (warp == 0 && lane == 0 && *abort_flag) {
    for (int g = max(0, issued - S); g < issued; ++g) drain_wait(&full[g % S], (g / S) & 1);
  }
  if (!skip && warp == 1 && lane == 0) drain_wait(mma_done, 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kGemmBN);
  }
}

// Fast path: sum the K-split partials in split order and apply the epilogue
// the invariant path fuses into the GEMM (same roundings; only the sum's
// association differs).  One thread per output element.
template <int EPI>
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int KS, int T, int N,
                                     __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ res) {
  pdl_wait();
  pdl_trigger();
  constexpr bool kGluOut = EPI == EPI_SWIGLU || EPI == EPI_GEGLU;
  const int outN = kGluOut ? N / 2 : N;
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<size_t>(T) * outN) return;
  const int t = static_cast<int>(i / outN), n = static_cast<int>(i % outN);
  const size_t plane = static_cast<size_t>(T) * N;
  float acc = 0.f, up = 0.f;
  for (int k = 0; k < KS; ++k) {
    acc = __fadd_rn(acc, part[k * plane + static_cast<size_t>(t) * N + n]);
    if (kGluOut) up = __fadd_rn(up, part[k * plane + static_cast<size_t>(t) * N + outN + n]);
  }
  if (EPI == EPI_BF16) {
    out[i] = __float2bfloat16_rn(acc);
  } else if (EPI == EPI_RESIDUAL) {
    out[i] = __float2bfloat16_rn(__fadd_rn(bf16_round(acc), __bfloat162float(res[i])));
  } else {
    const float g = bf16_round(acc);
    const float a = (EPI == EPI_SWIGLU) ? silu_f(g) : gelu_tanh_f(g);
    out[i] = __float2bfloat16_rn(__fmul_rn(a, bf16_round(up)));
  }
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  }
  return n;
}

template <int EPI>
int launch_one(const CUtensorMap& wmap, const CUtensorMap& xmap, const GemmArgs& a, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    VD_CUDA_TRY(cudaFuncSetAttribute(gemm_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes));
    configured = true;
  }
  const int tiles = ((a.T + a.bn - 1) / a.bn) * a.n_wtiles * a.k_splits;
  VD_CUDA_TRY(launch_k(gemm_kernel<EPI>, dim3(std::min(tiles, sm_count())), dim3(kThreads), kSmemBytes, s, wmap, xmap,
                       a));
  return VD_OK;
}

// The forced plan as one word (bm | bn << 9 | kpo << 18), so that a host
// thread setting it never races a launching thread reading it.
std::atomic<uint32_t> g_forced{0};
std::atomic<unsigned> g_plan_epoch{0};

GemmPlan forced_plan() {
  const uint32_t v = g_forced.load();
  GemmPlan p;
  p.bm = static_cast<int>(v & 511u);
  p.bn = static_cast<int>((v >> 9) & 511u);
  p.kpo = static_cast<int>((v >> 18) & 7u);
  return p;
}

int ilog2(int x) {
  int l = 0;
  while ((1 << (l + 1)) <= x) ++l;
  return l;
}

// Pipeline layout of a plan: kpo is halved until at least two stages fit.
void layout(GemmArgs& a, int act_rows) {
  for (;;) {
    a.b_box_rows = std::min(a.bn, act_rows);
    a.b_sub = (a.bn * 128 + 1023) / 1024 * 1024;
    a.stage_bytes = a.kpo * (a.bm * 128 + a.b_sub);
    a.stages = std::min(kMaxStages, kRingBytes / a.stage_bytes);
    if (a.stages >= 2 || a.kpo == 1) break;
    a.kpo >>= 1;
  }
}

}  // namespace

namespace {

// Estimated time (us) of one launch under a plan.  The model only ranks
// plans; its constants were fitted to the measured times of every plan on the
// Llama-3.1-8B-shaped matrices (QKV, O, gate/up, down, LM head) at 1 .. 8192
// tokens, where it picks within 10 % of the fastest plan everywhere.  A
// pipeline stage costs the longest of: its copies (a fixed issue cost per
// copy, or the copy's bytes at the per-SM fill rate), its MMAs (an N <= 32
// instruction takes about 49 cycles, N = 256 about 136), and the latency of a
// copy-and-MMA round trip shared by the stages in flight.  A launch costs its
// tiles' stages over the SMs, and at least the weights' bytes at HBM speed.
double plan_cost(int bm, int bn, int kpo, int T, int rows, int K, int ks) {
  constexpr double kCopyUs = 0.3, kActCopyUs = 0.05, kFillGBs = 60.0, kLatencyUs = 3.0, kTileUs = 0.5;
  constexpr double kExposedEpilogueUs = 2.0;  // per tile, when one accumulator fills TMEM
  constexpr double kClockMHz = 2070.0, kHbmGBs = 6800.0;
  int stage = 0, S = 0;
  for (;;) {
    stage = kpo * (bm * 128 + (bn * 128 + 1023) / 1024 * 1024);
    S = std::min(kMaxStages, kRingBytes / stage);
    if (S >= 2 || kpo == 1) break;
    kpo >>= 1;
  }
  if (S < 2) return 1e30;
  int bucket = 1;
  while (bucket < T) bucket <<= 1;
  const int brows = std::min(bn, bucket);
  const double tiles = static_cast<double>(rows / bm) * ((T + bn - 1) / bn) * ks;
  const double per_sm = std::ceil(tiles / sm_count());
  const double mma_clk = std::max(49.0, 136.0 * bn / 256) * (bm > kGemmBM ? 2 : 1);
  const double t_mma = 4.0 * kpo * mma_clk / kClockMHz;
  const double t_copy = std::max(kCopyUs, kpo * bm * 128 / kFillGBs / 1e3) +
                        kpo * std::max(kActCopyUs, brows * 128 / kFillGBs / 1e3);
  const double t_lat = (kLatencyUs + t_mma) / S;
  const double t_stage = std::max({t_copy, t_lat, t_mma});
  const double stages_per_tile = static_cast<double>(K / kGemmBK) / kpo / ks;
  const double t_hbm = static_cast<double>(rows) * K * 2 / kHbmGBs / 1e3;
  const bool one_acc = (bm > kGemmBM ? 2 : 1) * bn > kGemmBN;
  return std::max(per_sm * (stages_per_tile * t_stage + kTileUs + (one_acc ? kExposedEpilogueUs : 0)), t_hbm);
}

}  // namespace

namespace {
// Set when the shape self-check saw two tile shapes give different bits:
// every later launch then takes the one fixed shape below.
std::atomic<bool> g_shapes_pinned{false};
constexpr GemmPlan kPinnedPlan{128, 256, 1};
}  // namespace

GemmPlan gemm_plan(const WeightMaps& w, int T, int epi, int k_splits) {
  if (g_shapes_pinned.load() && k_splits == 1) return kPinnedPlan;
  const int KB = w.K / kGemmBK;
  const bool bm64_ok = epi != EPI_F32_SAMPLE && w.rows % 64 == 0 && (!w.glu || (w.rows / 2) % 32 == 0);
  int top = 16;  // no wider token tile than the activation bucket needs
  while (top < T && top < kGemmBN) top <<= 1;
  // 256-row tiles fill TMEM with one accumulator, so the epilogue no longer
  // overlaps the next tile's MMAs; measured, they pay off only for the LM
  // head's light fp32 epilogue at 512 tokens and more (about 16 % faster
  // there), and are chosen only then (a forced plan may take them anywhere).
  const bool bm256_ok = k_splits == 1 && w.rows % 256 == 0;
  const bool bm256_auto = bm256_ok && T >= 512 && (epi == EPI_F32 || epi == EPI_F32_SAMPLE);
  GemmPlan p;
  double best = 0;
  for (int bm : {kGemmBM, kGemmBM / 2, 2 * kGemmBM}) {
    if ((bm == kGemmBM / 2 && !bm64_ok) || (bm == 2 * kGemmBM && !bm256_auto)) continue;
    if (w.rows % bm) continue;
    for (int bn = 16; bn <= top; bn <<= 1)
      for (int kpo = 1; kpo <= 4; kpo <<= 1) {
        if (KB % kpo || (k_splits > 1 && kpo > 1) || (bm > kGemmBM && kpo > 1)) continue;
        const double c = plan_cost(bm, bn, kpo, T, w.rows, w.K, k_splits);
        if (p.bm == 0 || c < best) {
          best = c;
          p.bm = bm;
          p.bn = bn;
          p.kpo = kpo;
        }
      }
  }
  const GemmPlan f = forced_plan();
  if (f.bm == 128 || (f.bm == 64 && bm64_ok) || (f.bm == 256 && bm256_ok)) p.bm = f.bm;
  if (f.bn) p.bn = f.bn;
  if (f.kpo && k_splits == 1 && KB % f.kpo == 0) p.kpo = f.kpo;
  if (p.bm > kGemmBM) p.kpo = 1;  // 256-row tiles copy one K block at a time
  return p;
}

int set_forced_gemm_plan(GemmPlan p) {
  if ((p.bm != 0 && p.bm != 64 && p.bm != 128 && p.bm != 256) || (p.bn != 0 && (p.bn < 16 || p.bn > kGemmBN || (p.bn & (p.bn - 1)))) ||
      (p.kpo != 0 && p.kpo != 1 && p.kpo != 2 && p.kpo != 4))
    return fail(VD_ERR_INVALID_ARG,
                "GEMM plan: bm in {0, 64, 128, 256}, bn in {0, 16 .. 256} (a power of two), kpo in {0, 1, 2, 4}");
  const uint32_t v = static_cast<uint32_t>(p.bm) | static_cast<uint32_t>(p.bn) << 9 |
                     static_cast<uint32_t>(p.kpo) << 18;
  if (g_forced.exchange(v) != v) ++g_plan_epoch;  // captured step graphs stay valid for an unchanged plan
  return VD_OK;
}

unsigned gemm_plan_epoch() { return g_plan_epoch.load(); }

int launch_splitk_reduce(const float* part, int k_splits, int T, int N, int epi, void* out, const void* residual,
                         cudaStream_t s) {
  if (T <= 0) return VD_OK;
  const int outN = (epi == EPI_SWIGLU || epi == EPI_GEGLU) ? N / 2 : N;
  const dim3 grid(static_cast<unsigned>((static_cast<size_t>(T) * outN + 255) / 256));
  auto* o = static_cast<__nv_bfloat16*>(out);
  const auto* r = static_cast<const __nv_bfloat16*>(residual);
  switch (epi) {
    case EPI_BF16: VD_CUDA_TRY(launch_k(splitk_reduce_kernel<EPI_BF16>, grid, dim3(256), 0, s, part, k_splits, T, N, o, r)); break;
    case EPI_RESIDUAL: VD_CUDA_TRY(launch_k(splitk_reduce_kernel<EPI_RESIDUAL>, grid, dim3(256), 0, s, part, k_splits, T, N, o, r)); break;
    case EPI_SWIGLU: VD_CUDA_TRY(launch_k(splitk_reduce_kernel<EPI_SWIGLU>, grid, dim3(256), 0, s, part, k_splits, T, N, o, r)); break;
    case EPI_GEGLU: VD_CUDA_TRY(launch_k(splitk_reduce_kernel<EPI_GEGLU>, grid, dim3(256), 0, s, part, k_splits, T, N, o, r)); break;
    default: return fail(VD_ERR_INVALID_ARG, "split-K reduction epilogue");
  }
  return VD_OK;
}

namespace {
int launch_gemm_plan(const WeightMaps& w, const ActMaps& x, const GemmArgs& a0, int epi, const GemmPlan* plan,
                     cudaStream_t s) {
  if (a0.T <= 0) return VD_OK;
  GemmArgs a = a0;
  if (a.k_splits < 1) a.k_splits = 1;
  if ((a.k_splits > 1) != (epi == EPI_PARTIAL) || a.k_splits > a.K / kGemmBK)
    return fail(VD_ERR_INVALID_ARG, "K splits need the partial epilogue and at most one split per K block");
  if (a.K != w.K || x.rows < 1 || !x.maps) return fail(VD_ERR_INVALID_ARG, "GEMM operand shapes");
  const GemmPlan p = plan ? *plan : gemm_plan(w, a.T, epi, a.k_splits);
  a.bm = p.bm;
  a.bn = p.bn;
  a.kpo = p.kpo;
  layout(a, x.rows);
  if (a.stages < 2 || w.rows % a.bm || (a.K / kGemmBK) % a.kpo || (a.k_splits > 1 && a.kpo != 1))
    return fail(VD_ERR_INVALID_ARG, "GEMM plan does not fit the matrix");
  a.n_wtiles = w.rows / a.bm;
  const CUtensorMap& wm = w.m[a.bm == 64 ? 1 : a.bm == 256 ? 2 : 0][ilog2(a.kpo)];
  const CUtensorMap& xm = x.maps[ilog2(a.bn / 16)];
  switch (epi) {
    case EPI_BF16: return launch_one<EPI_BF16>(wm, xm, a, s);
    case EPI_RESIDUAL: return launch_one<EPI_RESIDUAL>(wm, xm, a, s);
    case EPI_F32: return launch_one<EPI_F32>(wm, xm, a, s);
    case EPI_PARTIAL: return launch_one<EPI_PARTIAL>(wm, xm, a, s);
    case EPI_F32_SAMPLE:
      if (!a.samp || !a.part_v || !a.part_i) return fail(VD_ERR_INVALID_ARG, "sampling epilogue without buffers");
      return launch_one<EPI_F32_SAMPLE>(wm, xm, a, s);
    case EPI_SWIGLU: return launch_one<EPI_SWIGLU>(wm, xm, a, s);
    case EPI_GEGLU: return launch_one<EPI_GEGLU>(wm, xm, a, s);
    default: return fail(VD_ERR_INVALID_ARG, "unknown GEMM epilogue");
  }
}

// Seeded bf16 test operands in [-2, 2): a 32-bit integer hash of the index.
__global__ void fill_probe_kernel(__nv_bfloat16* p, int n, uint32_t seed) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  uint32_t h = static_cast<uint32_t>(i) * 0x9E3779B1u ^ seed;
  h ^= h >> 15;
  h *= 0x2C1B3C6Du;
  h ^= h >> 12;
  h *= 0x297A2D39u;
  h ^= h >> 15;
  p[i] = __float2bfloat16_rn(static_cast<float>(static_cast<int>(h >> 8) - (1 << 23)) * (2.0f / (1 << 23)));
}
}  // namespace

int launch_gemm(const WeightMaps& w, const ActMaps& x, const GemmArgs& a0, int epi, cudaStream_t s) {
  return launch_gemm_plan(w, x, a0, epi, nullptr, s);
}

int gemm_shapes_self_check(int* result) {
  // The tile shape is chosen per launch because tcgen05.mma computes an
  // element of D the same way whatever the instruction's M and N: a
  // property of the hardware, measured, not documented.  Once per device,
  // before any step runs, compare the raw fp32 accumulators of every tile
  // shape on seeded operands (40 tokens, 256 rows, K = 512: several token
  // tiles at every width, a ragged last one); if any bit differs, pin every
  // later launch to one fixed shape.
  constexpr int kMaxDev = 64, T = 40, N = 256, K = 512;
  static std::mutex mu;
  static int state[kMaxDev];
  static bool init = false;
  int dev = 0;
  VD_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDev) return fail(VD_ERR_UNSUPPORTED, "device ordinal too large");
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (int& v : state) v = -1;
    init = true;
  }
  if (state[dev] >= 0) {
    *result = state[dev];
    return VD_OK;
  }
  const GemmPlan plans[] = {{128, 256, 1}, {64, 16, 4}, {64, 64, 2}, {128, 16, 1}, {128, 32, 4},
                            {128, 64, 2},  {128, 128, 1}, {256, 64, 1}, {256, 256, 1}};
  constexpr int kPlans = sizeof(plans) / sizeof(plans[0]);
  __nv_bfloat16 *A = nullptr, *W = nullptr;
  float* C = nullptr;
  int rc = VD_OK;
  auto cleanup = [&] {
    cudaFree(A);
    cudaFree(W);
    cudaFree(C);
  };
  if (cudaMalloc(&A, sizeof(__nv_bfloat16) * T * K) != cudaSuccess ||
      cudaMalloc(&W, sizeof(__nv_bfloat16) * N * K) != cudaSuccess ||
      cudaMalloc(&C, sizeof(float) * kPlans * T * N) != cudaSuccess) {
    cleanup();
    return fail(VD_ERR_CUDA, "GEMM shape self-check: allocation failed");
  }
  fill_probe_kernel<<<(T * K + 255) / 256, 256>>>(A, T * K, 0x1234567u);
  fill_probe_kernel<<<(N * K + 255) / 256, 256>>>(W, N * K, 0x89ABCDEu);
  WeightMaps wm;
  CUtensorMap xm[kNumBn];
  if ((rc = make_weight_maps(&wm, W, N, K, false))) {
    cleanup();
    return rc;
  }
  for (int i = 0; i < kNumBn && !rc; ++i) rc = make_map_2d(&xm[i], A, T, K, std::min(T, 16 << i));
  ActMaps xv;
  xv.maps = xm;
  xv.rows = T;
  for (int p = 0; p < kPlans && !rc; ++p) {
    GemmArgs g{};
    g.out = C + static_cast<size_t>(p) * T * N;
    g.T = T;
    g.K = K;
    g.ldo = N;
    g.glu_up_row = N;
    rc = launch_gemm_plan(wm, xv, g, EPI_F32, &plans[p], nullptr);
  }
  std::vector<float> h(static_cast<size_t>(kPlans) * T * N);
  if (!rc && cudaMemcpy(h.data(), C, sizeof(float) * h.size(), cudaMemcpyDeviceToHost) != cudaSuccess)
    rc = fail(VD_ERR_CUDA, "GEMM shape self-check: copy failed");
  cleanup();
  if (rc) return rc;
  bool same = true;
  for (int p = 1; p < kPlans && same; ++p)
    same = std::memcmp(h.data(), h.data() + static_cast<size_t>(p) * T * N, sizeof(float) * T * N) == 0;
  state[dev] = same ? 1 : 0;
  if (!same && !g_shapes_pinned.exchange(true)) ++g_plan_epoch;
  *result = state[dev];
  return VD_OK;
}

}  // namespace vd
