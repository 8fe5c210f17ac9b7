// Token choice: greedy argmax (lowest index among equal maxima) and seeded
// Gumbel-max sampling, argmax_i(l_i / T + G_i) with G_i = -log(-log(u_i)).
//
// The uniforms come from the counter-based Philox4x32-10 generator of
// Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2,
// 3" (SC'11), implemented here from that definition.  For vocabulary index
// i at sampler state (seed, step): key = (seed lo, seed hi), counter =
// (i / 4, step lo, step hi, 0x5644), word i % 4 of the block, and
// u = ((word >> 8) + 0.5) * 2^-24 (exact in fp32, never 0 or 1).  The
// sampler state is the per-request "sampler_0" of 深入解析 Vosti §二
// Definition 2.1.
//
// The reduction picks the unique (largest value, lowest index) pair, which
// no evaluation order can change, so the result is fixed by the row alone.
#include <limits.h>
#include <math.h>

#include "vd_device.cuh"
#include "vd_internal.h"

namespace vd {
namespace {

// Pass 1: CTA (row, chunk) picks the best (score, index) among kSampleChunk
// consecutive vocabulary entries with 16-byte loads.  Pass 2: one CTA per
// row picks among the chunk winners.  Both passes select the unique
// (largest score, lowest index) pair, so the split changes nothing.
constexpr int kSampleThreads = 256;
constexpr int kSampleChunk = kSampleThreads * 32;

__device__ __forceinline__ void warp_best(float& bv, int& bi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
}

__global__ void __launch_bounds__(kSampleThreads) sample_partial_kernel(const float* __restrict__ logits, int V,
                                                                       const vd_sampler* __restrict__ params,
                                                                       float* __restrict__ part_v,
                                                                       int* __restrict__ part_i) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, chunk = blockIdx.y;
  const float4* l4 = reinterpret_cast<const float4*>(logits + static_cast<size_t>(r) * V);
  const vd_sampler sp = params[r];
  const bool greedy = !(sp.temperature > 0.f);
  float bv = -INFINITY;
  int bi = INT_MAX;
  const int blk0 = chunk * (kSampleChunk / 4);
  const int nblk = min(kSampleChunk / 4, V / 4 - blk0);
  constexpr int kPer = kSampleChunk / 4 / kSampleThreads;  // float4 loads per thread, all issued first
  float4 xs[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int k = threadIdx.x + q * kSampleThreads;
    if (k < nblk) xs[q] = l4[blk0 + k];
  }
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int k = threadIdx.x + q * kSampleThreads;
    if (k >= nblk) break;
    const int blk = blk0 + k;
    const float4 x = xs[q];
    float v[4] = {x.x, x.y, x.z, x.w};
    if (!greedy) {
      const uint4 w = philox_block(sp.seed, sp.step, static_cast<uint32_t>(blk));
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = gumbel_score(v[j], ws[j], sp.temperature);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (better(v[j], blk * 4 + j, bv, bi)) {
        bv = v[j];
        bi = blk * 4 + j;
      }
  }
  warp_best(bv, bi);
  __shared__ float sv[kSampleThreads / 32];
  __shared__ int si[kSampleThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    bv = lane < kSampleThreads / 32 ? sv[lane] : -INFINITY;
    bi = lane < kSampleThreads / 32 ? si[lane] : INT_MAX;
    warp_best(bv, bi);
    if (lane == 0) {
      part_v[static_cast<size_t>(r) * gridDim.y + chunk] = bv;
      part_i[static_cast<size_t>(r) * gridDim.y + chunk] = bi;
    }
  }
}

// Pass 2: one CTA per row picks the best of the row's chunk winners.
constexpr int kFinalThreads = 256;
__global__ void __launch_bounds__(kFinalThreads) sample_final_kernel(const float* __restrict__ part_v,
                                                                     const int* __restrict__ part_i, int R, int nchunk,
                                                                     int* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  float bv = -INFINITY;
  int bi = INT_MAX;
  // Each thread's candidates are loaded kPer at a time (one memory round
  // trip per batch); the winner is unique under `better`, so the order in
  // which candidates are compared does not matter.
  constexpr int kPer = 16;
  for (int c0 = threadIdx.x; c0 < nchunk; c0 += kFinalThreads * kPer) {
    float v[kPer];
    int ix[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int c = c0 + u * kFinalThreads;
      v[u] = c < nchunk ? part_v[static_cast<size_t>(r) * nchunk + c] : -INFINITY;
      ix[u] = c < nchunk ? part_i[static_cast<size_t>(r) * nchunk + c] : INT_MAX;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u)
      if (better(v[u], ix[u], bv, bi)) {
        bv = v[u];
        bi = ix[u];
      }
  }
  warp_best(bv, bi);
  __shared__ float sv[kFinalThreads / 32];
  __shared__ int si[kFinalThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    bv = lane < kFinalThreads / 32 ? sv[lane] : -INFINITY;
    bi = lane < kFinalThreads / 32 ? si[lane] : INT_MAX;
    warp_best(bv, bi);
    if (lane == 0) out[r] = (bi == INT_MAX) ? 0 : bi;
  }
}

__global__ void philox_kernel(uint64_t seed, uint64_t step, int n, uint32_t* out) {
  pdl_wait();
  pdl_trigger();
  const int blk = blockIdx.x * blockDim.x + threadIdx.x;
  if (blk * 4 >= n) return;
  const uint4 w = philox_block(seed, step, static_cast<uint32_t>(blk));
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  for (int j = 0; j < 4 && blk * 4 + j < n; ++j) out[blk * 4 + j] = ws[j];
}

}  // namespace

int sample_chunks(int V) { return (V + kSampleChunk - 1) / kSampleChunk; }

int launch_sample(const float* logits, int R, int V, const vd_sampler* dev_params, float* part_v, int* part_i,
                  int* out, cudaStream_t s) {
  if (R <= 0) return VD_OK;
  if (V % 4) return fail(VD_ERR_UNSUPPORTED, "vocab must be a multiple of 4");
  const int nchunk = sample_chunks(V);
  VD_CUDA_TRY(launch_k(sample_partial_kernel, dim3(R, nchunk), dim3(kSampleThreads), 0, s, logits, V, dev_params,
                       part_v, part_i));
  VD_CUDA_TRY(launch_k(sample_final_kernel, dim3(R), dim3(kFinalThreads), 0, s, static_cast<const float*>(part_v),
                       static_cast<const int*>(part_i), R, nchunk, out));
  return VD_OK;
}

int launch_sample_final(const float* part_v, const int* part_i, int R, int nchunk, int* out, cudaStream_t s) {
  if (R <= 0) return VD_OK;
  VD_CUDA_TRY(launch_k(sample_final_kernel, dim3(R), dim3(kFinalThreads), 0, s, part_v, part_i, R, nchunk, out));
  return VD_OK;
}

int launch_philox(uint64_t seed, uint64_t step, int n, uint32_t* out, cudaStream_t s) {
  if (n <= 0) return VD_OK;
  const int blocks = (n + 4 * 256 - 1) / (4 * 256);
  VD_CUDA_TRY(launch_k(philox_kernel, dim3(blocks), dim3(256), 0, s, seed, step, n, out));
  return VD_OK;
}

}  // namespace vd
