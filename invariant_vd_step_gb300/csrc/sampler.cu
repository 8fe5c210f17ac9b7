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
// no summation order can change, so the result is fixed by the row alone.
#include <limits.h>
#include <math.h>

#include "vd_device.cuh"
#include "vd_internal.h"

namespace vd {
namespace {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

__device__ __forceinline__ uint4 philox_block(uint64_t seed, uint64_t step, uint32_t blk) {
  return philox4x32_10(make_uint4(blk, static_cast<uint32_t>(step), static_cast<uint32_t>(step >> 32), 0x5644u),
                       static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

constexpr int kSampleThreads = 512;

__global__ void __launch_bounds__(kSampleThreads) sample_kernel(const float* __restrict__ logits, int V,
                                                               const vd_sampler* __restrict__ params,
                                                               int* __restrict__ out) {
  const int r = blockIdx.x;
  const float* l = logits + static_cast<size_t>(r) * V;
  const vd_sampler sp = params[r];
  const bool greedy = !(sp.temperature > 0.f);
  float bv = -INFINITY;
  int bi = INT_MAX;
  for (int blk = threadIdx.x; blk * 4 < V; blk += kSampleThreads) {
    uint4 w = make_uint4(0, 0, 0, 0);
    if (!greedy) w = philox_block(sp.seed, sp.step, static_cast<uint32_t>(blk));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = blk * 4 + j;
      if (i >= V) break;
      float v = l[i];
      if (!greedy) {
        const float u = __fmul_rn(__fadd_rn(static_cast<float>(ws[j] >> 8), 0.5f), 5.9604644775390625e-8f);
        const float g = -logf(-logf(u));
        v = __fadd_rn(__fdiv_rn(v, sp.temperature), g);
      }
      if (better(v, i, bv, bi)) {
        bv = v;
        bi = i;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  __shared__ float sv[kSampleThreads / 32];
  __shared__ int si[kSampleThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < kSampleThreads / 32; ++k)
      if (better(sv[k], si[k], bv, bi)) {
        bv = sv[k];
        bi = si[k];
      }
    out[r] = (bi == INT_MAX) ? 0 : bi;
  }
}

__global__ void philox_kernel(uint64_t seed, uint64_t step, int n, uint32_t* out) {
  const int blk = blockIdx.x * blockDim.x + threadIdx.x;
  if (blk * 4 >= n) return;
  const uint4 w = philox_block(seed, step, static_cast<uint32_t>(blk));
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  for (int j = 0; j < 4 && blk * 4 + j < n; ++j) out[blk * 4 + j] = ws[j];
}

}  // namespace

int launch_sample(const float* logits, int R, int V, const vd_sampler* dev_params, int* out, cudaStream_t s) {
  if (R <= 0) return VD_OK;
  sample_kernel<<<R, kSampleThreads, 0, s>>>(logits, V, dev_params, out);
  VD_CUDA_TRY(cudaGetLastError());
  return VD_OK;
}

int launch_philox(uint64_t seed, uint64_t step, int n, uint32_t* out, cudaStream_t s) {
  if (n <= 0) return VD_OK;
  const int blocks = (n + 4 * 256 - 1) / (4 * 256);
  philox_kernel<<<blocks, 256, 0, s>>>(seed, step, n, out);
  VD_CUDA_TRY(cudaGetLastError());
  return VD_OK;
}

}  // namespace vd
