// Bandwidth-bound row kernels of the step: embedding gather, RMSNorm,
// RoPE + K/V scatter into the paged pool, and the debug K/V gather.
//
// Batch invariance ("Deterministic and bit-exact inference", technical
// section: batch-invariant RMSNorm): every reduction here runs inside one
// warp over one row, lane l summing elements l, l+32, ... (in 8-element
// chunks) in ascending order, followed by a fixed xor butterfly, so the
// result of a row depends on that row and the model dimension only.
#include "vd_device.cuh"
#include "vd_internal.h"

namespace vd {
namespace {

// Token t's id is tok[t], or feed[-1 - tok[t]] for an entry below zero (a
// token produced on the device by an earlier step).  A fed id outside the
// vocabulary is recorded in the status word and row 0 is read instead.
__global__ void embed_kernel(const uint4* __restrict__ E, const int* __restrict__ tok, const int* __restrict__ feed,
                             int V, int* status, float scale, uint4* __restrict__ x, int d8) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  int id = tok[t];
  if (id < 0) {
    id = feed ? feed[-1 - id] : -1;
    if (id < 0 || id >= V) {
      if (threadIdx.x == 0 && status) atomicCAS(status, 0, static_cast<int>(VD_ERR_OUT_OF_RANGE));
      id = 0;
    }
  }
  const size_t src = static_cast<size_t>(id) * d8;
  if (scale == 0.f) {
#pragma unroll 4
    for (int c = threadIdx.x; c < d8; c += blockDim.x) x[static_cast<size_t>(t) * d8 + c] = E[src + c];
  } else {
#pragma unroll 4
    for (int c = threadIdx.x; c < d8; c += blockDim.x) {
      const uint4 v = E[src + c];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = pack_bf16x2(__fmul_rn(bf16_lo(w[i]), scale), __fmul_rn(bf16_hi(w[i]), scale));
      x[static_cast<size_t>(t) * d8 + c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_lo(w[i]);
    f[2 * i + 1] = bf16_hi(w[i]);
  }
}

__device__ __forceinline__ float warp_sum_fixed(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// y[r] = bf16(x[row_idx[r]] * (1 / sqrt(mean(x^2) + eps)) * w)
//
// CH > 0: the row's CH chunks per lane are loaded into registers before the
// sum (all loads in flight at once) and reused for the output; CH == 0 is
// the streaming form for rows longer than 32 * 16 chunks.  Both sum the same
// terms in the same order.
template <int CH>
__global__ void rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, const int* __restrict__ row_idx,
                               const __nv_bfloat16* __restrict__ w, __nv_bfloat16* __restrict__ y, int rows, int d,
                               float eps, float off) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= rows) return;
  const int src = row_idx ? row_idx[r] : r;
  const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(src) * d);
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  uint4* yr = reinterpret_cast<uint4*>(y + static_cast<size_t>(r) * d);
  const int d8 = d >> 3;
  auto out8 = [&](const uint4& xv, const uint4& wv, int c, float inv) {
    float f[8], g[8];
    unpack8(xv, f);
    unpack8(wv, g);
    if (off != 0.f) {
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = __fadd_rn(g[i], off);
    }
    uint4 o;
    o.x = pack_bf16x2(__fmul_rn(__fmul_rn(f[0], inv), g[0]), __fmul_rn(__fmul_rn(f[1], inv), g[1]));
    o.y = pack_bf16x2(__fmul_rn(__fmul_rn(f[2], inv), g[2]), __fmul_rn(__fmul_rn(f[3], inv), g[3]));
    o.z = pack_bf16x2(__fmul_rn(__fmul_rn(f[4], inv), g[4]), __fmul_rn(__fmul_rn(f[5], inv), g[5]));
    o.w = pack_bf16x2(__fmul_rn(__fmul_rn(f[6], inv), g[6]), __fmul_rn(__fmul_rn(f[7], inv), g[7]));
    yr[c] = o;
  };
  auto add8 = [](float ss, const uint4& xv) {
    float f[8];
    unpack8(xv, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = __fadd_rn(ss, __fmul_rn(f[i], f[i]));
    return ss;
  };
  float ss = 0.f;
  if constexpr (CH > 0) {
    // the row and its gains in flight together: one memory round trip, not
    // one per gain chunk after the sum
    uint4 xv[CH], wv[CH];
#pragma unroll
    for (int k = 0; k < CH; ++k)
      if (lane + 32 * k < d8) {
        xv[k] = xr[lane + 32 * k];
        wv[k] = wr[lane + 32 * k];
      }
#pragma unroll
    for (int k = 0; k < CH; ++k)
      if (lane + 32 * k < d8) ss = add8(ss, xv[k]);
    ss = warp_sum_fixed(ss);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(d)), eps)));
#pragma unroll
    for (int k = 0; k < CH; ++k)
      if (lane + 32 * k < d8) out8(xv[k], wv[k], lane + 32 * k, inv);
  } else {
#pragma unroll 4
    for (int c = lane; c < d8; c += 32) ss = add8(ss, xr[c]);
    ss = warp_sum_fixed(ss);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(d)), eps)));
    for (int c = lane; c < d8; c += 32) out8(xr[c], wr[c], c, inv);
  }
}

// Sandwich norm of a sub-layer output h, residual add, and (optionally) the
// next pre-norm, one warp per row:
//   x = bf16(x + bf16(h * (1 / sqrt(mean(h^2) + eps)) * g_post))
//   y = bf16(x * (1 / sqrt(mean(x^2) + eps)) * g_pre)        (if w_pre)
// Both sums run in the lane-strided order of rmsnorm_kernel, so y equals what
// rmsnorm_kernel gives for the new x.  CH as in rmsnorm_kernel.
template <int CH>
__global__ void postnorm_residual_kernel(const __nv_bfloat16* __restrict__ h, __nv_bfloat16* __restrict__ x,
                                         const __nv_bfloat16* __restrict__ w_post,
                                         const __nv_bfloat16* __restrict__ w_pre, __nv_bfloat16* __restrict__ y,
                                         int rows, int d, float eps, float off) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= rows) return;
  const uint4* hr = reinterpret_cast<const uint4*>(h + static_cast<size_t>(r) * d);
  uint4* xr = reinterpret_cast<uint4*>(x + static_cast<size_t>(r) * d);
  uint4* yr = reinterpret_cast<uint4*>(y + static_cast<size_t>(r) * d);
  const uint4* wp = reinterpret_cast<const uint4*>(w_post);
  const uint4* wq = reinterpret_cast<const uint4*>(w_pre);
  const int d8 = d >> 3;
  auto add8 = [](float ss, const uint4& v) {
    float f[8];
    unpack8(v, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = __fadd_rn(ss, __fmul_rn(f[i], f[i]));
    return ss;
  };
  auto gains8 = [&](const uint4& wv, float* g) {
    unpack8(wv, g);
    if (off != 0.f) {
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = __fadd_rn(g[i], off);
    }
  };
  auto inv_of = [&](float ss) {
    ss = warp_sum_fixed(ss);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(d)), eps)));
  };
  // x + bf16(h * inv * g) for one chunk, rounded to bf16
  auto resid8 = [&](const uint4& hv, const uint4& xv, const uint4& gv, float inv) {
    float fh[8], fx[8], g[8], o[8];
    unpack8(hv, fh);
    unpack8(xv, fx);
    gains8(gv, g);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = __fadd_rn(fx[i], bf16_round(__fmul_rn(__fmul_rn(fh[i], inv), g[i])));
    return make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
  };
  auto norm8 = [&](const uint4& xv, const uint4& gv, float inv) {
    float f[8], g[8];
    unpack8(xv, f);
    gains8(gv, g);
    return make_uint4(pack_bf16x2(__fmul_rn(__fmul_rn(f[0], inv), g[0]), __fmul_rn(__fmul_rn(f[1], inv), g[1])),
                      pack_bf16x2(__fmul_rn(__fmul_rn(f[2], inv), g[2]), __fmul_rn(__fmul_rn(f[3], inv), g[3])),
                      pack_bf16x2(__fmul_rn(__fmul_rn(f[4], inv), g[4]), __fmul_rn(__fmul_rn(f[5], inv), g[5])),
                      pack_bf16x2(__fmul_rn(__fmul_rn(f[6], inv), g[6]), __fmul_rn(__fmul_rn(f[7], inv), g[7])));
  };
  if constexpr (CH > 0) {
    uint4 hv[CH], xv[CH], pv[CH], qv[CH];  // the row, the residual and both gains in flight together
#pragma unroll
    for (int k = 0; k < CH; ++k)
      if (lane + 32 * k < d8) {
        hv[k] = hr[lane + 32 * k];
        xv[k] = xr[lane + 32 * k];
        pv[k] = wp[lane + 32 * k];
        if (w_pre) qv[k] = wq[lane + 32 * k];
      }
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < CH; ++k)
      if (lane + 32 * k < d8) ss = add8(ss, hv[k]);
    const float inv = inv_of(ss);
#pragma unroll
    for (int k = 0; k < CH; ++k)
      if (lane + 32 * k < d8) {
        xv[k] = resid8(hv[k], xv[k], pv[k], inv);
        xr[lane + 32 * k] = xv[k];
      }
    if (!w_pre) return;
    float s2 = 0.f;
#pragma unroll
    for (int k = 0; k < CH; ++k)
      if (lane + 32 * k < d8) s2 = add8(s2, xv[k]);
    const float inv2 = inv_of(s2);
#pragma unroll
    for (int k = 0; k < CH; ++k)
      if (lane + 32 * k < d8) yr[lane + 32 * k] = norm8(xv[k], qv[k], inv2);
  } else {
    float ss = 0.f;
    for (int c = lane; c < d8; c += 32) ss = add8(ss, hr[c]);
    const float inv = inv_of(ss);
    float s2 = 0.f;
    for (int c = lane; c < d8; c += 32) {
      const uint4 xn = resid8(hr[c], xr[c], wp[c], inv);
      xr[c] = xn;
      s2 = add8(s2, xn);
    }
    if (!w_pre) return;
    const float inv2 = inv_of(s2);
    for (int c = lane; c < d8; c += 32) yr[c] = norm8(xr[c], wq[c], inv2);
  }
}

// One warp per (token, head).  Lane l owns the rotate-half pairs
// (i, i + hd/2) for i = l, l+32, ...  q heads -> q_out, k heads -> pool K
// slot, v heads -> pool V slot of the token's (page, position % 16).
constexpr int kRopeWarps = 8;
__global__ void __launch_bounds__(kRopeWarps * 32) rope_kv_kernel(RopeArgs a) {
  const int t = blockIdx.x;
  const int head = blockIdx.y * kRopeWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int nh = a.Hq + 2 * a.Hkv;
  const int hd = a.hd, half = hd >> 1;
  // The token's position and page slot (the step's description, written
  // before the step's first kernel) and its rotation factors (constant
  // tables) are read before the wait for the QKV GEMM, whose output is read
  // after it.
  const bool live = head < nh;
  const int p = live ? a.positions[t] : 0;
  const size_t page = live ? static_cast<size_t>(a.slot_page[t]) : 0;
  const int slot = p & 15;
  const int np = (half + 31) / 32;
  float cs[4] = {0.f, 0.f, 0.f, 0.f}, sn[4] = {0.f, 0.f, 0.f, 0.f};
  if (live && head < a.Hq + a.Hkv) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = lane + 32 * k;
      if (k < np && i < half) {
        cs[k] = a.cos_t[static_cast<size_t>(p) * half + i];
        sn[k] = a.sin_t[static_cast<size_t>(p) * half + i];
      }
    }
  }
  pdl_wait();
  pdl_trigger();
  if (!live) return;
  const __nv_bfloat16* src = a.qkv + (static_cast<size_t>(t) * nh + head) * hd;
  if (head >= a.Hq + a.Hkv) {  // v: plain copy
    const int g = head - a.Hq - a.Hkv;
    __nv_bfloat16* dst = a.pool + a.layer_elem0 + ((page * 2 + 1) * a.Hkv + g) * 16 * hd + slot * hd;
    for (int i = lane; i < hd; i += 32) dst[i] = src[i];
    return;
  }
  const bool is_q = head < a.Hq;
  float x1[4], x2[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    x1[k] = (k < np && i < half) ? __bfloat162float(src[i]) : 0.f;
    x2[k] = (k < np && i < half) ? __bfloat162float(src[i + half]) : 0.f;
  }
  const __nv_bfloat16* nw = is_q ? a.q_norm : a.k_norm;
  if (nw) {  // per-head RMSNorm (QK-norm), rounded to bf16 before RoPE
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      ss = __fadd_rn(ss, __fmul_rn(x1[k], x1[k]));
      ss = __fadd_rn(ss, __fmul_rn(x2[k], x2[k]));
    }
    ss = warp_sum_fixed(ss);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(hd)), a.eps)));
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = lane + 32 * k;
      if (k < np && i < half) {
        float g1 = __bfloat162float(nw[i]), g2 = __bfloat162float(nw[i + half]);
        if (a.gain_offset != 0.f) {
          g1 = __fadd_rn(g1, a.gain_offset);
          g2 = __fadd_rn(g2, a.gain_offset);
        }
        x1[k] = bf16_round(__fmul_rn(__fmul_rn(x1[k], inv), g1));
        x2[k] = bf16_round(__fmul_rn(__fmul_rn(x2[k], inv), g2));
      }
    }
  }
  __nv_bfloat16* dst;
  if (is_q) {
    dst = a.q_out + (static_cast<size_t>(t) * a.Hq + head) * hd;
  } else {
    const int g = head - a.Hq;
    dst = a.pool + a.layer_elem0 + ((page * 2 + 0) * a.Hkv + g) * 16 * hd + slot * hd;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    if (k < np && i < half) {
      const float c = cs[k], s = sn[k];
      dst[i] = __float2bfloat16_rn(__fsub_rn(__fmul_rn(x1[k], c), __fmul_rn(x2[k], s)));
      dst[i + half] = __float2bfloat16_rn(__fadd_rn(__fmul_rn(x2[k], c), __fmul_rn(x1[k], s)));
    }
  }
}

}  // namespace

int launch_embed(const void* embed, const int* tokens, const int* feed, int V, int* status, float scale, void* x,
                 int T, int d, cudaStream_t s) {
  if (T <= 0) return VD_OK;
  VD_CUDA_TRY(launch_k(embed_kernel, dim3(T), dim3(128), 0, s, static_cast<const uint4*>(embed), tokens, feed, V,
                       status, scale, static_cast<uint4*>(x), d / 8));
  return VD_OK;
}

int launch_rmsnorm(const void* x, const int* row_idx, const void* w, void* y, int rows, int d, float eps,
                   float gain_offset, cudaStream_t s) {
  if (rows <= 0) return VD_OK;
  const auto* xp = static_cast<const __nv_bfloat16*>(x);
  const auto* wp = static_cast<const __nv_bfloat16*>(w);
  auto* yp = static_cast<__nv_bfloat16*>(y);
  const int per_lane = (d / 8 + 31) / 32, blocks = (rows + 3) / 4;
  auto k = per_lane <= 1    ? rmsnorm_kernel<1>
           : per_lane <= 2  ? rmsnorm_kernel<2>
           : per_lane <= 4  ? rmsnorm_kernel<4>
           : per_lane <= 8  ? rmsnorm_kernel<8>
           : per_lane <= 12 ? rmsnorm_kernel<12>
           : per_lane <= 16 ? rmsnorm_kernel<16>
                            : rmsnorm_kernel<0>;
  VD_CUDA_TRY(launch_k(k, dim3(blocks), dim3(128), 0, s, xp, row_idx, wp, yp, rows, d, eps, gain_offset));
  return VD_OK;
}

int launch_postnorm_residual(const void* h, void* x, const void* w_post, const void* w_pre, void* y, int rows, int d,
                             float eps, float gain_offset, cudaStream_t s) {
  if (rows <= 0) return VD_OK;
  const auto* hp = static_cast<const __nv_bfloat16*>(h);
  auto* xp = static_cast<__nv_bfloat16*>(x);
  const auto* wp = static_cast<const __nv_bfloat16*>(w_post);
  const auto* wq = static_cast<const __nv_bfloat16*>(w_pre);
  auto* yp = static_cast<__nv_bfloat16*>(y);
  const int per_lane = (d / 8 + 31) / 32, blocks = (rows + 3) / 4;
  // register-resident forms hold four arrays of CH chunks per lane; past 12
  // chunks (d > 3072) they would spill, so longer rows stream
  auto k = per_lane <= 1    ? postnorm_residual_kernel<1>
           : per_lane <= 2  ? postnorm_residual_kernel<2>
           : per_lane <= 4  ? postnorm_residual_kernel<4>
           : per_lane <= 8  ? postnorm_residual_kernel<8>
           : per_lane <= 12 ? postnorm_residual_kernel<12>
                            : postnorm_residual_kernel<0>;
  VD_CUDA_TRY(launch_k(k, dim3(blocks), dim3(128), 0, s, hp, xp, wp, wq, yp, rows, d, eps, gain_offset));
  return VD_OK;
}

int launch_rope_kv(const RopeArgs& a, cudaStream_t s) {
  if (a.T <= 0) return VD_OK;
  const int nh = a.Hq + 2 * a.Hkv;
  dim3 grid(a.T, (nh + kRopeWarps - 1) / kRopeWarps);
  VD_CUDA_TRY(launch_k(rope_kv_kernel, grid, dim3(kRopeWarps * 32), 0, s, a));
  return VD_OK;
}


// ---------------------------------------------------------------- failure path
// Drives the bounded waits every pipelined kernel uses to their limit, with
// nothing in flight: thread 0 of warp 0 and thread 0 of warp 1 wait on an
// mbarrier that no thread ever arrives at.  The first to reach the limit
// records VD_ERR_TIMEOUT in the status word and raises the CTA's abort flag,
// which ends the other wait; then the teardown wait, which ignores the
// flag, gives up after the limit too, and the kernel returns.  out[0] = 1 if
// warp 0's wait gave up, out[1] = 1 if warp 1's did, out[2] = 1 if the
// teardown wait gave up.
namespace {
__global__ void wait_probe_kernel(int* status, uint64_t limit_ns, int* out) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    const bool ok = mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
    if (out) out[warp] = ok ? 0 : 1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool drained = drain_wait(&bar, 0, limit_ns);
    if (out) out[2] = drained ? 0 : 1;
  }
}
}  // namespace

int launch_wait_probe(int* status, uint64_t limit_ns, int* out, cudaStream_t s) {
  VD_CUDA_TRY(launch_k(wait_probe_kernel, dim3(1), dim3(64), 0, s, status, limit_ns, out));
  return VD_OK;
}

}  // namespace vd
