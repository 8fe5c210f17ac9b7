// Measurement ops: the ceilings the decode GEMMs are held against.
//
// mma_issue_kernel times one thread issuing a chain of tcgen05 MMAs into one
// accumulator, 16 per stage, as the GEMM's issuer does, optionally testing an
// mbarrier phase (already completed) before each stage: the per-instruction
// costs the issuer is designed against.
//
// tma_stream_kernel streams a bf16 weight matrix [rows][K] from HBM through
// shared memory with exactly the copies a GEMM launch of a given plan
// issues -- 3-D TMA boxes (64, BM, kpo) into a 200 KB ring of stages, in the
// same tile order (persistent CTAs, tile b, b + grid, ...) -- and, when
// asked, the same activation boxes per K block (the re-reads of the token
// tile, served from L2).  One thread per CTA issues the copies, another
// releases each stage as soon as it has landed; nothing is computed.  The
// time of one launch over B bytes is therefore the rate a weight stream of
// that size and copy shape reaches in one launch, launch, ramp-up and drain
// included: the honest yardstick for a decode GEMM, whose MMAs and epilogue
// come on top.  With K cut into parts (k_parts > 1) the same bytes are
// spread over more CTAs than a GEMM's row tiles allow: the rate one launch
// reaches with every SM streaming.  Every wait is bounded (vd_device.cuh).
#include "vd_device.cuh"
#include "vd_internal.h"

namespace vd {
namespace {

constexpr int kStreamRing = 200 * 1024;
constexpr int kStreamMaxStages = 12;
constexpr int kStreamSmem = 1024 + kStreamRing + 2 * kStreamMaxStages * 8 + 16;

struct StreamArgs {
  int n_tiles;     // tiles: weight row blocks of box_rows rows x K parts
  int k_parts;     // K ranges per row block (1: a tile spans the whole K, as in a GEMM)
  int ops;         // stages per tile (K blocks / kpo / k_parts)
  int kpo;         // K blocks per weight copy
  int box_rows;    // weight rows per tile
  int x_box_rows;  // activation rows per K block (0: no activation copies)
  int w_bytes;     // weight bytes of one stage
  int x_sub;       // shared-memory bytes of one activation block (1 KB multiple)
  int stage_bytes;
  int stages;
  uint32_t tx;     // bytes one stage receives
  int* status;
};

__global__ void __launch_bounds__(64, 1)
    tma_stream_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                      StreamArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStreamRing);
  uint64_t* empty = full + kStreamMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStreamMaxStages);
  const int S = a.stages;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&wmap);
    if (a.x_box_rows) tma_prefetch_desc(&xmap);
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  int issued = 0;
  if (threadIdx.x == 0) {  // producer: the GEMM's weight (and activation) copies, in its order
    int g = 0, s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < a.n_tiles; tile += gridDim.x)
      for (int op = 0; op < a.ops; ++op, ++g) {
        if (g >= S && !mbar_wait(&empty[s], ph ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], a.tx);
        uint8_t* st = smem + s * a.stage_bytes;
        const int kb = ((tile % a.k_parts) * a.ops + op) * a.kpo;  // first K block of the copy
        tma_load_3d(st, &wmap, &full[s], 0, (tile / a.k_parts) * a.box_rows, kb);
        if (a.x_box_rows)
          for (int j = 0; j < a.kpo; ++j)
            tma_load_2d(st + a.w_bytes + j * a.x_sub, &xmap, &full[s], (kb + j) * kGemmBK, 0);
        issued = g + 1;
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
  } else if (threadIdx.x == 32) {  // consumer: releases every stage once it has landed
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < a.n_tiles; tile += gridDim.x)
      for (int op = 0; op < a.ops; ++op) {
        if (!mbar_wait(&full[s], ph, abort_flag, a.status)) {
          ok = false;
          break;
        }
        mbar_arrive(&empty[s]);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
  }
  // Teardown after a timeout: let the copies already issued land.
  if (threadIdx.x == 0 && *abort_flag)
    for (int g = issued > S ? issued - S : 0; g < issued; ++g) drain_wait(&full[g % S], (g / S) & 1);
  __syncthreads();
}

// One CTA: thread 32 issues n_mma MMAs (M x N x 16, 16 per stage: four K
// blocks of four K steps) on zeroed operands -- A: four 128-row K blocks
// (64 KB), B: one 256-row block (32 KB) -- into one TMEM accumulator; WAIT 1
// or 2 tests a completed phase before each stage with test_wait or
// try_wait, WAIT 3 with test_wait one stage ahead (before the previous
// stage's MMAs).  out[0]: cycles from the first issue to the last, out[1]: to
// the completion of every MMA.
constexpr int kIssueA = 4 * 128 * 128, kIssueB = 256 * 128;
constexpr int kIssueSmem = 1024 + kIssueA + kIssueB;

template <int WAIT>
__global__ void __launch_bounds__(128, 1) mma_issue_kernel(int M, int N, int n_mma, long long* out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ uint64_t bars[2];  // [0] every MMA done, [1] a phase completed at set-up
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  for (int i = threadIdx.x; i < (kIssueA + kIssueB) / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(smem)[i] = 0;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_arrive(&bars[1]);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(&tmem_slot, 256);
    tmem_relinquish();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the zeros, for the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tacc = tmem_slot;
  if (threadIdx.x == 32) {
    const uint32_t idesc = umma_idesc_bf16(M, N);
    const uint32_t a_lo = sw128_desc_lo(smem_u32(smem)), b_lo = sw128_desc_lo(smem_u32(smem) + kIssueA);
    const long long t0 = clock64();
    uint32_t acc = 0;
    bool ok = true, next = mbar_test_wait(&bars[1], 0);
    for (int st = 0; st < n_mma / 16; ++st) {
      // As in the GEMM, the stage's MMAs are issued only once the test has
      // returned true, so the test's latency is on the issuing path.
      bool ready = true;
      if constexpr (WAIT == 1) ready = mbar_test_wait(&bars[1], 0);
      if constexpr (WAIT == 2) ready = mbar_try_wait(&bars[1], 0);
      if constexpr (WAIT == 3) ready = next;  // tested one stage ahead
      if (!ready) {
        ok = false;
        break;
      }
      if constexpr (WAIT == 3) next = mbar_test_wait(&bars[1], 0);  // the next stage's test, before this one's MMAs
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_lo(tacc, a_lo + j * ((128 * 128) >> 4) + 2 * kk, b_lo + 2 * kk, idesc, acc | j | kk);
      acc = 1;
    }
    const long long t1 = clock64();
    umma_commit(&bars[0]);
    if (!mbar_wait(&bars[0], 0, &abort_flag, status)) ok = false;
    const long long t2 = clock64();
    out[0] = ok ? t1 - t0 : -1;
    out[1] = ok ? t2 - t0 : -1;
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tacc, 256);
  }
}

int stream_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

}  // namespace

int launch_mma_issue_probe(int M, int N, int n_mma, int wait, long long* out, int* status, cudaStream_t s) {
  static bool configured[4] = {false, false, false, false};
  auto k = wait == 0   ? mma_issue_kernel<0>
           : wait == 1 ? mma_issue_kernel<1>
           : wait == 2 ? mma_issue_kernel<2>
                       : mma_issue_kernel<3>;
  if (!configured[wait]) {
    VD_CUDA_TRY(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kIssueSmem));
    configured[wait] = true;
  }
  VD_CUDA_TRY(launch_k(k, dim3(1), dim3(128), kIssueSmem, s, M, N, n_mma, out, status));
  return VD_OK;
}

int launch_tma_stream(const CUtensorMap& wmap, const CUtensorMap& xmap, int rows, int K, int box_rows, int kpo,
                      int x_box_rows, int k_parts, int ctas, int* status, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    VD_CUDA_TRY(cudaFuncSetAttribute(tma_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmem));
    configured = true;
  }
  StreamArgs a{};
  a.k_parts = k_parts;
  a.n_tiles = rows / box_rows * k_parts;
  a.kpo = kpo;
  a.ops = K / kGemmBK / kpo / k_parts;
  a.box_rows = box_rows;
  a.x_box_rows = x_box_rows;
  a.w_bytes = kpo * box_rows * 128;
  a.x_sub = x_box_rows ? (x_box_rows * 128 + 1023) / 1024 * 1024 : 0;
  a.stage_bytes = a.w_bytes + kpo * a.x_sub;
  a.stages = std::min(kStreamMaxStages, kStreamRing / a.stage_bytes);
  a.tx = static_cast<uint32_t>(kpo * (box_rows + x_box_rows) * 128);
  a.status = status;
  if (a.stages < 2) return fail(VD_ERR_INVALID_ARG, "stream probe: a stage does not fit the ring twice");
  const int grid = std::min(a.n_tiles, ctas > 0 ? ctas : stream_sm_count());
  VD_CUDA_TRY(launch_k(tma_stream_kernel, dim3(grid), dim3(64), kStreamSmem, s, wmap, xmap, a));
  return VD_OK;
}

}  // namespace vd
