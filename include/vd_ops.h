/*
 * vd_ops.h -- single-kernel entry points of libvd.so.
 *
 * Each call runs exactly one of the kernels vd_step uses, with the same
 * fixed configuration, on caller-provided device buffers.  They exist so
 * that each kernel can be checked on its own: against the CPU oracle on
 * seeded inputs, and against itself across batch shapes (the relational
 * contracts of 深入解析 Vosti §六 6.1 / 6.2).  Conventions (return codes,
 * validation before launch, dev/host pointers, streams) are those of vd.h.
 */
#ifndef VD_OPS_H_
#define VD_OPS_H_

#include <stdint.h>

#include "vd.h"

#ifdef __cplusplus
extern "C" {
#endif

enum {
  VD_EPI_BF16 = 0,      /* C = bf16(acc)                                       */
  VD_EPI_RESIDUAL = 1,  /* C = bf16(bf16(acc) + R); R may alias C              */
  VD_EPI_F32 = 2,       /* C = acc (float32)                                   */
  VD_EPI_SWIGLU = 3,    /* C[t][f] = bf16(silu(bf16(g)) * bf16(u))             */
  VD_EPI_GEGLU = 4      /* C[t][f] = bf16(gelu_tanh(bf16(g)) * bf16(u))        */
};

/* Batch-invariant bf16 GEMM [B §六 6.1 matmul contract: row x of a batched
 * run equals the singleton run bit for bit].  acc[t][n] = sum_k A[t][k] W[n][k]
 * in fp32 on tcgen05 tensor cores.  Every element of acc is one chain of
 * K = 16 MMA steps in ascending K order into a zeroed accumulator, with no
 * split-K, whatever T; the tile (BM weight rows x BN tokens, chosen per
 * launch, see vd_set_gemm_plan) sets only the instruction's M and N, which
 * leave each element's arithmetic unchanged.
 * A: dev bf16 [T][K]; W: dev bf16 [N][K] (GLU: [2F][K], rows F.. are "up",
 * N = F); C: dev [T][N] bf16 (float32 for VD_EPI_F32); residual: dev bf16
 * [T][N] or null.  Requires N % 128 == 0 (GLU: F % 64 == 0), K % 64 == 0,
 * 16-byte aligned pointers, T >= 1.  Errors: VD_ERR_INVALID_ARG,
 * VD_ERR_UNSUPPORTED, VD_ERR_CUDA. */
int vd_op_gemm(const void* A, const void* W, void* C, int32_t T, int32_t N, int32_t K, int32_t epilogue,
               const void* residual, void* stream);

/* GEMM launch shape override, process-wide, for every later GEMM launch
 * (vd_op_gemm and the GEMMs of vd_step / vd_step_sample): bm = weight rows
 * per tile (64, 128, or 256 = two M = 128 MMAs sharing each activation
 * block), bn = tokens per tile (16, 32, 64, 128 or 256), kpo = 64-wide K
 * blocks per weight copy (1, 2 or 4); 0 leaves a field to the per-launch
 * choice.  A field a launch cannot take is left to that choice too (bm 64
 * for the fused token choice of the LM head; bm 256 when the matrix's rows
 * are not a multiple of 256 or K is split; a kpo that does not divide
 * K / 64; kpo is 1 with bm 256 and is halved while two pipeline stages do
 * not fit).  The
 * plan changes speed only, never a bit of the result: it exists to test that
 * and to measure each shape.  Step graphs captured under another override are
 * not replayed.  (An engineering addition; the pages have no counterpart.)
 * Errors: VD_ERR_INVALID_ARG for values outside those sets. */
int vd_set_gemm_plan(int32_t bm, int32_t bn, int32_t kpo);

/* The plan a GEMM launch over T tokens against an N x K weight matrix (GLU:
 * 2N rows, N = F) with this epilogue takes, including a forced plan:
 * out[0] = bm, out[1] = bn, out[2] = kpo (host array).  epilogue: a VD_EPI_*
 * value, or 5 for the LM head with the fused token choice.  Needs no GPU
 * work (it reads the device's SM count).  Errors: VD_ERR_INVALID_ARG. */
int vd_gemm_plan_query(int32_t T, int32_t N, int32_t K, int32_t epilogue, int32_t out[3]);

/* The GEMM's tile shape (weight rows and tokens per tile) is chosen per
 * launch because the tensor cores compute each output element the same way
 * whatever the MMA instruction's M and N -- a property of the hardware that
 * was measured, not documented [B §六 6.1 asks for one reduction order per
 * element, which the K order alone fixes].  vd_create_model therefore runs,
 * once per device, every tile shape on seeded operands and compares the raw
 * fp32 results bit for bit.  Returns 1 if they all agreed (shapes stay
 * chosen per launch), 0 if any bit differed (every later launch takes one
 * fixed shape, 128 rows x 256 tokens x 1 K block per copy), -1 if the check
 * could not run.  Runs the check on the current device if no model did yet
 * (launches kernels and synchronises the device). */
int vd_gemm_shape_check(void);

/* Batch-invariant RMSNorm [T technical: batch-invariant RMSNorm]:
 * y[r] = bf16(x[r] / sqrt(mean(x[r]^2) + eps) * w), one warp per row, fixed
 * lane-strided sum of squares and fixed butterfly.  x, y: dev bf16 [rows][d],
 * w: dev bf16 [d]; d % 8 == 0. */
int vd_op_rmsnorm(const void* x, const void* w, void* y, int32_t rows, int32_t d, float eps, void* stream);

/* Unified paged attention + fixed-order split merge for `layer` of model m
 * over pool p [B §六 6.2: causal contract, masking rules, tile traversal;
 * T technical: fixed KV split size].  q: dev bf16 [T][Hq][hd] (rotated),
 * out: dev bf16 [T][Hq][hd].  Reads K/V of positions [0, cached_len+q_len)
 * through the batch's page tables (host descriptor as for vd_step; token ids
 * and logit rows are ignored).  The K/V of the new tokens must already be in
 * the pool. */
int vd_op_attention(vd_model* m, vd_kv_pool* p, int32_t layer, const vd_batch* b, const void* q, void* out,
                    void* stream);

/* vd_op_attention without any allocation: the same kernels, the same
 * arguments and the same bits, but the split partials go to a fixed device
 * array inside libvd.so instead of the model's workspace.  (No counterpart
 * in the paper: this is a deployment convenience of this library.)
 *
 * For callers that cannot allocate device memory at call time: a host that
 * has handed the whole device memory to its own allocator or memory pool
 * (a cudaMalloc from a library would fail or fragment that pool), and
 * latency-bound loops that cannot afford cudaMalloc/cudaFree, which may
 * synchronise the whole device.
 *
 * Limits and sharing:
 *  - scratch = num_tokens * n_heads * S * (head_dim + 2) * 4 bytes, where S
 *    is the largest number of 512-key splits of any request of the call
 *    (ceil((cached_len + q_len) / 512)); calls needing more than
 *    VD_ATTN_STATIC_SCRATCH_BYTES (16 MiB) are rejected with VD_ERR_CAPACITY
 *    before anything is launched;
 *  - the array exists once per device (every device that loads libvd.so
 *    holds it until the process exits) and is shared by all calls: calls
 *    that may run at the same time on the GPU (different streams, threads
 *    or models) race on it and must be ordered by the caller;
 *  - nothing in it needs to start at zero (each call writes every partial
 *    it reads), so it is never cleared;
 *  - every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress, a host-side lookup that allocates nothing), so
 *    a context re-created on the same device (after cudaDeviceReset) gets
 *    the new address; make the first call on a device before any stream
 *    capture, as that one also loads the library's module on the device;
 *  - arguments are validated exactly as vd_op_attention validates them
 *    (the same error codes for the same batch) before the scratch size is
 *    checked.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
#define VD_ATTN_STATIC_SCRATCH_BYTES (16u << 20)
int vd_op_attention_static(vd_model* m, vd_kv_pool* p, int32_t layer, const vd_batch* b, const void* q,
                           void* out, void* stream);

/* RoPE + K/V write for `layer` (and per-head QK RMSNorm if the model has
 * it): qkv dev bf16 [T][(Hq+2Hkv) hd] -> q_out dev bf16 [T][Hq][hd]; k and v
 * of token t go to the pool slot of (request, position) via the batch's
 * page tables [B §五 5.1: KV keyed to its logical prefix]. */
int vd_op_rope_kv(vd_model* m, vd_kv_pool* p, int32_t layer, const vd_batch* b, const void* qkv, void* q_out,
                  void* stream);

/* The sampler's Philox4x32-10 stream: out[i] = word used for vocabulary index
 * i at (seed, step); dev uint32 [n]. */
int vd_op_philox(uint64_t seed, uint64_t step, int32_t n, uint32_t* out, void* stream);

/* Measurement op (no counterpart in the paper; the yardstick of the decode
 * GEMMs): streams the dev bf16 matrix w [rows][K] from HBM through shared
 * memory with exactly the weight copies a GEMM launch with plan (box_rows,
 * kpo) issues -- 3-D TMA boxes of box_rows rows x kpo K blocks of 64, into
 * the GEMM's 200 KB ring, in its tile order -- and, if x_box_rows > 0, its
 * activation copies of x_box_rows rows of the dev bf16 x [x_rows][K] per K
 * block.  Nothing is computed or written; one launch's time is the rate a
 * weight stream of that size and copy shape reaches in one launch.
 * k_parts > 1 cuts each row block's K into that many tiles (the same bytes
 * over more CTAs than a GEMM's row tiles allow).
 * box_rows in {64, 128, 256} dividing rows; kpo in {1, 2, 4} dividing K/64
 * (1 for 256-row boxes); ctas = 0: one CTA per SM.  Every on-device wait
 * is bounded.  Errors: VD_ERR_INVALID_ARG. */
int vd_op_tma_stream(const void* w, int64_t rows, int64_t K, const void* x, int64_t x_rows, int32_t box_rows,
                     int32_t kpo, int32_t x_box_rows, int32_t k_parts, int32_t ctas, void* stream);

/* Measurement op (no counterpart in the paper; the figures the GEMM's MMA
 * issuer is designed against): one CTA, one thread issuing n_mma bf16
 * tcgen05 MMAs of M x N x 16 (fp32 accumulation) into one TMEM accumulator,
 * 16 per stage, on zeroed shared-memory operands; before each stage it tests
 * an mbarrier phase that has already completed with wait = 0 (no test),
 * 1 (mbarrier.test_wait) or 2 (mbarrier.try_wait), each stage's MMAs issued
 * only once the test returned true, or 3 (test_wait one stage ahead: the
 * next stage's test is issued before this stage's MMAs).  out: dev int64 [2],
 * SM clock cycles from the first issue to the last issue and to the
 * completion of every MMA (-1 if the final bounded wait gave up).  M in
 * {64, 128}; N a multiple of 16 in [16, 256]; n_mma a multiple of 16 in
 * [16, 65536]; wait in {0, 1, 2, 3}.  Errors: VD_ERR_INVALID_ARG. */
int vd_op_mma_issue_probe(int32_t M, int32_t N, int32_t n_mma, int32_t wait, int64_t* out, void* stream);

/* Test of the failure path of every on-device wait (the bounded waits of
 * the pipelined GEMM and attention kernels; no counterpart in the paper, it
 * exercises this library's own failure detection).  Launches one CTA whose
 * two waiting threads wait, with the limit limit_us, on an mbarrier that
 * nothing completes; nothing else is in flight and no memory but the
 * model's status word and `out` is touched.  The wait gives up, records
 * VD_ERR_TIMEOUT in the model's device status word (read and cleared by
 * vd_device_status) and the kernel returns, so the context stays usable.
 * While the status word holds the timeout, the step kernels of this model
 * skip their work (a failed step's outputs are not written); reading the
 * status clears it.  out (nullable): dev int32 [3], set to 1 for each wait
 * that gave up (warp 0's, warp 1's, the teardown wait).  limit_us in
 * [1, 2000000]; errors: VD_ERR_INVALID_ARG. */
int vd_op_wait_probe(vd_model* m, int32_t limit_us, int32_t* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* VD_OPS_H_ */
