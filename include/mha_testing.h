/*
 * mha_testing.h -- test, benchmark and diagnostic hooks of libmha.so.
 *
 * Not for production callers.  These entry points exist so that the tests
 * can run every kernel that can serve a problem (not only the one the
 * library would pick), force many work items per CTA, check the tensor-core
 * descriptors against a host matmul, and make the bounded device-side waits
 * expire on purpose.  None of them is part of the attention interface in
 * mha.h, and none is needed to use it.
 *
 * Scope.  The kernel-choice and launch-shape hooks (mha_set_*) are
 * thread-local: a value set on one host thread affects later calls made
 * from that thread only, so a test cannot change the kernels another thread
 * runs.  The device hooks (mha_test_*) act on the current device and affect
 * every later launch on it, from any thread.
 */
#ifndef MHA_GB300_TESTING_H
#define MHA_GB300_TESTING_H

#include "mha.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * mha_set_bf16_grid -- run the persistent bf16 forward kernels on `ctas`
 * CTAs (each loops over its share of the work items); 0 restores the default
 * of one CTA per SM.
 */
MHA_API void mha_set_bf16_grid(int ctas);

/*
 * mha_plan_prenorm -- the launch plan the Pre-LN forward (bf16) would use
 * for these sizes on a grid of `grid` CTAs, from the host logic alone (no
 * device needed).  out[0..5] = heads per chunk G, head groups per row block
 * H / G, CTAs per thread-block cluster (2: the two CTAs share each block's
 * row statistics), chunks whose statistics each CTA forms before its roles
 * start (0: at the chunk starts, or none when stats_given: the statistics
 * come from the no-allocation entry point's array), the grid after clamping
 * to the chunk count, and the chunk count.  Returns MHA_OK,
 * MHA_ERR_INVALID_ARG (non-positive sizes or grid, D not 64 or 128, null out)
 * or MHA_ERR_TOO_LARGE.
 */
MHA_API int mha_plan_prenorm(int B, int H, int Lq, int Lk, int D, int grid, int stats_given,
                             int64_t *out);

/*
 * mha_set_f32_kernel -- fp32 kernel choice.  0 = automatic: for D = 64 the
 * tensor-core kernel (three TF32 MMAs per product: hi*hi + lo*hi + hi*lo of
 * the operands split as x = hi + lo, fp32 accumulation in TMEM); for D = 128
 * the CUDA-core kernels: the short-key-range kernel (every visible K/V row of
 * a 16-row query block staged in shared memory at once) when Lk*D <= 16384,
 * else the tiled kernel (64-row query tiles, 64-key K/V tiles).  1 = always
 * the tiled CUDA-core kernel; 2 = the short-key-range kernel whenever
 * Lk*D <= 16384, else the tiled one; 3 = as 0.  Other values act as 0.
 */
MHA_API void mha_set_f32_kernel(int which);

/*
 * mha_set_bf16_decode -- 0 = automatic: bf16 mha_fwd calls with at most 8
 * query rows run the decode kernel (the keys of each (b, h) split over a
 * thread-block cluster of up to 8 CTAs, partial results combined in
 * distributed shared memory); 1 = never (always the tensor-core kernel).
 * Other values act as 0.
 */
MHA_API void mha_set_bf16_decode(int mode);

/*
 * mha_set_bf16_decode_splits -- split the visible keys of every (b, h) over
 * `splits` CTAs of the decode kernel (one cluster; values above 8 act as 8);
 * 0 restores the automatic choice (about one CTA per SM in total, at least
 * 256 keys per CTA; two per (b, h) when the problems number at least one per
 * SM and at most the CTAs resident at once).
 */
MHA_API void mha_set_bf16_decode_splits(int splits);

/*
 * mha_set_bwd_kernel -- mha_bwd kernel choice: 0 = automatic (bf16 on the
 * tensor cores, fp32 on CUDA cores); 1 = CUDA cores for both.  Other values
 * act as 0.  mha_bwd_workspace_size follows this choice.
 */
MHA_API void mha_set_bwd_kernel(int which);

/*
 * mha_set_pdl -- 1 (the default): every kernel is launched with programmatic
 * dependent launch allowed, so its grid can be scheduled while the previous
 * kernel of the stream finishes (each kernel still waits, on the device, for
 * that kernel's completion and writes before it touches global memory);
 * 0: ordinary launches.  Lets a test compare the two.
 */
MHA_API void mha_set_pdl(int on);

/*
 * mha_test_set_device_status -- OR `bits` into the device status word of
 * kernel unit `unit` on the current device (0 = bf16 forward, 1 = fp32
 * tensor-core forward, 2 = bf16 tensor-core backward, 3 = bf16 decode), as
 * an expired wait or a numeric flag would.  Lets a test check that
 * mha_device_status reports and clears every unit's word.  While a unit's
 * wait bits (0-15) are set its kernels return at once without writing their
 * outputs.  Returns MHA_OK, MHA_ERR_INVALID_ARG for an unknown unit, or
 * MHA_ERR_CUDA.
 */
MHA_API int mha_test_set_device_status(int unit, uint32_t bits);

/*
 * mha_test_set_wait_limit_ns -- the time limit of every bounded wait in the
 * tensor-core kernels on the current device, in nanoseconds; 0 restores the
 * default (2 s).  A tiny limit makes the first wait that is not satisfied at
 * once expire: the kernel then sets its status bit, drains the copies and
 * products already in flight (those drains keep the default limit) and
 * returns, so a test can check the expiry path without hanging anything.
 * Returns MHA_OK or MHA_ERR_CUDA.
 */
MHA_API int mha_test_set_wait_limit_ns(uint64_t ns);

/*
 * mha_selftest_umma -- diagnostic: one 128-row tcgen05 GEMM tile built
 * with exactly the shared-memory/TMEM descriptors the bf16 attention kernel
 * uses, so the descriptor encoding can be checked against a host matmul.
 *   variant 0: C[128,128] = A[128,K] * B[128,K]^T, both K-major in shared
 *              memory (the S = Q K^T step); K = 64 or 128.
 *   variant 1: C[128,N] = A[128,128] * B[128,N], A K-major and B N-major in
 *              shared memory (the P V step with P staged in shared memory).
 *   variant 2: as variant 1 but A is first written to tensor memory and the
 *              MMA reads it from there (the P V step the kernel uses).
 *   a, b bf16 row-major device buffers; c fp32 [128, N or 128] row-major.
 * Returns MHA_OK or a negative mha_status.
 */
MHA_API int mha_selftest_umma(int variant, int K_or_N, const void *a, const void *b,
                              float *c, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MHA_GB300_TESTING_H */
