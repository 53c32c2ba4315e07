/*
 * mha.h -- C ABI of the GB300 (sm_103a) fused masked multi-head attention
 * forward library (libmha.so).
 *
 * What is computed.  For every batch b, head h and query row i:
 *     s_j = scale * sum_d Q[b,h,i,d] * K[b,h,j,d]
 *     visible(i, j) = (j < len_b if MHA_MASK_KV_LEN) and (j <= i if MHA_MASK_CAUSAL)
 *     O[b,h,i,:] = sum_j softmax_j(s over visible j) * V[b,h,j,:]
 * with the softmax taken after subtracting the running row maximum (online
 * softmax), masked keys contributing exactly zero, and a row with no visible
 * key returning zeros.  mha_fwd_lse also returns each row's log-sum-exp, and
 * mha_bwd the gradients dq, dk, dv of sum(dout * O) from it.  Sources, cited by page title and section:
 *  - "How to fuse cross-attention and layer-norm into a single CUDA kernel?"
 *    (cms365.cn), knowledge points: S = QK^T -> P = softmax(S) -> O = PV;
 *    answer steps two to five: Pre-LayerNorm on the query rows and the
 *    extension signature (q, k, v, gamma, beta, eps).
 *  - "masked multi head attention" CUDA article (2kiu.com/news/6063113),
 *    sections 1, 3.1 and 6.1: causal and padding masks applied as -infinity
 *    before the softmax; an extern "C" wrapper over raw device pointers.
 *  - "Why attention must compute the max first" essay (gsyq.cn/news/340375),
 *    sections 2.3-2.4 (online softmax fused with QK^T and PV), 3.1 (max
 *    shift) and 5.2 (divide the logits by sqrt(d_k)).
 *
 * Conventions for every entry point.
 *  - Pointers are DEVICE pointers owned by the caller (mha_fwd_host: host
 *    tensors, device workspace); the library keeps no per-call state and
 *    allocates no device memory.  (mha_bwd and mha_fwd_host use a workspace
 *    the caller passes in, see mha_bwd_workspace_size and
 *    mha_fwd_host_workspace_size.)
 *  - Layouts are dense and row-major: q, out [B,H,Lq,D]; k, v [B,H,Lk,D];
 *    kv_lengths int32 [B].  Every tensor pointer must be 16-byte aligned.
 *  - Work is enqueued on `stream` (0 = legacy default stream); no entry
 *    point synchronises.  Results are valid once the stream reaches them.
 *  - Host-detectable errors return a negative mha_status and launch nothing.
 *    A launch failure returns MHA_ERR_CUDA.  Device-side waits are bounded:
 *    if one ever expires the kernel records it in a status word (see
 *    mha_device_status) and returns instead of hanging.
 *  - Values at masked key positions must be finite: a masked key's weight
 *    is exactly zero, and 0 * finite = 0.
 */
#ifndef MHA_GB300_H
#define MHA_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MHA_API __attribute__((visibility("default")))
#else
#define MHA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MHA_OK = 0,
    MHA_ERR_INVALID_ARG = -1,   /* null pointer, non-positive size, bad scale/eps, bad mask */
    MHA_ERR_UNSUPPORTED = -2,   /* D not in {64, 128}, dtype not handled by this entry point */
    MHA_ERR_MISALIGNED = -3,    /* a tensor pointer is not 16-byte aligned */
    MHA_ERR_CUDA = -4,          /* the CUDA runtime or driver reported an error */
    MHA_ERR_DEVICE = -5,        /* a kernel's bounded wait expired (see mha_device_status) */
    MHA_ERR_TOO_LARGE = -6      /* problem larger than a fixed-size scratch area allows */
} mha_status;

/* Mask kinds: bit flags, combinable (MHA_MASK_CAUSAL | MHA_MASK_KV_LEN). */
enum { MHA_MASK_NONE = 0, MHA_MASK_CAUSAL = 1, MHA_MASK_KV_LEN = 2 };

/* Element types of q/k/v/out (and x_q).  MHA_F32 runs on the tcgen05 tensor
 * cores with a three-term TF32 split when D = 64, on CUDA-core FFMA when
 * D = 128; MHA_BF16 runs on tcgen05 tensor cores.  Both accumulate in fp32. */
enum { MHA_F32 = 0, MHA_BF16 = 1 };

/*
 * mha_fwd -- fused masked multi-head attention forward.
 *   q           [B,H,Lq,D] of `dtype`
 *   k, v        [B,H,Lk,D] of `dtype`
 *   mask_kind   MHA_MASK_* bits.  Causal alignment is top-left: key j is
 *               visible to query i iff j <= i (also when Lq != Lk).
 *   kv_lengths  device int32 [B]; read only when MHA_MASK_KV_LEN is set (it
 *               must then be non-NULL).  Keys j >= kv_lengths[b] are hidden
 *               for every query row of batch b.  Values are clamped to
 *               [0, Lk] on the device; 0 gives all-zero output rows.
 *   out         [B,H,Lq,D] of `dtype`, written once.  Must not alias inputs.
 *   B, H, Lq    >= 0 (a zero extent is a no-op); Lk >= 0 (0 gives zeros).
 *   D           64 or 128.
 *   scale       logit multiplier, finite and > 0 (usually 1/sqrt(D)).
 *   dtype       MHA_F32 or MHA_BF16.
 *   stream      CUDA stream the kernel is enqueued on.
 * Returns MHA_OK or a negative mha_status.
 */
MHA_API int mha_fwd(const void *q, const void *k, const void *v, int mask_kind,
            const int32_t *kv_lengths, void *out, int B, int H, int Lq, int Lk,
            int D, float scale, int dtype, cudaStream_t stream);

/*
 * mha_fwd_lse -- mha_fwd that also writes each row's log-sum-exp, the
 * statistic the backward pass forms the softmax weights from again:
 *     lse[b,h,i] = log sum_{visible j} exp(s_ij)   (natural log, fp32)
 * and -INFINITY for a row with no visible key.  ("Why attention must compute
 * the max first", gsyq.cn, sections 2.1 and 3.1: it is the row maximum plus
 * the log of the shifted sum, both already held by the online softmax.)
 *   lse         device fp32 [B,H,Lq], 16-byte aligned, written once.
 *   dtype       MHA_F32 or MHA_BF16 (self-attention, every kernel of
 *               mha_fwd: the statistic comes from each kernel's own running
 *               maximum and sum).
 * Other arguments, layouts and errors as for mha_fwd.
 */
MHA_API int mha_fwd_lse(const void *q, const void *k, const void *v, int mask_kind,
                        const int32_t *kv_lengths, void *out, float *lse, int B, int H,
                        int Lq, int Lk, int D, float scale, int dtype, cudaStream_t stream);

/*
 * mha_fwd_host -- mha_fwd on tensors in HOST memory: the call copies q, k, v
 * (and kv_lengths) to the device, runs the forward and copies out back, with
 * the copies and the kernels of successive pieces overlapped.  The problems
 * are taken in pieces of consecutive heads of one batch (contiguous in every
 * tensor); each piece goes through one of two device slots in `workspace`:
 * its inputs are copied in on one internal stream while the previous piece
 * is computed on `stream` and the one before is copied out on another, so
 * the link carries inputs and outputs at the same time and the kernels run
 * behind the copies.  Results are identical to mha_fwd's on the same data.
 *   q, k, v, out, kv_lengths   HOST pointers, layouts as for mha_fwd
 *               (kv_lengths host int32 [B]).  Page-locked memory
 *               (cudaHostAlloc / cudaHostRegister) gives asynchronous,
 *               overlapped copies; pageable memory works but its copies are
 *               staged by the driver.  out must not overlap the inputs.
 *               The inputs are read, and out written, asynchronously: they
 *               must stay valid and untouched until `stream` reaches the end
 *               of the call.
 *   workspace   device scratch of at least mha_fwd_host_workspace_size(...)
 *               bytes, 16-byte aligned, owned by the caller, not used by
 *               anything else until `stream` reaches the end of the call.
 *   workspace_bytes  its size; too small returns MHA_ERR_INVALID_ARG.
 *   stream      every copy and kernel of the call is ordered after the work
 *               already enqueued on it, and the work enqueued on it later is
 *               ordered after them (two internal streams, created and
 *               released by the call, carry the copies).
 * Other arguments and errors as for mha_fwd.  Returns MHA_OK or a negative
 * mha_status.
 */
MHA_API int mha_fwd_host(const void *q, const void *k, const void *v, int mask_kind,
                         const int32_t *kv_lengths, void *out, int B, int H, int Lq, int Lk,
                         int D, float scale, int dtype, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * mha_fwd_host_workspace_size -- bytes of device workspace mha_fwd_host
 * needs for these sizes (two slots of one piece's q, k, v and out, plus the
 * lengths); 0 for an empty problem or an unsupported argument.
 */
MHA_API size_t mha_fwd_host_workspace_size(int B, int H, int Lq, int Lk, int D, int dtype);

/*
 * mha_bwd -- backward pass of mha_fwd: the gradients of the loss
 * sum(dout * O) with respect to q, k and v.  With p_ij the softmax weight
 * (formed again as exp(s_ij - lse_i) at visible positions, exactly 0 at
 * hidden ones) and the softmax Jacobian d p_ij / d s_ik = p_ij (delta_jk -
 * p_ik) ("Why attention must compute the max first", gsyq.cn, section 3.3):
 *     dP_ij = dout_i . v_j,   Delta_i = dout_i . o_i  (= sum_j p_ij dP_ij)
 *     dS_ij = p_ij (dP_ij - Delta_i)
 *     dv_j = sum_i p_ij dout_i
 *     dq_i = scale * sum_j dS_ij k_j,   dk_j = scale * sum_i dS_ij q_i
 * A row with no visible key passes no gradient; a key no row can see gets
 * zero dk and dv.
 *   q, k, v, mask_kind, kv_lengths, B, H, Lq, Lk, D, scale
 *               exactly as given to the forward call.
 *   out         the forward's output O [B,H,Lq,D].
 *   dout        dL/dO [B,H,Lq,D].
 *   lse         the forward's row log-sum-exp [B,H,Lq] (mha_fwd_lse).
 *   dq          [B,H,Lq,D]; dk, dv [B,H,Lk,D]: outputs of `dtype`, fully
 *               written (for fp32, dq is accumulated with atomic adds, so
 *               its last bits can differ between runs).  Must not alias any
 *               input.
 *   dtype       MHA_F32 or MHA_BF16: q, k, v, out, dout and the gradients
 *               all of that type, rounded once (to nearest even) for bf16.
 *   workspace   device scratch of at least mha_bwd_workspace_size(...) bytes,
 *               16-byte aligned, owned by the caller; its contents on entry
 *               do not matter and on return are unspecified.  It must not be
 *               used by anything else until the call's kernels have run.
 *   workspace_bytes  its size; too small (or a null workspace when a
 *               nonzero size is needed) returns MHA_ERR_INVALID_ARG.
 * Kernels.  fp32: CUDA-core FFMA, a row pass (Delta into the workspace, dq =
 * 0) and a key-tile kernel adding dq with fp32 atomics (its last bits can
 * differ between runs).  bf16 (default): the tensor cores, fp32 accumulation
 * in TMEM, P and dS rounded to bf16 for the products; the row pass (Delta)
 * and one launch holding two kinds of tile, interleaved heaviest first:
 * key-stationary tiles that write dk and dv, and query-stationary tiles that
 * write dq -- every element written once, the same on every run.  bf16 with
 * the CUDA-core test hook (mha_testing.h): fp32 arithmetic, dq through an
 * fp32 accumulator in the workspace and a conversion pass.
 * The library allocates no device memory.  Lq == 0 with Lk > 0 writes zero
 * dk and dv.  Returns MHA_OK or a negative mha_status.
 */
MHA_API int mha_bwd(const void *q, const void *k, const void *v, const void *out,
                    const void *dout, const float *lse, int mask_kind,
                    const int32_t *kv_lengths, void *dq, void *dk, void *dv, int B, int H,
                    int Lq, int Lk, int D, float scale, int dtype, void *workspace,
                    size_t workspace_bytes, cudaStream_t stream);

/*
 * mha_bwd_workspace_size -- bytes of workspace mha_bwd needs for these sizes
 * on the calling thread's kernel choice: 4*B*H*Lq (rounded up to 256) for
 * the per-row Delta, plus 4*B*H*Lq*D for bf16 on the CUDA-core test path.
 * Returns 0 for an empty problem or invalid sizes.
 */
MHA_API size_t mha_bwd_workspace_size(int B, int H, int Lq, int D, int dtype);

/*
 * prenorm_cross_attn_fwd -- Pre-LayerNorm cross-attention forward
 * (cms365.cn answer, steps two and three).  For every (b, i):
 *     xhat = (x_q[b,i,:] - mean) / sqrt(var + eps) * gamma + beta
 * over the H*D features of the row (biased variance), Q[b,h,i,:] is the
 * head-h slice xhat[h*D:(h+1)*D], and the attention above runs with the
 * padding mask only (kv_lengths, or none when it is NULL).  One kernel runs
 * on `stream` and allocates nothing: it groups the heads of each block of
 * 256 query rows into chunks, forms each row's mean and 1/sqrt(var + eps)
 * from the full row of x inside the kernel (in fp32, two passes; at D = 64
 * before any attention work, shared by the two CTAs of a thread-block
 * cluster that take chunks of the same rows), loads each head's slice of x
 * with TMA and normalises it in shared memory before the first QK^T
 * product.
 *   x_q         [B,Lq,H*D] bf16 (query-side activations)
 *   gamma, beta fp32 [H*D]
 *   eps         finite, >= 0
 *   k, v        [B,H,Lk,D] bf16 (encoder keys and values)
 *   kv_lengths  device int32 [B] or NULL (all Lk keys visible)
 *   out         [B,Lq,H*D] bf16 (heads merged back into the model dim)
 *   dtype       must be MHA_BF16 (MHA_ERR_UNSUPPORTED otherwise)
 * Other arguments as for mha_fwd.
 */
MHA_API int prenorm_cross_attn_fwd(const void *x_q, const float *gamma, const float *beta,
                           float eps, const void *k, const void *v,
                           const int32_t *kv_lengths, void *out, int B, int H,
                           int Lq, int Lk, int D, float scale, int dtype,
                           cudaStream_t stream);

/*
 * prenorm_cross_attn_residual_fwd -- Pre-LayerNorm cross-attention with the
 * residual add (cms365.cn answer, step four: the attention output is added
 * to the query-side input):
 *     out[b,i,:] = x_q[b,i,:] + (prenorm_cross_attn_fwd output)[b,i,:]
 * The sum is formed in fp32 inside the attention kernel's epilogue and
 * rounded to bf16 once; a row with no visible key returns x_q's row.
 *   Arguments, layouts and errors are those of prenorm_cross_attn_fwd (one
 *   kernel, no allocation).  out must not overlap x_q.
 */
MHA_API int prenorm_cross_attn_residual_fwd(const void *x_q, const float *gamma,
                            const float *beta, float eps, const void *k,
                            const void *v, const int32_t *kv_lengths, void *out,
                            int B, int H, int Lq, int Lk, int D, float scale,
                            int dtype, cudaStream_t stream);

/*
 * prenorm_cross_attn_fwd_noalloc -- the same computation as
 * prenorm_cross_attn_fwd, for callers that cannot let a library allocate
 * device memory: for example a serving runtime that reserves all GPU memory
 * for its own pools at start-up and gives libraries only the buffers it
 * planned, or a latency-critical loop in which an allocation could block or
 * fail.  (No counterpart on the pages; this is an interface addition.)
 *   Arguments, layouts and results are those of prenorm_cross_attn_fwd,
 *   bit for bit.  (prenorm_cross_attn_fwd forms the row statistics inside
 *   its one kernel and allocates nothing either; this entry point runs them
 *   as a separate pass first, into the array below.)
 *   Memory: calls no allocator.  The per-row statistics go to a fixed array
 *   of 262144 float2 (2 MiB) that is part of the library's device image and
 *   stays resident on every GPU that loads the library until the process
 *   exits.  B*Lq above 262144 returns MHA_ERR_TOO_LARGE without launching.
 *   Set-up: the first call on each device looks up the array's device
 *   address (cudaGetSymbolAddress) with that device current; make that first
 *   call before any stream capture.
 *   Sharing: every call uses the same array and it keeps the last call's
 *   values (nothing needs clearing: each call writes every row it reads).
 *   Calls whose kernels can overlap on the GPU (different streams, or
 *   different host threads, on one device) race on it; order them.
 */
MHA_API int prenorm_cross_attn_fwd_noalloc(const void *x_q, const float *gamma,
                                           const float *beta, float eps, const void *k,
                                           const void *v, const int32_t *kv_lengths,
                                           void *out, int B, int H, int Lq, int Lk, int D,
                                           float scale, int dtype, cudaStream_t stream);

/* Static, human-readable text for an mha_status value. */
MHA_API const char *mha_strerror(int status);

/*
 * mha_device_status -- read (and optionally clear) the device status words
 * the kernels set; *bits receives their union.
 *   Bits 0-15: a bounded wait expired at wait site k (site numbers are
 *   listed in the kernel sources).  The kernel returned without finishing,
 *   and later launches of the same kernel family return at once, without
 *   writing their outputs, until the bit is cleared.
 *   Bit 16: a forward row with visible keys ended with a softmax sum that
 *   is not positive and finite ("softmax sum != 1 is an error", cms365.cn
 *   answer, closing notes); bit 17: a forward output element is not finite.
 *   Both arise only from non-finite inputs; they do not stop later launches.
 * Synchronous: copies from the current device.  Returns MHA_OK or
 * MHA_ERR_CUDA.
 */
MHA_API int mha_device_status(uint32_t *bits, int clear);

#ifdef __cplusplus
}
#endif

#endif /* MHA_GB300_H */
