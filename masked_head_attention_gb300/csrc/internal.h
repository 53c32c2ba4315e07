// internal.h -- host-side declarations shared by the C-ABI layer (api.cu) and
// the kernel translation units.  Not part of the public interface.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace mha {

// Programmatic dependent launch.  Every kernel of this library is launched
// with it allowed, so its grid may be scheduled while the previous kernel of
// the stream is still finishing; each kernel starts with pdl_wait(), which
// returns once the previous grid has completed and its memory writes are
// visible, before it reads or writes global memory, and calls pdl_trigger()
// to let the next grid be scheduled in turn.  Without the attribute (or with
// a previous kernel that never triggers) both are no-ops and ordinary stream
// order applies.  The thread-local switch is a test hook (mha_set_pdl).
bool pdl_enabled();
void set_pdl(int on);

#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

// cudaLaunchKernelEx with programmatic dependent launch allowed (when
// pdl_enabled()) and up to one more launch attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, const cudaLaunchAttribute *extra,
                          Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (extra != nullptr) attr[n++] = *extra;
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// SM count and L2 size of the current device (cached per device).
struct DeviceInfo {
    int sms = 0;
    int l2 = 0;
};
DeviceInfo device_info();
// Raises `func`'s dynamic shared-memory limit to `bytes` on the current
// device, once per (function, device); thread-safe.  Function attributes
// belong to a device's context, so a process that launches on several GPUs
// sets each one.
cudaError_t set_smem_limit(const void *func, size_t bytes);

// cuTensorMapEncodeTiled from the driver (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// fp32 path (fwd_f32.cu): the 3xTF32 tensor-core kernel where it applies,
// else the CUDA-core kernels.  Arguments already validated.  `lse` (fp32
// [B,H,Lq], natural log) is written when non-null.  *driver_err receives a
// nonzero CUresult when tensor-map encoding failed.
cudaError_t launch_fwd_f32(const float *q, const float *k, const float *v,
                           const int32_t *kv_lengths, float *out, float *lse, int B, int H,
                           int Lq, int Lk, int D, int mask_kind, float scale,
                           cudaStream_t stream, int *driver_err);

// fp32 on the tensor cores with the three-term TF32 split (fwd_tf32.cu):
// D = 64 only (tf32x3_applies).  `lse` is written when non-null.  Returns
// cudaErrorInvalidValue with *driver_err set when tensor-map encoding fails.
bool tf32x3_applies(int D);
cudaError_t launch_fwd_tf32x3(const float *q, const float *k, const float *v,
                              const int32_t *kv_lengths, float *out, float *lse, int B, int H,
                              int Lq, int Lk, int D, int mask_kind, float scale,
                              cudaStream_t stream, int *driver_err);

// Backward (bwd.cu): dq, dk, dv from q, k, v, the forward output o, its row
// log-sum-exp and dout.  `delta` is device scratch of B*H*Lq floats.  fp32:
// dq is accumulated in place.  bf16: `dq_acc` is fp32 scratch of B*H*Lq*D
// floats, converted into dq at the end.
cudaError_t launch_bwd_f32(const float *q, const float *k, const float *v, const float *o,
                           const float *dout, const float *lse, const int32_t *kv_lengths,
                           float *dq, float *dk, float *dv, float *delta, int B, int H, int Lq,
                           int Lk, int D, int mask_kind, float scale, cudaStream_t stream);
// bf16 backward on the tensor cores (bwd_bf16.cu): key-stationary dK/dV tiles
// and query-stationary dQ tiles in one launch, from the forward's log-sum-exp
// and Delta (B*H*Lq floats each).  Every gradient element written once.
cudaError_t launch_bwd_bf16_tensor(const void *q, const void *k, const void *v, const void *dout,
                                   const float *lse, const float *delta, const int32_t *kv_lengths,
                                   void *dq, void *dk, void *dv, int B, int H, int Lq, int Lk, int D,
                                   int mask_kind, float scale, cudaStream_t stream, int *driver_err);
// The row pass alone (Delta = dout . o), for the tensor-core backward.
cudaError_t launch_bwd_row_delta_bf16(const void *o, const void *dout, float *delta, int64_t rows,
                                      int D, cudaStream_t stream);
// 3-D bf16 tensor map over a dense [d2][d1][d0] array, {64, box_rows, 1} box,
// 128-byte swizzle (fwd_bf16.cu).
CUresult encode_bf16_3d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1,
                        uint64_t d2, uint32_t box_rows);

cudaError_t launch_bwd_bf16(const void *q, const void *k, const void *v, const void *o,
                            const void *dout, const float *lse, const int32_t *kv_lengths,
                            void *dq, void *dk, void *dv, float *dq_acc, float *delta, int B,
                            int H, int Lq, int Lk, int D, int mask_kind, float scale,
                            cudaStream_t stream);

// bf16 tensor-core path (fwd_bf16.cu).  x/gamma/beta are null for plain
// self-attention; for the Pre-LN variant q is null and x/gamma/beta are set.
struct Bf16Call {
    const void *q;          // [B,H,Lq,D] (self-attention) or null
    const void *x;          // [B,Lq,H*D] (Pre-LN) or null
    const void *residual;   // Pre-LN: added to the output ([B,Lq,H*D], i.e. x) or null
    const float *gamma;
    const float *beta;
    float eps;
    const void *k;          // [B,H,Lk,D]
    const void *v;
    const int32_t *kv_lengths;
    void *out;              // [B,H,Lq,D] or [B,Lq,H*D]
    float *lse;             // self-attention: row log-sum-exp [B,H,Lq] (natural log), or null
    int B, H, Lq, Lk, D;
    int mask_kind;
    float scale;
};

// Returns cudaSuccess or the first CUDA error; *driver_err receives a
// nonzero CUresult when tensor-map encoding failed.  Pre-LN variant: with
// `ln_stats` null the attention kernel forms every row's (mean,
// 1/sqrt(var + eps)) itself (one launch, no scratch); otherwise `ln_stats` is
// device scratch of B*Lq float2 that a standalone pass fills first.
cudaError_t launch_fwd_bf16(const Bf16Call &c, cudaStream_t stream, int *driver_err,
                            float2 *ln_stats);

// Decode path (decode_bf16.cu): bf16 self-attention with at most
// kDecodeMaxRows query rows, keys split over a thread-block cluster.
constexpr int kDecodeMaxRows = 8;
bool decode_applies(const Bf16Call &c);
cudaError_t launch_decode_bf16(const Bf16Call &c, int num_sms, cudaStream_t stream);
void set_decode_override(int which);
void set_decode_splits(int splits);

// Diagnostic single-tile tcgen05 GEMM (fwd_bf16.cu).
cudaError_t launch_selftest_umma(int variant, int K_or_N, const void *a, const void *b,
                                 float *c, cudaStream_t stream, int *driver_err);

// No-allocation Pre-LN: device address of the fixed row-statistics array
// (looked up once per device, with that device current).  Fails with
// cudaErrorInvalidValue when `rows` exceeds kNoAllocMaxRows.
constexpr int64_t kNoAllocMaxRows = 262144;
cudaError_t noalloc_ln_stats(int64_t rows, float2 **ptr);

// Device status word and wait limit of each unit with bounded waits or
// numeric flags (fwd_bf16.cu, fwd_tf32.cu, bwd_bf16.cu, decode_bf16.cu; each
// keeps its own):
//   op 0: *bits = the word, cleared afterwards when value != 0;
//   op 1: OR `value` into the word;
//   op 2: wait limit = `value` ns (0 restores the default of 2 s).
cudaError_t status_ctl_fwd_bf16(int op, uint64_t value, uint32_t *bits);
cudaError_t status_ctl_fwd_tf32(int op, uint64_t value, uint32_t *bits);
cudaError_t status_ctl_bwd_bf16(int op, uint64_t value, uint32_t *bits);
cudaError_t status_ctl_decode_bf16(int op, uint64_t value, uint32_t *bits);
constexpr int kStatusUnits = 4;

// Launch-configuration overrides used by tests and benchmark sweeps (0 = default).
void set_bf16_grid_override(int ctas);

// Launch plan of the Pre-LN bf16 forward (host logic only): heads per chunk G,
// head groups per row block n_hg = H / G, CTAs per cluster cs (2 when the
// prologue's shared statistics pair up), chunks whose statistics the prologue
// forms per CTA (0: formed at the chunk starts, or read from the caller's
// array when stats_given), the grid and the chunk count.
struct PrenormPlan {
    int G, n_hg, cs, pre_chunks, grid;
    long long n_chunks;
};
PrenormPlan plan_prenorm(int B, int H, int Lq, int Lk, int D, int grid, bool stats_given);
void set_f32_kernel_override(int which);

}  // namespace mha
