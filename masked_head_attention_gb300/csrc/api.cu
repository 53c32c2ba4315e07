// api.cu -- the extern "C" boundary of libmha.so: argument validation,
// dispatch by (entry point, dtype, D), and status reporting.  Host code only;
// the kernels live in fwd_f32.cu, fwd_tf32.cu, fwd_bf16.cu, decode_bf16.cu and
// bwd.cu.
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/mha.h"
#include "../../include/mha_testing.h"
#include "internal.h"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA; }

// The units with bounded waits, in the numbering of mha_test_set_device_status.
cudaError_t status_ctl(int unit, int op, uint64_t value, uint32_t *bits) {
    switch (unit) {
        case 0: return mha::status_ctl_fwd_bf16(op, value, bits);
        case 1: return mha::status_ctl_fwd_tf32(op, value, bits);
        case 2: return mha::status_ctl_bwd_bf16(op, value, bits);
        case 3: return mha::status_ctl_decode_bf16(op, value, bits);
        default: return cudaErrorInvalidValue;
    }
}

// Backward kernel choice: 0 automatic (bf16 on the tensor cores, fp32 on CUDA
// cores), 1 CUDA cores for both.
thread_local int g_bwd_kernel = 0;

// Programmatic dependent launch on (1, the default) or off (0); test hook.
thread_local int g_pdl = 1;

// Shared checks of the shape arguments; 1 means "nothing to do".
int check_shape(int B, int H, int Lq, int Lk, int D, float scale, int *empty) {
    *empty = 0;
    if (B < 0 || H < 0 || Lq < 0 || Lk < 0) return MHA_ERR_INVALID_ARG;
    if (!(std::isfinite(scale) && scale > 0.f)) return MHA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return MHA_ERR_UNSUPPORTED;
    if (B > 65535) return MHA_ERR_INVALID_ARG;                 // grid z of the fp32 path
    const int64_t n_qt = ((int64_t)Lq + 127) / 128;
    if ((int64_t)B * H * (n_qt > 0 ? n_qt : 1) > 0x7fffffffLL) return MHA_ERR_INVALID_ARG;
    if (B == 0 || H == 0 || Lq == 0) *empty = 1;
    return MHA_OK;
}

}  // namespace

namespace mha {
bool pdl_enabled() { return g_pdl != 0; }
void set_pdl(int on) { g_pdl = on != 0 ? 1 : 0; }
}  // namespace mha

extern "C" {

int mha_fwd(const void *q, const void *k, const void *v, int mask_kind,
            const int32_t *kv_lengths, void *out, int B, int H, int Lq, int Lk, int D,
            float scale, int dtype, cudaStream_t stream) {
    int empty = 0;
    int st = check_shape(B, H, Lq, Lk, D, scale, &empty);
    if (st != MHA_OK) return st;
    if (mask_kind < 0 || mask_kind > (MHA_MASK_CAUSAL | MHA_MASK_KV_LEN)) return MHA_ERR_INVALID_ARG;
    if (dtype != MHA_F32 && dtype != MHA_BF16) return MHA_ERR_UNSUPPORTED;
    if (empty) return MHA_OK;
    if (!q || !out || (Lk > 0 && (!k || !v))) return MHA_ERR_INVALID_ARG;
    if ((mask_kind & MHA_MASK_KV_LEN) && !kv_lengths) return MHA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || (Lk > 0 && (!aligned16(k) || !aligned16(v))))
        return MHA_ERR_MISALIGNED;
    if (dtype == MHA_F32) {
        int drv = 0;
        const cudaError_t e = mha::launch_fwd_f32(
            static_cast<const float *>(q), static_cast<const float *>(k),
            static_cast<const float *>(v), kv_lengths, static_cast<float *>(out), nullptr, B, H,
            Lq, Lk, D, mask_kind, scale, stream, &drv);
        return drv != 0 ? MHA_ERR_CUDA : from_cuda(e);
    }
    mha::Bf16Call c{};
    c.q = q;
    c.k = k;
    c.v = v;
    c.kv_lengths = kv_lengths;
    c.out = out;
    c.B = B;
    c.H = H;
    c.Lq = Lq;
    c.Lk = Lk;
    c.D = D;
    c.mask_kind = mask_kind;
    c.scale = scale;
    int drv = 0;
    cudaError_t e = mha::launch_fwd_bf16(c, stream, &drv, nullptr);
    if (drv != 0) return MHA_ERR_CUDA;
    return from_cuda(e);
}

int mha_fwd_lse(const void *q, const void *k, const void *v, int mask_kind,
                const int32_t *kv_lengths, void *out, float *lse, int B, int H, int Lq, int Lk,
                int D, float scale, int dtype, cudaStream_t stream) {
    int empty = 0;
    int st = check_shape(B, H, Lq, Lk, D, scale, &empty);
    if (st != MHA_OK) return st;
    if (mask_kind < 0 || mask_kind > (MHA_MASK_CAUSAL | MHA_MASK_KV_LEN)) return MHA_ERR_INVALID_ARG;
    if (dtype != MHA_F32 && dtype != MHA_BF16) return MHA_ERR_UNSUPPORTED;
    if (empty) return MHA_OK;
    if (!q || !out || !lse || (Lk > 0 && (!k || !v))) return MHA_ERR_INVALID_ARG;
    if ((mask_kind & MHA_MASK_KV_LEN) && !kv_lengths) return MHA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(lse) ||
        (Lk > 0 && (!aligned16(k) || !aligned16(v))))
        return MHA_ERR_MISALIGNED;
    int drv = 0;
    cudaError_t e;
    if (dtype == MHA_F32) {
        e = mha::launch_fwd_f32(static_cast<const float *>(q), static_cast<const float *>(k),
                                static_cast<const float *>(v), kv_lengths,
                                static_cast<float *>(out), lse, B, H, Lq, Lk, D, mask_kind, scale,
                                stream, &drv);
    } else {
        mha::Bf16Call c{};
        c.q = q;
        c.k = k;
        c.v = v;
        c.kv_lengths = kv_lengths;
        c.out = out;
        c.lse = lse;
        c.B = B;
        c.H = H;
        c.Lq = Lq;
        c.Lk = Lk;
        c.D = D;
        c.mask_kind = mask_kind;
        c.scale = scale;
        e = mha::launch_fwd_bf16(c, stream, &drv, nullptr);
    }
    return drv != 0 ? MHA_ERR_CUDA : from_cuda(e);
}

size_t mha_bwd_workspace_size(int B, int H, int Lq, int D, int dtype) {
    if (B <= 0 || H <= 0 || Lq <= 0 || (D != 64 && D != 128)) return 0;
    if (dtype != MHA_F32 && dtype != MHA_BF16) return 0;
    const size_t rows = (size_t)B * H * Lq;
    const size_t delta_bytes = (sizeof(float) * rows + 255) & ~(size_t)255;
    const bool tensor = dtype == MHA_BF16 && g_bwd_kernel != 1;
    return delta_bytes + (dtype == MHA_BF16 && !tensor ? sizeof(float) * rows * D : 0);
}

int mha_bwd(const void *q, const void *k, const void *v, const void *out, const void *dout,
            const float *lse, int mask_kind, const int32_t *kv_lengths, void *dq, void *dk,
            void *dv, int B, int H, int Lq, int Lk, int D, float scale, int dtype,
            void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    int empty = 0;
    int st = check_shape(B, H, Lq, Lk, D, scale, &empty);
    if (st != MHA_OK) return st;
    if (mask_kind < 0 || mask_kind > (MHA_MASK_CAUSAL | MHA_MASK_KV_LEN)) return MHA_ERR_INVALID_ARG;
    if (dtype != MHA_F32 && dtype != MHA_BF16) return MHA_ERR_UNSUPPORTED;
    // Lq == 0 with keys present still owes zero dk and dv.
    if (B == 0 || H == 0 || (Lq == 0 && Lk == 0)) return MHA_OK;
    (void)empty;
    if ((Lq > 0 && (!q || !out || !dout || !lse || !dq)) || (Lk > 0 && (!k || !v || !dk || !dv)))
        return MHA_ERR_INVALID_ARG;
    if ((mask_kind & MHA_MASK_KV_LEN) && !kv_lengths) return MHA_ERR_INVALID_ARG;
    // Per-row Delta = dout . o (and, for bf16 on CUDA cores, the fp32 dq
    // accumulator) live in the caller's workspace.
    const size_t need = mha_bwd_workspace_size(B, H, Lq, D, dtype);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return MHA_ERR_INVALID_ARG;
    if ((Lq > 0 && (!aligned16(q) || !aligned16(out) || !aligned16(dout) || !aligned16(lse) ||
                    !aligned16(dq))) ||
        (Lk > 0 && (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv))) ||
        (need > 0 && !aligned16(workspace)))
        return MHA_ERR_MISALIGNED;
    const bool tensor = dtype == MHA_BF16 && g_bwd_kernel != 1;
    const size_t rows = (size_t)B * H * Lq;
    const size_t delta_bytes = (sizeof(float) * rows + 255) & ~(size_t)255;
    char *ws = static_cast<char *>(workspace);
    float *delta = need > 0 ? reinterpret_cast<float *>(ws) : nullptr;
    cudaError_t e;
    int drv = 0;
    if (tensor) {
        e = mha::launch_bwd_row_delta_bf16(out, dout, delta, (int64_t)rows, D, stream);
        if (e == cudaSuccess)
            e = mha::launch_bwd_bf16_tensor(q, k, v, dout, lse, delta, kv_lengths, dq, dk, dv, B, H,
                                            Lq, Lk, D, mask_kind, scale, stream, &drv);
    } else if (dtype == MHA_F32)
        e = mha::launch_bwd_f32(static_cast<const float *>(q), static_cast<const float *>(k),
                                static_cast<const float *>(v), static_cast<const float *>(out),
                                static_cast<const float *>(dout), lse, kv_lengths,
                                static_cast<float *>(dq), static_cast<float *>(dk),
                                static_cast<float *>(dv), delta, B, H, Lq, Lk, D, mask_kind, scale,
                                stream);
    else
        e = mha::launch_bwd_bf16(q, k, v, out, dout, lse, kv_lengths, dq, dk, dv,
                                 need > 0 ? reinterpret_cast<float *>(ws + delta_bytes) : nullptr,
                                 delta, B, H, Lq, Lk, D, mask_kind, scale, stream);
    if (drv != 0) return MHA_ERR_CUDA;
    return from_cuda(e);
}

}  // extern "C"

namespace {

// Pre-LN cross-attention: one kernel, which forms the row statistics of x
// itself; `residual` is x_q for the residual variant, else null.
int prenorm_fused(const void *x_q, const float *gamma, const float *beta, float eps,
                  const void *k, const void *v, const int32_t *kv_lengths, void *out, int B,
                  int H, int Lq, int Lk, int D, float scale, int dtype, cudaStream_t stream,
                  const void *residual) {
    int empty = 0;
    int st = check_shape(B, H, Lq, Lk, D, scale, &empty);
    if (st != MHA_OK) return st;
    if (dtype != MHA_BF16) return MHA_ERR_UNSUPPORTED;
    if (!(std::isfinite(eps) && eps >= 0.f)) return MHA_ERR_INVALID_ARG;
    if ((int64_t)H * D > 65536) return MHA_ERR_INVALID_ARG;
    if (empty) return MHA_OK;
    if (!x_q || !gamma || !beta || !out || (Lk > 0 && (!k || !v))) return MHA_ERR_INVALID_ARG;
    if (!aligned16(x_q) || !aligned16(out) || !aligned16(gamma) || !aligned16(beta) ||
        (Lk > 0 && (!aligned16(k) || !aligned16(v))))
        return MHA_ERR_MISALIGNED;
    mha::Bf16Call c{};
    c.x = x_q;
    c.residual = residual;
    c.gamma = gamma;
    c.beta = beta;
    c.eps = eps;
    c.k = k;
    c.v = v;
    c.kv_lengths = kv_lengths;
    c.out = out;
    c.B = B;
    c.H = H;
    c.Lq = Lq;
    c.Lk = Lk;
    c.D = D;
    c.mask_kind = kv_lengths ? MHA_MASK_KV_LEN : MHA_MASK_NONE;
    c.scale = scale;
    int drv = 0;
    cudaError_t e = mha::launch_fwd_bf16(c, stream, &drv, nullptr);
    if (drv != 0) return MHA_ERR_CUDA;
    return from_cuda(e);
}

}  // namespace

extern "C" {

int prenorm_cross_attn_fwd(const void *x_q, const float *gamma, const float *beta, float eps,
                           const void *k, const void *v, const int32_t *kv_lengths, void *out,
                           int B, int H, int Lq, int Lk, int D, float scale, int dtype,
                           cudaStream_t stream) {
    return prenorm_fused(x_q, gamma, beta, eps, k, v, kv_lengths, out, B, H, Lq, Lk, D, scale,
                         dtype, stream, nullptr);
}

int prenorm_cross_attn_residual_fwd(const void *x_q, const float *gamma, const float *beta,
                                    float eps, const void *k, const void *v,
                                    const int32_t *kv_lengths, void *out, int B, int H, int Lq,
                                    int Lk, int D, float scale, int dtype, cudaStream_t stream) {
    return prenorm_fused(x_q, gamma, beta, eps, k, v, kv_lengths, out, B, H, Lq, Lk, D, scale,
                         dtype, stream, x_q);
}

int prenorm_cross_attn_fwd_noalloc(const void *x_q, const float *gamma, const float *beta,
                                   float eps, const void *k, const void *v,
                                   const int32_t *kv_lengths, void *out, int B, int H, int Lq,
                                   int Lk, int D, float scale, int dtype, cudaStream_t stream) {
    int empty = 0;
    int st = check_shape(B, H, Lq, Lk, D, scale, &empty);
    if (st != MHA_OK) return st;
    if (dtype != MHA_BF16) return MHA_ERR_UNSUPPORTED;
    if (!(std::isfinite(eps) && eps >= 0.f)) return MHA_ERR_INVALID_ARG;
    if ((int64_t)H * D > 65536) return MHA_ERR_INVALID_ARG;
    if ((int64_t)B * Lq > mha::kNoAllocMaxRows) return MHA_ERR_TOO_LARGE;
    if (empty) return MHA_OK;
    if (!x_q || !gamma || !beta || !out || (Lk > 0 && (!k || !v))) return MHA_ERR_INVALID_ARG;
    if (!aligned16(x_q) || !aligned16(out) || !aligned16(gamma) || !aligned16(beta) ||
        (Lk > 0 && (!aligned16(k) || !aligned16(v))))
        return MHA_ERR_MISALIGNED;
    float2 *stats = nullptr;
    if (mha::noalloc_ln_stats((int64_t)B * Lq, &stats) != cudaSuccess) return MHA_ERR_CUDA;
    mha::Bf16Call c{};
    c.x = x_q;
    c.gamma = gamma;
    c.beta = beta;
    c.eps = eps;
    c.k = k;
    c.v = v;
    c.kv_lengths = kv_lengths;
    c.out = out;
    c.B = B;
    c.H = H;
    c.Lq = Lq;
    c.Lk = Lk;
    c.D = D;
    c.mask_kind = kv_lengths ? MHA_MASK_KV_LEN : MHA_MASK_NONE;
    c.scale = scale;
    int drv = 0;
    cudaError_t e = mha::launch_fwd_bf16(c, stream, &drv, stats);
    if (drv != 0) return MHA_ERR_CUDA;
    return from_cuda(e);
}

const char *mha_strerror(int status) {
    switch (status) {
        case MHA_OK: return "success";
        case MHA_ERR_INVALID_ARG: return "invalid argument (null pointer, bad size, scale, eps or mask)";
        case MHA_ERR_UNSUPPORTED: return "unsupported configuration (D must be 64 or 128; dtype not handled)";
        case MHA_ERR_MISALIGNED: return "a tensor pointer is not 16-byte aligned";
        case MHA_ERR_CUDA: return "CUDA runtime or driver error";
        case MHA_ERR_DEVICE: return "a kernel's bounded wait expired (see mha_device_status)";
        case MHA_ERR_TOO_LARGE: return "B*Lq exceeds the fixed scratch of prenorm_cross_attn_fwd_noalloc (262144 rows)";
        default: return "unknown status";
    }
}

int mha_device_status(uint32_t *bits, int clear) {
    // Each unit with bounded waits keeps its own word; report their union.
    uint32_t all = 0;
    cudaError_t e = cudaSuccess;
    for (int u = 0; u < mha::kStatusUnits && e == cudaSuccess; ++u) {
        uint32_t w = 0;
        e = status_ctl(u, 0, clear != 0 ? 1 : 0, &w);
        all |= w;
    }
    if (bits) *bits = all;
    return from_cuda(e);
}

int mha_test_set_device_status(int unit, uint32_t bits) {
    if (unit < 0 || unit >= mha::kStatusUnits) return MHA_ERR_INVALID_ARG;
    return from_cuda(status_ctl(unit, 1, bits, nullptr));
}

int mha_test_set_wait_limit_ns(uint64_t ns) {
    cudaError_t e = cudaSuccess;
    for (int u = 0; u < mha::kStatusUnits && e == cudaSuccess; ++u) e = status_ctl(u, 2, ns, nullptr);
    return from_cuda(e);
}

int mha_selftest_umma(int variant, int K_or_N, const void *a, const void *b, float *c,
                      cudaStream_t stream) {
    if (variant < 0 || variant > 2) return MHA_ERR_INVALID_ARG;
    if (K_or_N != 64 && K_or_N != 128) return MHA_ERR_UNSUPPORTED;
    if (!a || !b || !c) return MHA_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(c)) return MHA_ERR_MISALIGNED;
    int drv = 0;
    cudaError_t e = mha::launch_selftest_umma(variant, K_or_N, a, b, c, stream, &drv);
    if (drv != 0) return MHA_ERR_CUDA;
    return from_cuda(e);
}

// Test and benchmark hooks (mha_testing.h); thread-local state.
void mha_set_bf16_grid(int ctas) { mha::set_bf16_grid_override(ctas); }

void mha_set_f32_kernel(int which) { mha::set_f32_kernel_override(which); }

void mha_set_bf16_decode(int mode) { mha::set_decode_override(mode); }

void mha_set_bf16_decode_splits(int splits) { mha::set_decode_splits(splits); }

void mha_set_bwd_kernel(int which) { g_bwd_kernel = (which == 1) ? 1 : 0; }
void mha_set_pdl(int on) { mha::set_pdl(on); }

}  // extern "C"
