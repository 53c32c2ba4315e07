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

// mha_fwd_host: the problems go through the device in pieces of `heads`
// consecutive heads of one batch (contiguous in q, k, v and out), each held in
// one of two workspace slots.  A piece carries at most kHostPieceBytes of q,
// k, v and out unless one head alone is larger.
constexpr int64_t kHostPieceBytes = 64ll << 20;

struct HostPlan {
    int heads = 1;              // heads per piece
    size_t q_bytes = 0;         // one piece of q (and of out)
    size_t k_bytes = 0;         // one piece of k (and of v)
    size_t off_k = 0, off_v = 0, off_out = 0, slot = 0;   // offsets inside a slot
    size_t off_lens = 0;        // after the two slots
    size_t total = 0;
};

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Returns false for an empty problem or unsupported arguments.
bool host_plan(int B, int H, int Lq, int Lk, int D, int dtype, HostPlan *pl) {
    if (B <= 0 || H <= 0 || Lq <= 0 || Lk < 0 || (D != 64 && D != 128)) return false;
    if (dtype != MHA_F32 && dtype != MHA_BF16) return false;
    const int64_t esz = dtype == MHA_F32 ? 4 : 2;
    const int64_t per_head = (2 * (int64_t)Lq + 2 * (int64_t)Lk) * D * esz;
    int heads = 1;
    for (int g = 1; g <= H; ++g)
        if (H % g == 0 && g * per_head <= kHostPieceBytes) heads = g;
    pl->heads = heads;
    pl->q_bytes = (size_t)heads * Lq * D * esz;
    pl->k_bytes = (size_t)heads * Lk * D * esz;
    pl->off_k = round256(pl->q_bytes);
    pl->off_v = pl->off_k + round256(pl->k_bytes);
    pl->off_out = pl->off_v + round256(pl->k_bytes);
    pl->slot = pl->off_out + round256(pl->q_bytes);
    pl->off_lens = 2 * pl->slot;
    pl->total = pl->off_lens + round256(sizeof(int32_t) * (size_t)B);
    return true;
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

size_t mha_fwd_host_workspace_size(int B, int H, int Lq, int Lk, int D, int dtype) {
    HostPlan pl;
    return host_plan(B, H, Lq, Lk, D, dtype, &pl) ? pl.total : 0;
}

int mha_fwd_host(const void *q, const void *k, const void *v, int mask_kind,
                 const int32_t *kv_lengths, void *out, int B, int H, int Lq, int Lk, int D,
                 float scale, int dtype, void *workspace, size_t workspace_bytes,
                 cudaStream_t stream) {
    int empty = 0;
    int st = check_shape(B, H, Lq, Lk, D, scale, &empty);
    if (st != MHA_OK) return st;
    if (mask_kind < 0 || mask_kind > (MHA_MASK_CAUSAL | MHA_MASK_KV_LEN)) return MHA_ERR_INVALID_ARG;
    if (dtype != MHA_F32 && dtype != MHA_BF16) return MHA_ERR_UNSUPPORTED;
    if (empty) return MHA_OK;
    if (!q || !out || (Lk > 0 && (!k || !v))) return MHA_ERR_INVALID_ARG;
    const bool use_lens = (mask_kind & MHA_MASK_KV_LEN) != 0;
    if (use_lens && !kv_lengths) return MHA_ERR_INVALID_ARG;
    HostPlan pl;
    if (!host_plan(B, H, Lq, Lk, D, dtype, &pl)) return MHA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < pl.total) return MHA_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return MHA_ERR_MISALIGNED;

    // Two copy streams (in, out) and the events that order them with the
    // kernels on `stream`; slot s's in-copy waits for the out-copy of the
    // piece that used the slot before (which itself followed that piece's
    // kernel).
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t start = nullptr, done_in[2] = {}, done_kernel[2] = {}, done_out[2] = {};
    bool ok = cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&start, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < 2; ++i)
        ok = cudaEventCreateWithFlags(&done_in[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&done_kernel[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&done_out[i], cudaEventDisableTiming) == cudaSuccess;
    // Everything already on `stream` (e.g. an earlier call using the same
    // workspace) comes first.
    ok = ok && cudaEventRecord(start, stream) == cudaSuccess &&
         cudaStreamWaitEvent(s_in, start, 0) == cudaSuccess &&
         cudaStreamWaitEvent(s_out, start, 0) == cudaSuccess;
    char *ws = static_cast<char *>(workspace);
    const int32_t *dlens = nullptr;
    if (ok && use_lens) {
        ok = cudaMemcpyAsync(ws + pl.off_lens, kv_lengths, sizeof(int32_t) * (size_t)B,
                             cudaMemcpyHostToDevice, s_in) == cudaSuccess;
        dlens = reinterpret_cast<const int32_t *>(ws + pl.off_lens);
    }
    st = ok ? MHA_OK : MHA_ERR_CUDA;
    const int per_batch = H / pl.heads;
    const int64_t pieces = (int64_t)B * per_batch;
    for (int64_t c = 0; st == MHA_OK && c < pieces; ++c) {
        const int b = (int)(c / per_batch), h0 = (int)(c % per_batch) * pl.heads, sl = (int)(c & 1);
        char *slot = ws + sl * pl.slot;
        const size_t first = (size_t)b * H + h0;   // first (b, h) problem of the piece
        const char *qh = static_cast<const char *>(q) + first * pl.q_bytes / pl.heads;
        char *oh = static_cast<char *>(out) + first * pl.q_bytes / pl.heads;
        ok = cudaStreamWaitEvent(s_in, done_out[sl], 0) == cudaSuccess &&
             cudaMemcpyAsync(slot, qh, pl.q_bytes, cudaMemcpyHostToDevice, s_in) == cudaSuccess;
        if (ok && Lk > 0) {
            const size_t koff = first * pl.k_bytes / pl.heads;
            ok = cudaMemcpyAsync(slot + pl.off_k, static_cast<const char *>(k) + koff, pl.k_bytes,
                                 cudaMemcpyHostToDevice, s_in) == cudaSuccess &&
                 cudaMemcpyAsync(slot + pl.off_v, static_cast<const char *>(v) + koff, pl.k_bytes,
                                 cudaMemcpyHostToDevice, s_in) == cudaSuccess;
        }
        ok = ok && cudaEventRecord(done_in[sl], s_in) == cudaSuccess &&
             cudaStreamWaitEvent(stream, done_in[sl], 0) == cudaSuccess;
        if (!ok) {
            st = MHA_ERR_CUDA;
            break;
        }
        st = mha_fwd(slot, Lk > 0 ? slot + pl.off_k : nullptr, Lk > 0 ? slot + pl.off_v : nullptr,
                     mask_kind, dlens ? dlens + b : nullptr, slot + pl.off_out, 1, pl.heads, Lq, Lk,
                     D, scale, dtype, stream);
        if (st != MHA_OK) break;
        ok = cudaEventRecord(done_kernel[sl], stream) == cudaSuccess &&
             cudaStreamWaitEvent(s_out, done_kernel[sl], 0) == cudaSuccess &&
             cudaMemcpyAsync(oh, slot + pl.off_out, pl.q_bytes, cudaMemcpyDeviceToHost, s_out) ==
                 cudaSuccess &&
             cudaEventRecord(done_out[sl], s_out) == cudaSuccess;
        if (!ok) st = MHA_ERR_CUDA;
    }
    // Later work on `stream` follows every copy of the call (both copy
    // streams end before their last event: the out-stream's last copy
    // follows the last kernel, which followed the last in-copy).
    cudaEvent_t end = nullptr;
    if (s_in && s_out && cudaEventCreateWithFlags(&end, cudaEventDisableTiming) == cudaSuccess) {
        bool j = cudaEventRecord(end, s_out) == cudaSuccess &&
                 cudaStreamWaitEvent(stream, end, 0) == cudaSuccess &&
                 cudaEventRecord(end, s_in) == cudaSuccess &&
                 cudaStreamWaitEvent(stream, end, 0) == cudaSuccess;
        if (!j && st == MHA_OK) st = MHA_ERR_CUDA;
        cudaEventDestroy(end);
    } else if (st == MHA_OK) {
        st = MHA_ERR_CUDA;
    }
    // Released once the device has finished with them.
    for (int i = 0; i < 2; ++i) {
        if (done_in[i]) cudaEventDestroy(done_in[i]);
        if (done_kernel[i]) cudaEventDestroy(done_kernel[i]);
        if (done_out[i]) cudaEventDestroy(done_out[i]);
    }
    if (start) cudaEventDestroy(start);
    if (s_in) cudaStreamDestroy(s_in);
    if (s_out) cudaStreamDestroy(s_out);
    return st;
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

int mha_plan_prenorm(int B, int H, int Lq, int Lk, int D, int grid, int stats_given, int64_t *out) {
    if (out == nullptr || B <= 0 || H <= 0 || Lq <= 0 || Lk < 0 || grid <= 0 || (D != 64 && D != 128))
        return MHA_ERR_INVALID_ARG;
    if ((int64_t)H * D > 65536 || (int64_t)B * H * ((Lq + 255) / 256) > 0x7fffffffll) return MHA_ERR_TOO_LARGE;
    const mha::PrenormPlan pl = mha::plan_prenorm(B, H, Lq, Lk, D, grid, stats_given != 0);
    out[0] = pl.G;
    out[1] = pl.n_hg;
    out[2] = pl.cs;
    out[3] = pl.pre_chunks;
    out[4] = pl.grid;
    out[5] = pl.n_chunks;
    return MHA_OK;
}

void mha_set_f32_kernel(int which) { mha::set_f32_kernel_override(which); }

void mha_set_bf16_decode(int mode) { mha::set_decode_override(mode); }

void mha_set_bf16_decode_splits(int splits) { mha::set_decode_splits(splits); }

void mha_set_bwd_kernel(int which) { g_bwd_kernel = (which == 1) ? 1 : 0; }
void mha_set_pdl(int on) { mha::set_pdl(on); }

}  // extern "C"
