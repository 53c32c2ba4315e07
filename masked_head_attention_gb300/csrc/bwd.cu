// bwd.cu -- backward pass of fused masked multi-head attention on CUDA-core
// FFMA (sm_103a): dq, dk, dv from q, k, v, the forward's output o, its row
// log-sum-exp lse and the output gradient dout.  fp32 or bf16 inputs; the
// arithmetic is fp32 either way, and the gradients come out in the input type
// (for bf16, dq is accumulated in an fp32 workspace and converted at the end).
//
// The softmax weights are never stored by the forward; here they are formed
// again from the saved row statistic, p_ij = exp(s_ij - lse_i), and the
// softmax Jacobian d p_ij / d s_ik = p_ij (delta_jk - p_ik) ("Why attention
// must compute the max first", gsyq.cn, section 3.3) is applied as
//     dS_ij = p_ij (dP_ij - Delta_i),  dP_ij = dout_i . v_j,
// where Delta_i = sum_j p_ij dP_ij = dout_i . o_i (the two are equal because
// o_i = sum_j p_ij v_j), so it costs one dot product per row instead of a
// pass over the keys.
//
// Kernels:
//  1. bwd_row_delta: Delta_i = dout_i . o_i for every row, and the fp32 dq
//     accumulator zeroed (dq is accumulated by the second kernel).  HBM-bound,
//     one pass.
//  2. mha_bwd_f32_kernel: one CTA of 256 threads owns a 64-key tile of one
//     (b, h) with K and V resident in shared memory, and walks the query
//     tiles of 64 rows that can see any of its keys (under the causal rule:
//     rows >= the tile's first key).  Per query tile it stages Q, dout, lse
//     and Delta, forms S = Q K^T and dP = dout V^T together (each thread a
//     4 x 4 block), P and dS, then accumulates dV += P^T dout and
//     dK += dS^T Q in registers (each thread 4 keys x D/16 columns) and adds
//     its share of dQ = dS K into global memory with 16-byte fp32 atomic
//     adds.  dK (times scale) and dV are written once at the end; keys no
//     row can see get zeros.
//  3. (bf16) bwd_dq_convert: the fp32 dq accumulator to bf16.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kBwdBM = 64;        // query rows per tile
constexpr int kBwdBN = 64;        // keys per CTA
constexpr int kBwdThreads = 256;  // 16 x 16: ty owns 4 rows (or keys), tx 4 columns

template <int D>
struct BwdCfg {
    static constexpr int LD = D + 4;        // padded row stride of Q/K/V/dout tiles (floats)
    static constexpr int LDP = kBwdBN + 4;  // padded row stride of the P and dS tiles
    static constexpr int OC = D / 16;       // accumulator columns per thread
    static constexpr size_t kSmem =
        sizeof(float) * ((size_t)4 * 64 * LD + (size_t)2 * kBwdBM * LDP + 2 * kBwdBM);
};

// Four consecutive elements as fp32 (bf16: an 8-byte load, widened).
__device__ __forceinline__ float4 load4(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}
// Four consecutive elements from fp32 (bf16: rounded to nearest even).
__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 v) {
    uint2 u;
    u.x = pack_bf16x2(v.x, v.y);
    u.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2 *>(p) = u;
}

// Rows [row0, row0 + 64) of a [rows, D] matrix into a padded fp32 tile;
// rows at or beyond `nrows` become zero.
template <int D, typename T>
__device__ __forceinline__ void bwd_load_tile(float *dst, const T *__restrict__ src, int row0,
                                              int nrows, int tid) {
    constexpr int V4 = D / 4;
#pragma unroll
    for (int idx = tid; idx < 64 * V4; idx += kBwdThreads) {
        const int r = idx / V4, c = idx % V4;
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row0 + r < nrows) val = load4(src + (size_t)(row0 + r) * D + 4 * c);
        *reinterpret_cast<float4 *>(dst + r * BwdCfg<D>::LD + 4 * c) = val;
    }
}

// Delta_i = dout_i . o_i; dq_i = 0 (the fp32 accumulator; skipped when dq is
// null).  A half-warp (16 lanes) per row.
template <int D, typename T>
__global__ void __launch_bounds__(256)
    bwd_row_delta_kernel(const T *__restrict__ o, const T *__restrict__ dout,
                         float *__restrict__ delta, float *__restrict__ dq, int64_t rows) {
    pdl_wait();      // the stream's previous kernel has completed; its writes are visible
    pdl_trigger();   // the next kernel may be scheduled
    constexpr int PER = D / 64;   // groups of 4 elements per lane
    const int64_t row = (int64_t)blockIdx.x * 16 + (threadIdx.x >> 4);
    const int lane = threadIdx.x & 15;
    float acc = 0.f;
    if (row < rows) {
        const T *po = o + row * D;
        const T *pg = dout + row * D;
        float4 *pq = dq != nullptr ? reinterpret_cast<float4 *>(dq + row * D) : nullptr;
#pragma unroll
        for (int t = 0; t < PER; ++t) {
            const float4 a = load4(po + 4 * (lane + 16 * t)), g = load4(pg + 4 * (lane + 16 * t));
            acc = fmaf(a.x, g.x, acc);
            acc = fmaf(a.y, g.y, acc);
            acc = fmaf(a.z, g.z, acc);
            acc = fmaf(a.w, g.w, acc);
            if (dq != nullptr) pq[lane + 16 * t] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && lane == 0) delta[row] = acc;
}

template <int D, typename T>
__global__ void __launch_bounds__(kBwdThreads, D == 64 ? 2 : 1)
    mha_bwd_f32_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                       const T *__restrict__ dout, const float *__restrict__ lse,
                       const float *__restrict__ delta, const int32_t *__restrict__ kv_lengths,
                       float *__restrict__ dq, T *__restrict__ dk, T *__restrict__ dv, int H,
                       int Lq, int Lk, int mask_kind, float scale, float scale_log2) {
    pdl_wait();      // the stream's previous kernel has completed; its writes are visible
    pdl_trigger();   // the next kernel may be scheduled
    using C = BwdCfg<D>;
    constexpr int OC = C::OC;
    extern __shared__ float4 bwd_smem[];
    float *sK = reinterpret_cast<float *>(bwd_smem);
    float *sV = sK + 64 * C::LD;
    float *sQ = sV + 64 * C::LD;
    float *sG = sQ + 64 * C::LD;          // dout tile
    float *sP = sG + 64 * C::LD;          // P  [query][key]
    float *sS = sP + kBwdBM * C::LDP;     // dS [query][key]
    float *sL = sS + kBwdBM * C::LDP;     // lse * log2(e) per query row
    float *sDl = sL + kBwdBM;             // Delta per query row

    // Key tile 0 (the heaviest under a causal mask) is launched first.
    const int k0 = blockIdx.x * kBwdBN;
    const int h = blockIdx.y, b = blockIdx.z;
    const size_t bh = (size_t)b * H + h;
    const T *Qg = q + bh * (size_t)Lq * D;
    const T *Kg = k + bh * (size_t)Lk * D;
    const T *Vg = v + bh * (size_t)Lk * D;
    const T *Gg = dout + bh * (size_t)Lq * D;
    const float *Lg = lse + bh * (size_t)Lq;
    const float *Dg = delta + bh * (size_t)Lq;
    float *dQg = dq + bh * (size_t)Lq * D;

    const bool causal = (mask_kind & 1) != 0;
    int len = Lk;
    if (mask_kind & 2) len = max(0, min((int)kv_lengths[b], Lk));
    // Query tiles that can see a key of this tile: none if the tile starts at
    // or past the valid length; under the causal rule rows >= k0 only.
    const int n_qt = (Lq + kBwdBM - 1) / kBwdBM;
    const int qt0 = causal ? k0 / kBwdBM : 0;
    const int qt1 = (k0 < len) ? n_qt : qt0;

    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;

    // dV and dK accumulators as column pairs for the packed fp32x2 FMA (two
    // FMAs per instruction: the same FMA-pipe rate in half the issue slots).
    float2 accv[4][OC / 2], acck[4][OC / 2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < OC / 2; ++c) {
            accv[i][c] = make_float2(0.f, 0.f);
            acck[i][c] = make_float2(0.f, 0.f);
        }

    if (qt0 < qt1) {
        bwd_load_tile<D, T>(sK, Kg, k0, Lk, tid);
        bwd_load_tile<D, T>(sV, Vg, k0, Lk, tid);
    }

    for (int qt = qt0; qt < qt1; ++qt) {
        const int q0 = qt * kBwdBM;
        __syncthreads();   // the previous tile is done with sQ, sG, sP, sS, sL, sDl
        bwd_load_tile<D, T>(sQ, Qg, q0, Lq, tid);
        bwd_load_tile<D, T>(sG, Gg, q0, Lq, tid);
        if (tid < kBwdBM) {
            const int row = q0 + tid;
            sL[tid] = row < Lq ? Lg[row] * 1.4426950408889634f : 0.f;
            sDl[tid] = row < Lq ? Dg[row] : 0.f;
        }
        __syncthreads();

        // S = Q K^T and dP = dout V^T for rows ty*4 + i, keys tx + 16 j.
        float s[4][4], dp[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                s[i][j] = 0.f;
                dp[i][j] = 0.f;
            }
#pragma unroll 2
        for (int d = 0; d < D; d += 4) {
            float4 qa[4], ga[4], kb[4], vb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                qa[i] = *reinterpret_cast<const float4 *>(sQ + (ty * 4 + i) * C::LD + d);
                ga[i] = *reinterpret_cast<const float4 *>(sG + (ty * 4 + i) * C::LD + d);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                kb[j] = *reinterpret_cast<const float4 *>(sK + (tx + 16 * j) * C::LD + d);
                vb[j] = *reinterpret_cast<const float4 *>(sV + (tx + 16 * j) * C::LD + d);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[i][j] = fmaf(qa[i].x, kb[j].x, s[i][j]);
                    s[i][j] = fmaf(qa[i].y, kb[j].y, s[i][j]);
                    s[i][j] = fmaf(qa[i].z, kb[j].z, s[i][j]);
                    s[i][j] = fmaf(qa[i].w, kb[j].w, s[i][j]);
                    dp[i][j] = fmaf(ga[i].x, vb[j].x, dp[i][j]);
                    dp[i][j] = fmaf(ga[i].y, vb[j].y, dp[i][j]);
                    dp[i][j] = fmaf(ga[i].z, vb[j].z, dp[i][j]);
                    dp[i][j] = fmaf(ga[i].w, vb[j].w, dp[i][j]);
                }
        }

        // P = 2^(s * scale * log2(e) - lse * log2(e)) at visible positions, else
        // exactly 0; dS = P (dP - Delta).  Only a tile crossing the visible end
        // of a row (or the end of Lq) needs the element test.
        const bool edge = (k0 + kBwdBN > len) || (causal && k0 + kBwdBN - 1 > q0) ||
                          (q0 + kBwdBM > Lq);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rl = ty * 4 + i, row = q0 + rl;
            const int vis_end = causal ? min(len, row + 1) : len;
            const float l2 = sL[rl], dl = sDl[rl];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int key = k0 + tx + 16 * j;
                float p = ex2_approx(fmaf(s[i][j], scale_log2, -l2));
                if (edge && (key >= vis_end || row >= Lq)) p = 0.f;
                sP[rl * C::LDP + tx + 16 * j] = p;
                sS[rl * C::LDP + tx + 16 * j] = p * (dp[i][j] - dl);
            }
        }
        __syncthreads();

        // dV += P^T dout and dK += dS^T Q for keys ty*4 + i, columns tx*4 (+ 64).
#pragma unroll 4
        for (int r = 0; r < kBwdBM; ++r) {
            const float4 pa = *reinterpret_cast<const float4 *>(sP + r * C::LDP + ty * 4);
            const float4 sa = *reinterpret_cast<const float4 *>(sS + r * C::LDP + ty * 4);
            const float pr[4] = {pa.x, pa.y, pa.z, pa.w};
            const float sr[4] = {sa.x, sa.y, sa.z, sa.w};
#pragma unroll
            for (int hv = 0; hv < OC / 4; ++hv) {
                const float4 g = *reinterpret_cast<const float4 *>(sG + r * C::LD + tx * 4 + 64 * hv);
                const float4 qq = *reinterpret_cast<const float4 *>(sQ + r * C::LD + tx * 4 + 64 * hv);
                const float2 g01 = make_float2(g.x, g.y), g23 = make_float2(g.z, g.w);
                const float2 q01 = make_float2(qq.x, qq.y), q23 = make_float2(qq.z, qq.w);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 pp = make_float2(pr[i], pr[i]), ss = make_float2(sr[i], sr[i]);
                    accv[i][2 * hv + 0] = __ffma2_rn(pp, g01, accv[i][2 * hv + 0]);
                    accv[i][2 * hv + 1] = __ffma2_rn(pp, g23, accv[i][2 * hv + 1]);
                    acck[i][2 * hv + 0] = __ffma2_rn(ss, q01, acck[i][2 * hv + 0]);
                    acck[i][2 * hv + 1] = __ffma2_rn(ss, q23, acck[i][2 * hv + 1]);
                }
            }
        }

        // dQ (rows ty*4 + i, columns tx*4 (+ 64)) += scale * dS K, added to the
        // global accumulator with one 16-byte atomic per 4 columns.
        float2 accq[4][OC / 2];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int c = 0; c < OC / 2; ++c) accq[i][c] = make_float2(0.f, 0.f);
#pragma unroll 2
        for (int j = 0; j < kBwdBN; j += 4) {
            float4 sa[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                sa[i] = *reinterpret_cast<const float4 *>(sS + (ty * 4 + i) * C::LDP + j);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const float *krow = sK + (j + jj) * C::LD + tx * 4;
#pragma unroll
                for (int hv = 0; hv < OC / 4; ++hv) {
                    const float4 kk = *reinterpret_cast<const float4 *>(krow + 64 * hv);
                    const float2 k01 = make_float2(kk.x, kk.y), k23 = make_float2(kk.z, kk.w);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float w = jj == 0 ? sa[i].x : jj == 1 ? sa[i].y : jj == 2 ? sa[i].z : sa[i].w;
                        const float2 ww = make_float2(w, w);
                        accq[i][2 * hv + 0] = __ffma2_rn(ww, k01, accq[i][2 * hv + 0]);
                        accq[i][2 * hv + 1] = __ffma2_rn(ww, k23, accq[i][2 * hv + 1]);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = q0 + ty * 4 + i;
            if (row >= Lq) continue;
#pragma unroll
            for (int hv = 0; hv < OC / 4; ++hv)
                atomicAdd(reinterpret_cast<float4 *>(dQg + (size_t)row * D + tx * 4 + 64 * hv),
                          make_float4(accq[i][2 * hv].x * scale, accq[i][2 * hv].y * scale,
                                      accq[i][2 * hv + 1].x * scale, accq[i][2 * hv + 1].y * scale));
        }
    }

    // dK = scale * dS^T Q, dV = P^T dout for the tile's keys (zeros where no
    // row could see the key).
    T *dKg = dk + bh * (size_t)Lk * D;
    T *dVg = dv + bh * (size_t)Lk * D;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int key = k0 + ty * 4 + i;
        if (key >= Lk) continue;
#pragma unroll
        for (int hv = 0; hv < OC / 4; ++hv) {
            const size_t off = (size_t)key * D + tx * 4 + 64 * hv;
            store4(dVg + off, make_float4(accv[i][2 * hv].x, accv[i][2 * hv].y,
                                          accv[i][2 * hv + 1].x, accv[i][2 * hv + 1].y));
            store4(dKg + off, make_float4(acck[i][2 * hv].x * scale, acck[i][2 * hv].y * scale,
                                          acck[i][2 * hv + 1].x * scale, acck[i][2 * hv + 1].y * scale));
        }
    }
}

// dq (bf16) from the fp32 accumulator, 8 elements per thread.
__global__ void __launch_bounds__(256)
    bwd_dq_convert_kernel(const float *__restrict__ acc, __nv_bfloat16 *__restrict__ dq, int64_t n8) {
    pdl_wait();      // the stream's previous kernel has completed; its writes are visible
    pdl_trigger();   // the next kernel may be scheduled
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= n8) return;
    const float4 a = __ldg(reinterpret_cast<const float4 *>(acc) + 2 * i);
    const float4 b = __ldg(reinterpret_cast<const float4 *>(acc) + 2 * i + 1);
    uint4 u;
    u.x = pack_bf16x2(a.x, a.y);
    u.y = pack_bf16x2(a.z, a.w);
    u.z = pack_bf16x2(b.x, b.y);
    u.w = pack_bf16x2(b.z, b.w);
    reinterpret_cast<uint4 *>(dq)[i] = u;
}

template <int D, typename T>
cudaError_t launch_bwd(const T *q, const T *k, const T *v, const T *o, const T *dout,
                       const float *lse, const int32_t *kv, float *dq_acc, T *dk, T *dv,
                       float *delta, int B, int H, int Lq, int Lk, int mask_kind, float scale,
                       cudaStream_t stream) {
    const int64_t rows = (int64_t)B * H * Lq;
    cudaError_t e = cudaSuccess;
    if (rows > 0) {
        e = launch_kernel(bwd_row_delta_kernel<D, T>, dim3((unsigned)((rows + 15) / 16)), dim3(256),
                          0, stream, nullptr, o, dout, delta, dq_acc, rows);
    }
    if (e != cudaSuccess || Lk == 0) return e;
    constexpr size_t smem = BwdCfg<D>::kSmem;
    e = set_smem_limit(reinterpret_cast<const void *>(mha_bwd_f32_kernel<D, T>), smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((Lk + kBwdBN - 1) / kBwdBN, H, B);
    return launch_kernel(mha_bwd_f32_kernel<D, T>, grid, dim3(kBwdThreads), smem, stream, nullptr,
                         q, k, v, dout, lse, delta, kv, dq_acc, dk, dv, H, Lq, Lk, mask_kind, scale,
                         scale * 1.4426950408889634f);
}

}  // namespace

cudaError_t launch_bwd_f32(const float *q, const float *k, const float *v, const float *o,
                           const float *dout, const float *lse, const int32_t *kv_lengths,
                           float *dq, float *dk, float *dv, float *delta, int B, int H, int Lq,
                           int Lk, int D, int mask_kind, float scale, cudaStream_t stream) {
    if (D == 64)
        return launch_bwd<64, float>(q, k, v, o, dout, lse, kv_lengths, dq, dk, dv, delta, B, H,
                                     Lq, Lk, mask_kind, scale, stream);
    return launch_bwd<128, float>(q, k, v, o, dout, lse, kv_lengths, dq, dk, dv, delta, B, H, Lq,
                                  Lk, mask_kind, scale, stream);
}

cudaError_t launch_bwd_row_delta_bf16(const void *o, const void *dout, float *delta, int64_t rows,
                                      int D, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    using bf = __nv_bfloat16;
    const unsigned grid = (unsigned)((rows + 15) / 16);
    float *no_dq = nullptr;
    if (D == 64)
        return launch_kernel(bwd_row_delta_kernel<64, bf>, dim3(grid), dim3(256), 0, stream, nullptr,
                             static_cast<const bf *>(o), static_cast<const bf *>(dout), delta, no_dq,
                             rows);
    return launch_kernel(bwd_row_delta_kernel<128, bf>, dim3(grid), dim3(256), 0, stream, nullptr,
                         static_cast<const bf *>(o), static_cast<const bf *>(dout), delta, no_dq,
                         rows);
}

cudaError_t launch_bwd_bf16(const void *q, const void *k, const void *v, const void *o,
                            const void *dout, const float *lse, const int32_t *kv_lengths,
                            void *dq, void *dk, void *dv, float *dq_acc, float *delta, int B,
                            int H, int Lq, int Lk, int D, int mask_kind, float scale,
                            cudaStream_t stream) {
    using bf = __nv_bfloat16;
    const bf *Q = static_cast<const bf *>(q), *K = static_cast<const bf *>(k);
    const bf *V = static_cast<const bf *>(v), *O = static_cast<const bf *>(o);
    const bf *G = static_cast<const bf *>(dout);
    bf *dK = static_cast<bf *>(dk), *dV = static_cast<bf *>(dv);
    cudaError_t e =
        D == 64 ? launch_bwd<64, bf>(Q, K, V, O, G, lse, kv_lengths, dq_acc, dK, dV, delta, B, H,
                                     Lq, Lk, mask_kind, scale, stream)
                : launch_bwd<128, bf>(Q, K, V, O, G, lse, kv_lengths, dq_acc, dK, dV, delta, B, H,
                                      Lq, Lk, mask_kind, scale, stream);
    if (e != cudaSuccess) return e;
    const int64_t n8 = (int64_t)B * H * Lq * D / 8;
    if (n8 == 0) return cudaSuccess;
    return launch_kernel(bwd_dq_convert_kernel, dim3((unsigned)((n8 + 255) / 256)), dim3(256), 0,
                         stream, nullptr, static_cast<const float *>(dq_acc), static_cast<bf *>(dq),
                         n8);
}

}  // namespace mha
