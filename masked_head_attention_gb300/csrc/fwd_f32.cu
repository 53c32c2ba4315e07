// fwd_f32.cu -- fused masked multi-head attention forward for fp32 inputs on
// CUDA-core FFMA (sm_103a).
//
// One CTA of 256 threads owns a 64-row query tile of one (b, h).  K and V
// tiles of 64 keys are staged in shared memory; each thread keeps a 4 x 4
// block of logits and a 4 x (D/16) block of the output in registers.  The
// softmax is the online form (running row max m, rescaled running sum l),
// with the row reductions done by warp shuffles inside the 16 lanes that
// share a row group, the mask computed from (row, col, length) in registers
// and key tiles beyond the causal limit or the valid length never loaded.
//
// Page sections this follows ("masked multi head attention" CUDA article,
// 2kiu.com): 2 (one fused kernel, skip masked work), 3.1 (mask computed in
// the kernel, -infinity before the softmax), 3.2 (row max by warp shuffles);
// "Why attention must compute the max first" (gsyq.cn): 2.3-2.4 (online
// softmax fused between QK^T and PV, scores never written to memory).
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kBM = 64;        // query rows per CTA
constexpr int kBN = 64;        // keys per tile
constexpr int kThreads = 256;  // 16 x 16 thread grid: ty owns 4 rows, tx 4 key columns

template <int D>
struct F32Cfg {
    static constexpr int LD = D + 4;     // padded row stride of the Q/K/V tiles (floats)
    static constexpr int LDP = kBN + 4;  // padded row stride of the P tile
    static constexpr int OC = D / 16;    // output columns per thread
    static constexpr size_t kSmem = sizeof(float) * (size_t)(kBM * LD + 2 * kBN * LD + kBM * LDP);
};

// Copy rows [row0, row0 + 64) of a [rows, D] fp32 matrix into a padded tile;
// rows at or beyond `nrows` become zero.
template <int D>
__device__ __forceinline__ void load_tile(float *dst, const float *__restrict__ src, int row0,
                                          int nrows, int tid) {
    constexpr int V4 = D / 4;
#pragma unroll
    for (int idx = tid; idx < kBN * V4; idx += kThreads) {
        const int r = idx / V4, c = idx % V4;
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row0 + r < nrows)
            val = __ldg(reinterpret_cast<const float4 *>(src + (size_t)(row0 + r) * D) + c);
        *reinterpret_cast<float4 *>(dst + r * F32Cfg<D>::LD + 4 * c) = val;
    }
}

// Natural-log log-sum-exp of a row from its base-2 running maximum m2 (of
// the logits times scale * log2(e)) and its sum l of 2^(x - m2):
// lse = ln(2) * (m2 + log2(l)); -infinity when the row saw no visible key.
__device__ __forceinline__ float row_lse(float m2, float l) {
    if (m2 == -INFINITY || !(l > 0.f)) return -INFINITY;
    return 0.69314718055994531f * (m2 + log2f(l));
}

template <int D>
__global__ void __launch_bounds__(kThreads)
    mha_fwd_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                       const float *__restrict__ v, const int32_t *__restrict__ kv_lengths,
                       float *__restrict__ out, float *__restrict__ lse, int H, int Lq, int Lk,
                       int mask_kind, float scale_log2) {
    using C = F32Cfg<D>;
    extern __shared__ float4 f32_smem[];
    float *sQ = reinterpret_cast<float *>(f32_smem);
    float *sK = sQ + kBM * C::LD;
    float *sV = sK + kBN * C::LD;
    float *sP = sV + kBN * C::LD;

    // Heaviest causal query tiles are launched first.
    const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    const int q0 = qt * kBM;
    const size_t bh = (size_t)b * H + h;
    const float *Qg = q + bh * (size_t)Lq * D;
    const float *Kg = k + bh * (size_t)Lk * D;
    const float *Vg = v + bh * (size_t)Lk * D;
    float *Og = out + bh * (size_t)Lq * D;

    const bool causal = (mask_kind & 1) != 0;
    int len = Lk;
    if (mask_kind & 2) len = max(0, min((int)kv_lengths[b], Lk));
    int kend = len;                                   // keys at or past kend are hidden for all rows
    if (causal) kend = min(kend, q0 + kBM);
    const int n_kt = (kend + kBN - 1) / kBN;

    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;

    load_tile<D>(sQ, Qg, q0, Lq, tid);

    float o[4][C::OC];
    float m[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < C::OC; ++c) o[i][c] = 0.f;
    }

    for (int t = 0; t < n_kt; ++t) {
        const int k0 = t * kBN;
        __syncthreads();  // the previous tile's P.V is done with sK, sV, sP
        load_tile<D>(sK, Kg, k0, Lk, tid);
        load_tile<D>(sV, Vg, k0, Lk, tid);
        __syncthreads();

        // S = Q K^T for rows 4*ty + i and keys tx + 16*j.
        float s[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 4
        for (int d = 0; d < D; d += 4) {
            float4 qa[4], kb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                qa[i] = *reinterpret_cast<const float4 *>(sQ + (ty * 4 + i) * C::LD + d);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                kb[j] = *reinterpret_cast<const float4 *>(sK + (tx + 16 * j) * C::LD + d);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[i][j] = fmaf(qa[i].x, kb[j].x, s[i][j]);
                    s[i][j] = fmaf(qa[i].y, kb[j].y, s[i][j]);
                    s[i][j] = fmaf(qa[i].z, kb[j].z, s[i][j]);
                    s[i][j] = fmaf(qa[i].w, kb[j].w, s[i][j]);
                }
        }

        // Scale into the base-2 domain and mask; only a tile that crosses the
        // visible end of some row needs the element test.
        const bool edge = (k0 + kBN > len) || (causal && k0 + kBN - 1 > q0);
        float mt[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = q0 + ty * 4 + i;
            const int vis_end = causal ? min(len, row + 1) : len;
            mt[i] = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float x = s[i][j] * scale_log2;
                if (edge && (k0 + tx + 16 * j >= vis_end)) x = -INFINITY;
                s[i][j] = x;
                mt[i] = fmaxf(mt[i], x);
            }
        }
#pragma unroll
        for (int off = 1; off < 16; off <<= 1)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                mt[i] = fmaxf(mt[i], __shfl_xor_sync(0xffffffffu, mt[i], off));

        // Online softmax update (base 2): m_new = max(m, tile max),
        // alpha = 2^(m - m_new), p = 2^(s - m_new), l = alpha * l + sum p.
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float m_new = fmaxf(m[i], mt[i]);
            const float msub = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2_approx(m[i] - msub);
            m[i] = m_new;
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float pj = ex2_approx(s[i][j] - msub);
                s[i][j] = pj;
                rs += pj;
            }
            l[i] = fmaf(l[i], alpha, rs);
#pragma unroll
            for (int c = 0; c < C::OC; ++c) o[i][c] *= alpha;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) sP[(ty * 4 + i) * C::LDP + tx + 16 * j] = s[i][j];
        __syncthreads();

        // O += P V for rows 4*ty + i and output columns 4*tx (+ 64).
#pragma unroll 2
        for (int j = 0; j < kBN; j += 4) {
            float4 pa[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                pa[i] = *reinterpret_cast<const float4 *>(sP + (ty * 4 + i) * C::LDP + j);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const float *vrow = sV + (j + jj) * C::LD + tx * 4;
                float4 vv[C::OC / 4];
#pragma unroll
                for (int hv = 0; hv < C::OC / 4; ++hv)
                    vv[hv] = *reinterpret_cast<const float4 *>(vrow + 64 * hv);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float pv = jj == 0 ? pa[i].x : jj == 1 ? pa[i].y : jj == 2 ? pa[i].z : pa[i].w;
#pragma unroll
                    for (int hv = 0; hv < C::OC / 4; ++hv) {
                        o[i][4 * hv + 0] = fmaf(pv, vv[hv].x, o[i][4 * hv + 0]);
                        o[i][4 * hv + 1] = fmaf(pv, vv[hv].y, o[i][4 * hv + 1]);
                        o[i][4 * hv + 2] = fmaf(pv, vv[hv].z, o[i][4 * hv + 2]);
                        o[i][4 * hv + 3] = fmaf(pv, vv[hv].w, o[i][4 * hv + 3]);
                    }
                }
            }
        }
    }

    // O / l; a row that saw no visible key (l == 0) is written as zeros.
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float lt = l[i];
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        const int row = q0 + ty * 4 + i;
        if (lse != nullptr && tx == 0 && row < Lq)
            lse[bh * (size_t)Lq + row] = row_lse(m[i], lt);
        if (row < Lq) {
            float *dst = Og + (size_t)row * D + tx * 4;
#pragma unroll
            for (int hv = 0; hv < C::OC / 4; ++hv)
                *reinterpret_cast<float4 *>(dst + 64 * hv) =
                    make_float4(o[i][4 * hv] * inv, o[i][4 * hv + 1] * inv,
                                o[i][4 * hv + 2] * inv, o[i][4 * hv + 3] * inv);
        }
    }
}

// ---------------------------------------------------------------------------
// Short key ranges (Lk * D <= 16384): a CTA of 4 warps owns 16 query rows of
// one (b, h) and stages every key row any of them can see, K and V, in shared
// memory once (cp.async; S starts as soon as K has landed, while V is still
// in flight).  There is no key-tile loop.  Warp w owns rows 4w..4w+3: for S
// each lane takes keys lane, lane + 32, ... (every key block advances through
// D together: 4 x blocks independent chains); for P.V each lane takes D/32
// output columns, with even and odd keys in separate accumulators.  P goes
// through shared memory as [key][4 rows], one broadcast 16-byte load per key.
// Many small CTAs, latest (heaviest under a causal mask) query blocks first,
// replace a few long serial ones when B * H * Lq is small.
// ---------------------------------------------------------------------------
// Short key ranges (Lk * D <= 16384, e.g. L = 128 at D = 64): a launch of
// many small CTAs with the shortest critical path.  CTA = 16 query rows of
// one (b, h): eight warps of two rows.  K and V stream through shared memory
// in chunks of 32 keys on a two-stage cp.async ring, so the first chunk's
// work starts after one load latency and later chunks land while earlier
// ones are used; chunks past the keys any of the CTA's rows can see are never
// loaded.  Per chunk a lane takes one key for S (the query rows broadcast from
// shared memory, its K row read with 16-byte loads from rows padded to D + 4
// floats: conflict-free), the warp runs the online softmax of each row by
// shuffles (running max, rescaled running sum, base-2 exponent), and for P.V
// the lane takes D/32 output columns with each key's weight broadcast by a
// shuffle.  The latest (for a causal mask the heaviest) query blocks launch
// first.
// ---------------------------------------------------------------------------
constexpr int kSmallRows = 16;                        // query rows per CTA
constexpr int kSmallWarps = 8;
constexpr int kSmallR = kSmallRows / kSmallWarps;     // query rows per warp
constexpr int kSmallThreads = 32 * kSmallWarps;
constexpr int kSmallChunk = 32;                       // keys per chunk (one per lane)
constexpr int kSmallMaxKD = 16384;                    // Lk * D limit of this kernel
// Automatic choice for D = 64: this kernel below this many (row, key) pairs
// (B * H * Lq * Lk), the tensor-core kernel above.
constexpr int64_t kSmallAutoWork = 1ll << 22;

template <int D>
struct SmallCfg {
    static constexpr int LDK = D + 4;                        // padded K row (floats)
    static constexpr int kKChunk = kSmallChunk * LDK;        // floats per K stage
    static constexpr int kVChunk = kSmallChunk * D;          // floats per V stage
    static constexpr size_t kSmem = sizeof(float) * ((size_t)kSmallRows * D + 2 * (kKChunk + kVChunk));
};

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kSmallThreads)
    mha_fwd_f32_small_kernel(const float *__restrict__ q, const float *__restrict__ k,
                             const float *__restrict__ v, const int32_t *__restrict__ kv_lengths,
                             float *__restrict__ out, float *__restrict__ lse, int H, int Lq,
                             int Lk, int mask_kind, float scale_log2) {
    using C = SmallCfg<D>;
    constexpr int DC = D / 32;   // output columns per lane
    constexpr int R = kSmallR;
    constexpr int V4 = D / 4;
    extern __shared__ float4 small_smem[];
    float *sQ = reinterpret_cast<float *>(small_smem);   // [16][D]
    float *sK = sQ + kSmallRows * D;                      // [2][32][LDK]
    float *sV = sK + 2 * C::kKChunk;                      // [2][32][D]

    const int h = blockIdx.y, b = blockIdx.z;
    const int q0 = ((int)gridDim.x - 1 - (int)blockIdx.x) * kSmallRows;
    const size_t bh = (size_t)b * H + h;
    const float *Qg = q + bh * (size_t)Lq * D;
    const float *Kg = k + bh * (size_t)Lk * D;
    const float *Vg = v + bh * (size_t)Lk * D;
    float *Og = out + bh * (size_t)Lq * D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const bool causal = (mask_kind & 1) != 0;
    int len = Lk;
    if (mask_kind & 2) len = max(0, min((int)kv_lengths[b], Lk));
    int kend = len;                                   // keys any row of the CTA can see
    if (causal) kend = min(kend, q0 + kSmallRows);
    kend = max(kend, 0);
    const int nch = (kend + kSmallChunk - 1) / kSmallChunk;

    // Chunk c into stage c & 1; keys at or past kend are zero (finite, and
    // their weights are exactly 0).
    auto load_chunk = [&](int c) {
        float *dK = sK + (c & 1) * C::kKChunk;
        float *dV = sV + (c & 1) * C::kVChunk;
        for (int idx = tid; idx < kSmallChunk * V4; idx += kSmallThreads) {
            const int r = idx / V4, cc = idx % V4;
            const int key = c * kSmallChunk + r;
            if (key < kend) {
                cp_async16(dK + r * C::LDK + 4 * cc, Kg + (size_t)key * D + 4 * cc);
                cp_async16(dV + r * D + 4 * cc, Vg + (size_t)key * D + 4 * cc);
            } else {
                *reinterpret_cast<float4 *>(dK + r * C::LDK + 4 * cc) = make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4 *>(dV + r * D + 4 * cc) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        cp_async_commit();
    };
    for (int idx = tid; idx < kSmallRows * V4; idx += kSmallThreads) {
        const int r = idx / V4, cc = idx % V4;
        if (q0 + r < Lq)
            cp_async16(sQ + r * D + 4 * cc, Qg + (size_t)(q0 + r) * D + 4 * cc);
        else
            *reinterpret_cast<float4 *>(sQ + r * D + 4 * cc) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (nch > 0) load_chunk(0);   // the Q copies join the first group
    else cp_async_commit();
    if (nch > 1) load_chunk(1);

    const float *Qw = sQ + R * warp * D;
    int vis_end[R];
    float m[R], l[R], o[R][DC];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int row = q0 + R * warp + r;
        vis_end[r] = causal ? min(len, row + 1) : len;
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int cc = 0; cc < DC; ++cc) o[r][cc] = 0.f;
    }
    for (int c = 0; c < nch; ++c) {
        if (c + 1 < nch)
            cp_async_wait_group<1>();
        else
            cp_async_wait_group<0>();
        __syncthreads();
        // S for the warp's rows and key c * 32 + lane.
        const float *Kl = sK + (c & 1) * C::kKChunk + lane * C::LDK;
        float sc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) sc[r] = 0.f;
#pragma unroll 8
        for (int d = 0; d < D; d += 4) {
            const float4 kk = *reinterpret_cast<const float4 *>(Kl + d);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float4 qq = *reinterpret_cast<const float4 *>(Qw + r * D + d);
                sc[r] = fmaf(qq.x, kk.x, sc[r]);
                sc[r] = fmaf(qq.y, kk.y, sc[r]);
                sc[r] = fmaf(qq.z, kk.z, sc[r]);
                sc[r] = fmaf(qq.w, kk.w, sc[r]);
            }
        }
        // Mask, base-2 logits, online softmax per row (warp shuffles).
        const int key = c * kSmallChunk + lane;
        float p[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float x = key < vis_end[r] ? sc[r] * scale_log2 : -INFINITY;
            float cm = x;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
            const float m_new = fmaxf(m[r], cm);
            const float msub = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2_approx(m[r] - msub);
            p[r] = ex2_approx(x - msub);
            float ps = p[r];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
            l[r] = fmaf(l[r], alpha, ps);
            m[r] = m_new;
#pragma unroll
            for (int cc = 0; cc < DC; ++cc) o[r][cc] *= alpha;
        }
        // O += P V: the lane's D/32 columns, each key's weight by shuffle.
        const float *Vl = sV + (c & 1) * C::kVChunk + lane * DC;
#pragma unroll 8
        for (int j = 0; j < kSmallChunk; ++j) {
            float vv[DC];
            if (DC == 2) {
                const float2 t = *reinterpret_cast<const float2 *>(Vl + j * D);
                vv[0] = t.x;
                vv[DC - 1] = t.y;
            } else {
                const float4 t = *reinterpret_cast<const float4 *>(Vl + j * D);
                vv[0] = t.x;
                vv[1] = t.y;
                vv[DC - 2] = t.z;
                vv[DC - 1] = t.w;
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float pj = __shfl_sync(0xffffffffu, p[r], j);
#pragma unroll
                for (int cc = 0; cc < DC; ++cc) o[r][cc] = fmaf(pj, vv[cc], o[r][cc]);
            }
        }
        __syncthreads();   // every warp is done with stage c & 1
        if (c + 2 < nch) load_chunk(c + 2);
    }
    if (nch == 0) cp_async_wait_group<0>();
    // O / l; a row that saw no visible key (l == 0) is written as zeros.
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int row = q0 + R * warp + r;
        const bool live = row < Lq;
        const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
        report_flag(live && !finite_f(l[r]), kFlagSum);
        float res[DC];
        float rsum = 0.f;
#pragma unroll
        for (int cc = 0; cc < DC; ++cc) {
            res[cc] = o[r][cc] * inv;
            rsum += res[cc];
        }
        report_flag(live && !finite_f(rsum), kFlagNonFinite);
        if (!live) continue;
        float *dst = Og + (size_t)row * D + lane * DC;
        if (DC == 2)
            *reinterpret_cast<float2 *>(dst) = make_float2(res[0], res[DC - 1]);
        else
            *reinterpret_cast<float4 *>(dst) = make_float4(res[0], res[1], res[DC - 2], res[DC - 1]);
        if (lse != nullptr && lane == 0) lse[bh * (size_t)Lq + row] = row_lse(m[r], l[r]);
    }
}

template <int D>
cudaError_t launch_small(const float *q, const float *k, const float *v, const int32_t *kv,
                         float *out, float *lse, int B, int H, int Lq, int Lk, int mask_kind, float scale,
                         cudaStream_t stream) {
    constexpr size_t smem = SmallCfg<D>::kSmem;
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(mha_fwd_f32_small_kernel<D>), smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((Lq + kSmallRows - 1) / kSmallRows, H, B);
    mha_fwd_f32_small_kernel<D><<<grid, kSmallThreads, smem, stream>>>(
        q, k, v, kv, out, lse, H, Lq, Lk, mask_kind, scale * 1.4426950408889634f);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch(const float *q, const float *k, const float *v, const int32_t *kv,
                   float *out, float *lse, int B, int H, int Lq, int Lk, int mask_kind, float scale,
                   cudaStream_t stream) {
    constexpr size_t smem = F32Cfg<D>::kSmem;
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(mha_fwd_f32_kernel<D>), smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((Lq + kBM - 1) / kBM, H, B);
    const float scale_log2 = scale * 1.4426950408889634f;
    mha_fwd_f32_kernel<D><<<grid, kThreads, smem, stream>>>(q, k, v, kv, out, lse, H, Lq, Lk,
                                                            mask_kind, scale_log2);
    return cudaGetLastError();
}

// 0 automatic, 1 tiled only, 2 short-key kernel where it applies, 3 the
// tensor-core (3xTF32) kernel where it applies (D = 64).
thread_local int g_f32_kernel = 0;

}  // namespace

void set_f32_kernel_override(int which) { g_f32_kernel = which; }

cudaError_t launch_fwd_f32(const float *q, const float *k, const float *v,
                           const int32_t *kv_lengths, float *out, float *lse, int B, int H,
                           int Lq, int Lk, int D, int mask_kind, float scale,
                           cudaStream_t stream, int *driver_err) {
    *driver_err = 0;
    const int which = (g_f32_kernel >= 1 && g_f32_kernel <= 3) ? g_f32_kernel : 0;
    // Small problems with short key ranges are latency-bound: the CUDA-core
    // short-key kernel's many small CTAs finish sooner than the tensor-core
    // kernel's 128-row items.
    const bool short_keys = (int64_t)Lk * D <= kSmallMaxKD;
    const bool small_problem = short_keys && (int64_t)B * H * Lq * Lk <= kSmallAutoWork;
    if ((which == 3 || (which == 0 && !small_problem)) && tf32x3_applies(D))
        return launch_fwd_tf32x3(q, k, v, kv_lengths, out, lse, B, H, Lq, Lk, D, mask_kind, scale,
                                 stream, driver_err);
    if (short_keys && which != 1) {
        if (D == 64)
            return launch_small<64>(q, k, v, kv_lengths, out, lse, B, H, Lq, Lk, mask_kind, scale,
                                    stream);
        return launch_small<128>(q, k, v, kv_lengths, out, lse, B, H, Lq, Lk, mask_kind, scale,
                                 stream);
    }
    if (D == 64)
        return launch<64>(q, k, v, kv_lengths, out, lse, B, H, Lq, Lk, mask_kind, scale, stream);
    return launch<128>(q, k, v, kv_lengths, out, lse, B, H, Lq, Lk, mask_kind, scale, stream);
}

}  // namespace mha
