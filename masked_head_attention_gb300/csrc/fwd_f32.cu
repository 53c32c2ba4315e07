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
    pdl_wait();      // the stream's previous kernel has completed; its writes are visible
    pdl_trigger();   // the next kernel may be scheduled
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
constexpr int kSmallRows = 16;
constexpr int kSmallR = 4;                               // query rows per warp (2 or 4)
constexpr int kSmallWarps = kSmallRows / kSmallR;
constexpr int kSmallThreads = 32 * kSmallWarps;
constexpr int kSmallMaxKD = 16384;   // Lk * D limit (K and V: 2 x 64 KB + padding)

template <int D>
struct SmallCfg {
    static constexpr int LDK = D + 4;                 // padded K row (conflict-free 16-byte loads)
    static constexpr int kMaxKeys = kSmallMaxKD / D;  // 256 (D = 64) or 128 (D = 128)
    static constexpr int KB = kMaxKeys / 32;          // key blocks of 32 per lane
    static size_t smem(int keys) {
        return sizeof(float) * ((size_t)keys * LDK + (size_t)keys * D + kSmallRows * D +
                                (size_t)kSmallWarps * keys * kSmallR);
    }
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

// Q.K for the warp's R query rows against keys kb*32 + lane, kb < NKB.
template <int D, int NKB, int KB>
__device__ __forceinline__ void small_scores(const float *sK, const float *Qw, int lane,
                                             float (&s)[kSmallR][KB]) {
    constexpr int LDK = SmallCfg<D>::LDK;
#pragma unroll 2
    for (int d = 0; d < D; d += 4) {
        float4 qq[kSmallR];
#pragma unroll
        for (int r = 0; r < kSmallR; ++r) qq[r] = *reinterpret_cast<const float4 *>(Qw + r * D + d);
#pragma unroll
        for (int kb = 0; kb < NKB; ++kb) {
            const float4 kk = *reinterpret_cast<const float4 *>(sK + (kb * 32 + lane) * LDK + d);
#pragma unroll
            for (int r = 0; r < kSmallR; ++r) {
                s[r][kb] = fmaf(qq[r].x, kk.x, s[r][kb]);
                s[r][kb] = fmaf(qq[r].y, kk.y, s[r][kb]);
                s[r][kb] = fmaf(qq[r].z, kk.z, s[r][kb]);
                s[r][kb] = fmaf(qq[r].w, kk.w, s[r][kb]);
            }
        }
    }
}

// acc[r][c] += P[key][r] * V[key][lane*DC + c] for the warp's rows.
template <int D>
__device__ __forceinline__ void small_pv_key(const float *Pw, const float *Vl, int key,
                                             float (&acc)[kSmallR][D / 32]) {
    constexpr int DC = D / 32;
    static_assert(kSmallR == 2 || kSmallR == 4, "P is read as one float2 / float4 per key");
    float pp[kSmallR];
    if (kSmallR == 4) {
        const float4 t = *reinterpret_cast<const float4 *>(Pw + key * kSmallR);
        pp[0] = t.x;
        pp[1] = t.y;
        pp[kSmallR - 2] = t.z;
        pp[kSmallR - 1] = t.w;
    } else {
        const float2 t = *reinterpret_cast<const float2 *>(Pw + key * kSmallR);
        pp[0] = t.x;
        pp[1] = t.y;
    }
    float vv[DC];
    if (DC == 2) {
        const float2 t = *reinterpret_cast<const float2 *>(Vl + (size_t)key * D);
        vv[0] = t.x;
        vv[1] = t.y;
    } else {
        const float4 t = *reinterpret_cast<const float4 *>(Vl + (size_t)key * D);
        vv[0] = t.x;
        vv[1] = t.y;
        vv[DC - 2] = t.z;
        vv[DC - 1] = t.w;
    }
#pragma unroll
    for (int c = 0; c < DC; ++c)
#pragma unroll
        for (int r = 0; r < kSmallR; ++r) acc[r][c] = fmaf(pp[r], vv[c], acc[r][c]);
}

template <int D>
__global__ void __launch_bounds__(kSmallThreads, 2)
    mha_fwd_f32_small_kernel(const float *__restrict__ q, const float *__restrict__ k,
                             const float *__restrict__ v, const int32_t *__restrict__ kv_lengths,
                             float *__restrict__ out, float *__restrict__ lse, int H, int Lq,
                             int Lk, int mask_kind, float scale_log2, int keys_cap) {
    pdl_wait();      // the stream's previous kernel has completed; its writes are visible
    pdl_trigger();   // the next kernel may be scheduled
    using C = SmallCfg<D>;
    constexpr int DC = D / 32;   // output columns per lane
    constexpr int R = kSmallR;
    extern __shared__ float4 small_smem[];
    float *sK = reinterpret_cast<float *>(small_smem);   // [keys_cap][LDK]
    float *sV = sK + (size_t)keys_cap * C::LDK;          // [keys_cap][D]
    float *sQ = sV + (size_t)keys_cap * D;               // [16][D]
    float *sP = sQ + kSmallRows * D;                     // [warps][keys_cap][R]

    // Latest (for causal masks the heaviest) query blocks are launched first.
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

    constexpr int V4 = D / 4;
    for (int idx = tid; idx < kend * V4; idx += kSmallThreads) {
        const int r = idx / V4, c = idx % V4;
        cp_async16(sK + r * C::LDK + 4 * c, Kg + (size_t)r * D + 4 * c);
    }
    cp_async_commit();
    for (int idx = tid; idx < kend * V4; idx += kSmallThreads) {
        const int r = idx / V4, c = idx % V4;
        cp_async16(sV + r * D + 4 * c, Vg + (size_t)r * D + 4 * c);
    }
    cp_async_commit();
    for (int idx = tid; idx < kSmallRows * V4; idx += kSmallThreads) {
        const int r = idx / V4, c = idx % V4;
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (q0 + r < Lq) val = __ldg(reinterpret_cast<const float4 *>(Qg + (size_t)(q0 + r) * D) + c);
        *reinterpret_cast<float4 *>(sQ + r * D + 4 * c) = val;
    }
    cp_async_wait_group<1>();   // K has landed (V may still be in flight)
    __syncthreads();

    const int r0 = q0 + R * warp;                    // first row of this warp
    int kw = len;                                    // keys any of the warp's rows can see
    if (causal) kw = min(kw, r0 + R);
    kw = max(kw, 0);
    const int nkb = (kw + 31) / 32;
    const float *Qw = sQ + R * warp * D;

    // S for the warp's rows and keys kb*32 + lane.
    float s[R][C::KB];
#pragma unroll
    for (int kb = 0; kb < C::KB; ++kb)
#pragma unroll
        for (int r = 0; r < R; ++r) s[r][kb] = 0.f;
    switch (nkb) {
#define MHA_SMALL_S_CASE(N)                                                              \
    case N:                                                                              \
        if (N <= C::KB) small_scores<D, (N <= C::KB ? N : 1), C::KB>(sK, Qw, lane, s);   \
        break;
        MHA_SMALL_S_CASE(1)
        MHA_SMALL_S_CASE(2)
        MHA_SMALL_S_CASE(3)
        MHA_SMALL_S_CASE(4)
        MHA_SMALL_S_CASE(5)
        MHA_SMALL_S_CASE(6)
        MHA_SMALL_S_CASE(7)
        MHA_SMALL_S_CASE(8)
#undef MHA_SMALL_S_CASE
        default:
            break;
    }
    // Mask, scale into base 2, row max / exp / row sum (warp shuffles).
    float l[R], mrow[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int row = r0 + r;
        const int vis_end = causal ? min(len, row + 1) : len;
        float mx = -INFINITY;
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) {
            const int key = kb * 32 + lane;
            const float x = (kb < nkb && key < vis_end) ? s[r][kb] * scale_log2 : -INFINITY;
            s[r][kb] = x;
            mx = fmaxf(mx, x);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m = (mx == -INFINITY) ? 0.f : mx;
        float sum = 0.f;
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) {
            const float pj = ex2_approx(s[r][kb] - m);
            s[r][kb] = pj;
            sum += pj;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        l[r] = sum;
        mrow[r] = mx;
    }
    if (lse != nullptr && lane < R && r0 + lane < Lq) {
        float mm = mrow[0], ll = l[0];
#pragma unroll
        for (int r = 1; r < R; ++r)
            if (lane == r) {
                mm = mrow[r];
                ll = l[r];
            }
        lse[bh * (size_t)Lq + r0 + lane] = row_lse(mm, ll);
    }
    float *Pw = sP + (size_t)warp * keys_cap * R;
#pragma unroll
    for (int kb = 0; kb < C::KB; ++kb)
        if (kb < nkb)
        {
            float *dst = Pw + (kb * 32 + lane) * R;
            if (R == 4)
                *reinterpret_cast<float4 *>(dst) =
                    make_float4(s[0][kb], s[1][kb], s[R - 2][kb], s[R - 1][kb]);
            else
                *reinterpret_cast<float2 *>(dst) = make_float2(s[0][kb], s[1][kb]);
        }
    cp_async_wait_group<0>();   // V has landed
    __syncthreads();

    // O = P V for the warp's rows, lane's columns lane*DC .. lane*DC + DC - 1;
    // even and odd keys go to separate accumulators (two chains per output).
    float o[2][R][DC];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < DC; ++c) o[h2][r][c] = 0.f;
    const float *Vl = sV + lane * DC;
    int key = 0;
#pragma unroll 4
    for (; key + 1 < kw; key += 2) {
        small_pv_key<D>(Pw, Vl, key, o[0]);
        small_pv_key<D>(Pw, Vl, key + 1, o[1]);
    }
    if (key < kw) small_pv_key<D>(Pw, Vl, key, o[0]);
    // O / l; a row that saw no visible key (l == 0) is written as zeros.
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int row = r0 + r;
        if (row >= Lq) continue;
        const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
        float *dst = Og + (size_t)row * D + lane * DC;
        float res[DC];
#pragma unroll
        for (int c = 0; c < DC; ++c) res[c] = (o[0][r][c] + o[1][r][c]) * inv;
        if (DC == 2)
            *reinterpret_cast<float2 *>(dst) = make_float2(res[0], res[1]);
        else
            *reinterpret_cast<float4 *>(dst) = make_float4(res[0], res[1], res[DC - 2], res[DC - 1]);
    }
}

template <int D>
cudaError_t launch_small(const float *q, const float *k, const float *v, const int32_t *kv,
                         float *out, float *lse, int B, int H, int Lq, int Lk, int mask_kind, float scale,
                         cudaStream_t stream) {
    using C = SmallCfg<D>;
    const int keys_cap = ((Lk + 31) / 32) * 32;
    const size_t smem = C::smem(keys_cap);
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(mha_fwd_f32_small_kernel<D>), C::smem(C::kMaxKeys));
    if (e != cudaSuccess) return e;
    const dim3 grid((Lq + kSmallRows - 1) / kSmallRows, H, B);
    return launch_kernel(mha_fwd_f32_small_kernel<D>, grid, dim3(kSmallThreads), smem, stream, nullptr,
                         q, k, v, kv, out, lse, H, Lq, Lk, mask_kind, scale * 1.4426950408889634f,
                         keys_cap);
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
    return launch_kernel(mha_fwd_f32_kernel<D>, grid, dim3(kThreads), smem, stream, nullptr, q, k, v,
                         kv, out, lse, H, Lq, Lk, mask_kind, scale_log2);
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
    if ((which == 0 || which == 3) && tf32x3_applies(D))
        return launch_fwd_tf32x3(q, k, v, kv_lengths, out, lse, B, H, Lq, Lk, D, mask_kind, scale,
                                 stream, driver_err);
    if ((int64_t)Lk * D <= kSmallMaxKD && which != 1) {
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
