// decode_bf16.cu -- masked multi-head attention forward for a few query rows
// (Lq <= 8) against a long bf16 key/value cache: the decode step of a
// KV-cached model, or its short chunks.  Same semantics as the main kernels
// (top-left causal rule, per-batch valid lengths, scale, zero rows when no key
// is visible); only the work split differs.
//
// The step is memory-bound (every visible K/V row is read once and used for
// at most 8 query rows), so the keys of one (b, h) are split over a
// thread-block cluster of up to 8 CTAs, each streaming its own contiguous key
// range:
//   - 8 warps per CTA; a warp takes blocks of 32 keys (lane = key) and forms
//     S for all R query rows with 16-byte loads of its key's K row (Q is
//     broadcast from shared memory), then runs an exact online softmax per
//     row (warp max / sum by shuffles) and adds P.V with lanes over the
//     output columns (each V row read once, coalesced).
//   - The 8 warps' partial (max, sum, O) meet in shared memory; the CTAs'
//     partials meet on cluster rank 0 through distributed shared memory, and
//     rank 0 writes O once.  No workspace in global memory, no mbarrier
//     waits: the only waits are the cluster's hardware barriers, which every
//     CTA reaches unconditionally.
//
// Page sections this follows: "masked multi head attention" CUDA article
// (2kiu.com) 6.3 (attention against a cached K/V, llama.cpp-style); "Why
// attention must compute the max first" (gsyq.cn) 2.3-2.4 (online softmax
// with the max shift; partial results combined by rescaling with the
// difference of their maxima).
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kDecWarps = 8;
constexpr int kDecThreads = 32 * kDecWarps;
constexpr int kDecMaxCluster = 8;
// Batches up to this count are ordered by visible length (below).
constexpr int kDecRankMaxB = 256;

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Partial result of a set of keys for R query rows: running max (base-2
// logits), sum of 2^(s - max), and O = sum of 2^(s - max) V.
template <int D, int R>
struct DecPartial {
    float m[R];
    float l[R];
    float o[R][D];
};

// 16-byte asynchronous copy global -> shared memory (completion per thread:
// cp.async.wait_group).
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Per-warp V staging: one 32-key block of V rows (32 x D bf16), filled by
// asynchronous copies issued together with the block's K loads.
template <int D>
constexpr size_t dec_smem_bytes() {
    return (size_t)kDecWarps * 32 * D * sizeof(__nv_bfloat16);
}

// Few query rows: two CTAs per SM (a (b, h) problem per CTA, 256 of them
// resident at once on 152 SMs).
template <int D, int R>
__global__ void __launch_bounds__(kDecThreads, R <= 2 ? 2 : 1)
    attn_decode_bf16_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                            const __nv_bfloat16 *__restrict__ v, const int32_t *__restrict__ kv_lengths,
                            __nv_bfloat16 *__restrict__ out, float *__restrict__ lse, int B, int H,
                            int Lq, int Lk, int mask_kind, float scale_log2) {
    pdl_wait();      // the stream's previous kernel has completed; its writes are visible
    pdl_trigger();   // the next kernel may be scheduled
    constexpr int DC = D / 32;   // output columns per lane
    __shared__ __align__(16) uint32_t sQ2[R][D / 2];   // Q rows as bf16 pairs (as given)
    __shared__ DecPartial<D, R> sW[kDecWarps];   // per-warp partials
    __shared__ DecPartial<D, R> sC;              // this CTA's partial (read by cluster rank 0)
    __shared__ __align__(16) float sP[kDecWarps][R][32];   // each warp's block weights
    extern __shared__ uint4 dec_smem[];          // [warp][32 keys][D] bf16 V staging

    const int split = blockIdx.x, nsplit = gridDim.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool causal = (mask_kind & 1) != 0;
    // Keys any query row of batch bb can see.
    auto visible = [&](int bb) {
        int len = Lk;
        if (kv_lengths != nullptr) len = max(0, min((int)kv_lengths[bb], Lk));
        return causal ? min(len, Lq) : len;
    };
    // Problem order: with per-batch lengths (and at most kDecRankMaxB
    // batches) grid row y takes the batch of rank y / H by decreasing visible
    // length (ties by index), so the longest problems start first and the
    // shortest fill the end of the launch; else y = b * H + h.
    int bh = blockIdx.y;
    if (kv_lengths != nullptr && B <= kDecRankMaxB) {
        __shared__ int s_batch;
        const int want = (int)blockIdx.y / H;
        for (int cand = tid; cand < B; cand += kDecThreads) {
            const int lc = visible(cand);
            int rank = 0;
            for (int o = 0; o < B; ++o) {
                const int lo = visible(o);
                rank += (lo > lc || (lo == lc && o < cand)) ? 1 : 0;
            }
            if (rank == want) s_batch = cand;   // ranks are a permutation: one writer
        }
        __syncthreads();
        bh = s_batch * H + (int)blockIdx.y % H;
    }
    const int kend = visible(bh / H);
    // This problem's keys in nsplit contiguous chunks of a multiple of 32.
    const int chunk = max(32, (((kend + nsplit - 1) / nsplit + 31) / 32) * 32);
    const int k0 = split * chunk, k1 = min(kend, k0 + chunk);

    const __nv_bfloat16 *Qg = q + (size_t)bh * Lq * D;
    const __nv_bfloat16 *Kg = k + (size_t)bh * Lk * D;
    const __nv_bfloat16 *Vg = v + (size_t)bh * Lk * D;
    for (int e = tid; e < R * D / 2; e += kDecThreads) {
        const int r = e / (D / 2), d2 = e % (D / 2);
        sQ2[r][d2] = r < Lq ? reinterpret_cast<const uint32_t *>(Qg + (size_t)r * D)[d2] : 0u;
    }
    __syncthreads();

    float m[R], l[R], o[R][DC];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int c = 0; c < DC; ++c) o[r][c] = 0.f;
    }
    __nv_bfloat16 *sVw = reinterpret_cast<__nv_bfloat16 *>(dec_smem) + (size_t)warp * 32 * D;
    for (int base = k0 + 32 * warp; base < k1; base += 32 * kDecWarps) {
        const int key = base + lane;
        const bool live = key < k1;
        // The block's V rows go to this warp's staging slot by asynchronous
        // copies (rows past the range copy the last valid row; their weight is
        // 0), so they are in flight together with the K loads below.  The
        // previous block's reads of the slot finished before this point
        // (__syncwarp at the end of the loop body).
        {
            constexpr int kChunks = D / 8;   // 16-byte chunks per row
#pragma unroll
            for (int t = lane; t < 32 * kChunks; t += 32) {
                const int jr = t / kChunks, c8 = t % kChunks;
                const int vrow = min(base + jr, k1 - 1);
                cp_async16(sVw + jr * D + c8 * 8, Vg + (size_t)vrow * D + c8 * 8);
            }
            cp_async_commit();
        }
        // Every load of the block's K rows is issued before any use (keys past
        // the range read the last valid row and are masked below).
        const uint4 *kr = reinterpret_cast<const uint4 *>(Kg + (size_t)min(key, k1 - 1) * D);
        uint4 ku[D / 8];
#pragma unroll
        for (int c8 = 0; c8 < D / 8; ++c8) ku[c8] = __ldg(kr + c8);
        // S for this lane's key and every row.
        float s[R];
#pragma unroll
        for (int r = 0; r < R; ++r) s[r] = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < D / 8; ++c8) {
            const uint4 u = ku[c8];
            const float kf[8] = {bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y),
                                 bf_lo(u.z), bf_hi(u.z), bf_lo(u.w), bf_hi(u.w)};
#pragma unroll
            for (int r = 0; r < R; ++r) {
                // Eight Q elements in one broadcast read.
                const uint4 qv = *reinterpret_cast<const uint4 *>(&sQ2[r][c8 * 4]);
                const float qf[8] = {bf_lo(qv.x), bf_hi(qv.x), bf_lo(qv.y), bf_hi(qv.y),
                                     bf_lo(qv.z), bf_hi(qv.z), bf_lo(qv.w), bf_hi(qv.w)};
#pragma unroll
                for (int e = 0; e < 8; ++e) s[r] = fmaf(qf[e], kf[e], s[r]);
            }
        }
        // Mask, block max, rescale, exponentials, row sums (base 2).
        float p[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const bool vis = live && r < Lq && (!causal || key <= r);
            const float x = vis ? s[r] * scale_log2 : -INFINITY;
            float mb = x;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
            const float m_new = fmaxf(m[r], mb);
            const float msub = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2_approx(m[r] - msub);
            m[r] = m_new;
            p[r] = ex2_approx(x - msub);
            float ps = p[r];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
            l[r] = fmaf(l[r], alpha, ps);
#pragma unroll
            for (int c = 0; c < DC; ++c) o[r][c] *= alpha;
            sP[warp][r][lane] = p[r];
        }
        // O += P V over the block's keys from the staged V rows; lane holds
        // output columns lane*DC ...; the weights come four keys at a time
        // from shared memory (one broadcast read).  Rows past the range carry
        // weight 0 (their p is 2^-inf) and their staged V rows are finite
        // copies, so a group of four is taken whole.
        cp_async_wait_all();
        __syncwarp();
        const int nk = min(32, k1 - base);
#pragma unroll 2
        for (int j0 = 0; j0 < 32; j0 += 4) {
            if (j0 >= nk) break;
            float4 p4[R];
#pragma unroll
            for (int r = 0; r < R; ++r) p4[r] = *reinterpret_cast<const float4 *>(&sP[warp][r][j0]);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const __nv_bfloat16 *vr = sVw + (j0 + jj) * D + lane * DC;
                float vv[DC];
                if (DC == 4) {
                    const uint2 u = *reinterpret_cast<const uint2 *>(vr);
                    vv[0] = bf_lo(u.x);
                    vv[1] = bf_hi(u.x);
                    vv[DC - 2] = bf_lo(u.y);
                    vv[DC - 1] = bf_hi(u.y);
                } else {
                    const uint32_t u = *reinterpret_cast<const uint32_t *>(vr);
                    vv[0] = bf_lo(u);
                    vv[DC - 1] = bf_hi(u);
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float pj = jj == 0 ? p4[r].x : jj == 1 ? p4[r].y : jj == 2 ? p4[r].z : p4[r].w;
#pragma unroll
                    for (int c = 0; c < DC; ++c) o[r][c] = fmaf(pj, vv[c], o[r][c]);
                }
            }
        }
        __syncwarp();   // the slot is free for the next block's copies
    }
    // Warp partials -> shared memory.
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (lane == 0) {
            sW[warp].m[r] = m[r];
            sW[warp].l[r] = l[r];
        }
#pragma unroll
        for (int c = 0; c < DC; ++c) sW[warp].o[r][lane * DC + c] = o[r][c];
    }
    __syncthreads();
    // CTA partial: combine the warps with 2^(m_w - m) (warp r handles row r).
    if (warp < R) {
        const int r = warp;
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, sW[w].m[r]);
        const float msub = (mm == -INFINITY) ? 0.f : mm;
        float ll = 0.f, oc[DC];
#pragma unroll
        for (int c = 0; c < DC; ++c) oc[c] = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
            const float f = ex2_approx(sW[w].m[r] - msub);
            ll = fmaf(sW[w].l[r], f, ll);
#pragma unroll
            for (int c = 0; c < DC; ++c) oc[c] = fmaf(sW[w].o[r][lane * DC + c], f, oc[c]);
        }
        if (lane == 0) {
            sC.m[r] = mm;
            sC.l[r] = ll;
        }
#pragma unroll
        for (int c = 0; c < DC; ++c) sC.o[r][lane * DC + c] = oc[c];
    }
    // Cluster: rank 0 combines every CTA's partial and writes O (bf16).
    cluster_sync_all();
    if (cluster_ctarank() == 0 && warp < R && warp < Lq) {
        const int r = warp;
        float mm = -INFINITY;
        for (int s = 0; s < nsplit; ++s) mm = fmaxf(mm, ld_cluster_f32(map_to_rank(&sC.m[r], s)));
        const float msub = (mm == -INFINITY) ? 0.f : mm;
        float ll = 0.f, oc[DC];
#pragma unroll
        for (int c = 0; c < DC; ++c) oc[c] = 0.f;
        for (int s = 0; s < nsplit; ++s) {
            const float f = ex2_approx(ld_cluster_f32(map_to_rank(&sC.m[r], s)) - msub);
            ll = fmaf(ld_cluster_f32(map_to_rank(&sC.l[r], s)), f, ll);
#pragma unroll
            for (int c = 0; c < DC; ++c)
                oc[c] = fmaf(ld_cluster_f32(map_to_rank(&sC.o[r][lane * DC + c], s)), f, oc[c]);
        }
        // A row that saw no visible key is written as zeros.
        const float inv = ll > 0.f ? 1.f / ll : 0.f;
        // Its sum is 0 with no visible key and at least 1 otherwise, unless an
        // input was not finite.
        bool nonfinite = false;
#pragma unroll
        for (int c = 0; c < DC; ++c) nonfinite |= !finite_f(oc[c] * inv);
        report_flag(!finite_f(ll), kFlagSum);
        report_flag(nonfinite, kFlagNonFinite);
        if (lse != nullptr && lane == 0)
            lse[(size_t)bh * Lq + r] =
                (ll > 0.f && mm != -INFINITY) ? 0.69314718055994531f * (mm + log2f(ll)) : -INFINITY;
        __nv_bfloat16 *dst = out + ((size_t)bh * Lq + r) * D + lane * DC;
#pragma unroll
        for (int c = 0; c < DC; ++c) dst[c] = __float2bfloat16_rn(oc[c] * inv);
    }
    // No CTA leaves while rank 0 may still read its shared memory.
    cluster_sync_all();
}

thread_local int g_decode_override = 0;  // 0 automatic, 1 never
thread_local int g_decode_splits = 0;   // 0 automatic, else CTAs per (b, h) (at most 8)

template <int D, int R>
cudaError_t launch_dec(const Bf16Call &c, int splits, cudaStream_t stream) {
    constexpr size_t smem = dec_smem_bytes<D>();
    // The limit covers the dynamic part (the V staging slots) only; the
    // static arrays come on top of it.
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(attn_decode_bf16_kernel<D, R>), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute cluster;
    cluster.id = cudaLaunchAttributeClusterDimension;
    cluster.val.clusterDim.x = (unsigned)splits;
    cluster.val.clusterDim.y = 1;
    cluster.val.clusterDim.z = 1;
    return launch_kernel(attn_decode_bf16_kernel<D, R>, dim3((unsigned)splits, (unsigned)(c.B * c.H), 1),
                         dim3(kDecThreads), smem, stream, &cluster,
                         reinterpret_cast<const __nv_bfloat16 *>(c.q),
                         reinterpret_cast<const __nv_bfloat16 *>(c.k),
                         reinterpret_cast<const __nv_bfloat16 *>(c.v),
                         (c.mask_kind & 2) ? c.kv_lengths : nullptr,
                         reinterpret_cast<__nv_bfloat16 *>(c.out), c.lse, c.B, c.H, c.Lq, c.Lk,
                         c.mask_kind, c.scale * 1.4426950408889634f);
}

template <int D>
cudaError_t launch_dec_rows(const Bf16Call &c, int splits, cudaStream_t stream) {
    if (c.Lq <= 1) return launch_dec<D, 1>(c, splits, stream);
    if (c.Lq <= 2) return launch_dec<D, 2>(c, splits, stream);
    if (c.Lq <= 4) return launch_dec<D, 4>(c, splits, stream);
    return launch_dec<D, 8>(c, splits, stream);
}

}  // namespace

cudaError_t status_ctl_decode_bf16(int op, uint64_t value, uint32_t *bits) {
    return unit_status_ctl(op, value, bits);
}

void set_decode_override(int which) { g_decode_override = which; }
void set_decode_splits(int splits) { g_decode_splits = splits; }

bool decode_applies(const Bf16Call &c) {
    // (b, h) problems are the grid's y dimension (at most 65535).
    return c.x == nullptr && c.Lq <= kDecodeMaxRows && g_decode_override != 1 &&
           (int64_t)c.B * c.H <= 65535;
}

cudaError_t launch_decode_bf16(const Bf16Call &c, int num_sms, cudaStream_t stream) {
    // Keys any row can see at most (each CTA splits its own problem's
    // visible keys into chunks of a multiple of 32).
    const int kend = (c.mask_kind & 1) ? (c.Lq < c.Lk ? c.Lq : c.Lk) : c.Lk;
    const int64_t BH = (int64_t)c.B * c.H;
    // About one CTA per SM in total, at least 256 keys per CTA, at most a
    // portable cluster of 8.  With at least one (b, h) per SM: two CTAs per
    // problem while one CTA per problem would fit in a single wave (few-row
    // launches hold two CTAs per SM), which evens out the end of the launch;
    // else one.  Measured on the 8 x 32-head decode step with cache lengths
    // 4096..8192 (longest problems first): one CTA per (b, h) 163 us, two
    // 161, three 164, four 168, eight 189.
    const int64_t slots = (int64_t)num_sms * (c.Lq <= 2 ? 2 : 1);
    int64_t want = ((int64_t)num_sms + BH - 1) / BH;
    if (BH >= num_sms && BH <= slots) want = 2;
    const int64_t by_keys = (kend + 255) / 256;
    if (want > by_keys) want = by_keys;
    if (want > kDecMaxCluster) want = kDecMaxCluster;
    if (want < 1) want = 1;
    if (g_decode_splits > 0) want = g_decode_splits < kDecMaxCluster ? g_decode_splits : kDecMaxCluster;
    const int splits = (int)want;
    return c.D == 64 ? launch_dec_rows<64>(c, splits, stream)
                     : launch_dec_rows<128>(c, splits, stream);
}

}  // namespace mha
