// fwd_bf16.cu -- fused masked multi-head attention forward for bf16 inputs on
// the sm_103a tensor cores (tcgen05 MMAs accumulating in TMEM, operands
// staged by TMA), and the Pre-LayerNorm cross-attention variant.
//
// Work item = one 128-row query tile of one (b, h).  CTA = 6 warps:
//   warps 0-3  softmax warpgroup: thread t owns query row t of the tile (TMEM
//              lane t).  Reads a 128 x 128 fp32 logit tile S from TMEM, masks
//              it from (row, col, length), runs the online softmax (running
//              max and rescaled running sum in registers), writes P as bf16
//              back into TMEM and rescales the O accumulator when the max
//              grows; finally divides O by the row sum and stores it through
//              shared memory with TMA.  In the Pre-LN variant it also
//              normalises the query rows and writes the Q tile to shared memory.
//   warp 4     TMA producer: Q tile once per item, then K and V tiles of 128
//              keys into a two-stage ring; key tiles past the causal limit or
//              the valid length are never loaded.
//   warp 5     MMA issuer: S_j = Q K_j^T (shared x shared -> TMEM) and
//              O += P_j V_j (P read from TMEM, V from shared memory).  Owns the
//              TMEM allocation.
// S is double-buffered in TMEM so S_{j+1} runs on the tensor cores while the
// softmax works on S_j.  All hand-offs are mbarriers; every wait is bounded.
//
// Page sections this follows: "Why attention must compute the max first"
// (gsyq.cn) 2.3-2.4 and 3.1 (online softmax with the max shift, fused between
// QK^T and PV, scores kept on chip); "masked multi head attention" CUDA
// article (2kiu.com) 2 and 3.1 (skip fully masked tiles, mask in-kernel as
// -infinity before the softmax); "How to fuse cross-attention and
// layer-norm into a single CUDA kernel?" (cms365.cn) answer steps one to
// four (Pre-LN fused into the Q load, cross-attention with online softmax,
// one write of O).
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kTileRows = 128;        // query rows per tile = keys per tile
constexpr int kHalfBytes = 128 * 128;  // one 128-row x 64-column bf16 box (16 KB)
constexpr int kThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
// TMEM column map (lane = query row): two S buffers, O, two P buffers.
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP0 = 384, kColP1 = 448;
// Conditional rescale: O and l keep a stale max until the tile max exceeds
// it by more than this many powers of two.  Exact after the final O / l.
constexpr float kRescaleThreshold = 8.0f;

struct AttnParams {
    CUtensorMap tm_q;     // Q [B*H][Lq][D], box {64, 128, 1}
    CUtensorMap tm_k;     // K [B*H][Lk][D]
    CUtensorMap tm_v;     // V [B*H][Lk][D]
    CUtensorMap tm_o;     // out: [B*H][Lq][D], or [B][Lq][H*D] for Pre-LN
    const __nv_bfloat16 *x;   // Pre-LN input [B][Lq][H*D]
    const float *gamma;
    const float *beta;
    float eps;
    const int32_t *kv_lengths;   // null unless the kv-length mask is on
    int B, H, Lq, Lk;
    int causal;
    float scale_log2;     // scale * log2(e)
    int n_qt;             // query tiles per (b, h)
    int n_items;          // B * H * n_qt
};

struct __align__(8) Bars {
    uint64_t q_full, q_empty;
    uint64_t k_full[2], v_full[2], kv_empty[2];
    uint64_t s_full[2], p_full[2], pv_done[2];
    uint64_t o_free;
    uint64_t wg_bar;     // bounded barrier of the 128 softmax threads
    uint64_t drain;      // teardown after an abort: in-flight MMAs done
    uint32_t tmem_base;
    int abort;
    float ln_mean[kTileRows];
    float ln_rstd[kTileRows];
};

template <int D>
struct Layout {
    static constexpr int NH = D / 64;                      // 64-column halves per tile
    static constexpr uint32_t kTile = NH * kHalfBytes;     // one 128 x D bf16 tile
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + kTile;             // two stages
    static constexpr uint32_t kV = kK + 2 * kTile;         // two stages
    static constexpr uint32_t kO = kV + 2 * kTile;         // epilogue staging
    static constexpr uint32_t kBars = kO + kTile;
    static constexpr size_t kSmem = 1024 + kBars + sizeof(Bars);
};

struct Item {
    int b, h, bh, q0;
    int len;      // visible keys of batch b (clamped)
    int n_kv;     // key tiles to visit
};

__device__ __forceinline__ Item decode_item(const AttnParams &p, int item) {
    Item it;
    const int BH = p.B * p.H;
    const int qt = p.n_qt - 1 - item / BH;     // heaviest (latest) query tiles first
    it.bh = item % BH;
    it.b = it.bh / p.H;
    it.h = it.bh % p.H;
    it.q0 = qt * kTileRows;
    int len = p.Lk;
    if (p.kv_lengths) len = max(0, min((int)p.kv_lengths[it.b], p.Lk));
    it.len = len;
    int kend = len;
    if (p.causal) kend = min(kend, it.q0 + kTileRows);
    it.n_kv = (kend + kTileRows - 1) / kTileRows;
    return it;
}

// Descriptor of K-step kk (16 bf16 along K) of a K-major 128-row tile stored
// as 64-column halves of 16 KB in the 128-byte swizzled layout.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile_saddr, int kk) {
    return sdesc_sw128(tile_saddr + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
}

// Descriptor of K-step kk (16 keys) of an MN-major [128 keys x N] tile (V),
// stored as 64-column halves: 8-key groups are 1024 B apart, halves 16 KB.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile_saddr, int kk) {
    return sdesc_sw128(tile_saddr + kk * 2048, kHalfBytes, 1024);
}

// Byte offset of 16-byte chunk `c` (0..D/8-1) of row `r` in a tile stored as
// 64-column halves with the 128-byte swizzle (what TMA reads and writes).
__device__ __forceinline__ uint32_t swz_off(int r, int c) {
    return (uint32_t)((c >> 3) * kHalfBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }
__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

// ---------------------------------------------------------------------------
// Pre-LN prologue: per-row mean and 1/sqrt(var + eps) of x[b, q0 + r, :] over
// the H*D features (fp32, shifted sums), then the head-h slice normalised,
// scaled by gamma, shifted by beta and written as bf16 into the Q tile.
// Thread t handles row t.
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void prenorm_q_tile(const AttnParams &p, const Item &it, uint8_t *sQ,
                                               int t) {
    const int N = p.H * D;
    const int row = it.q0 + t;
    uint8_t *dst_row_base = sQ;
    if (row < p.Lq) {
        const __nv_bfloat16 *xr = p.x + ((size_t)it.b * p.Lq + row) * (size_t)N;
        const uint4 *xv = reinterpret_cast<const uint4 *>(xr);
        const float shift = __bfloat162float(xr[0]);
        float s1 = 0.f, s2 = 0.f;
        const int nchunk = N / 8;
#pragma unroll 4
        for (int c = 0; c < nchunk; ++c) {
            const uint4 u = __ldg(xv + c);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a = __uint_as_float(w[e] << 16) - shift;
                const float bb = __uint_as_float(w[e] & 0xFFFF0000u) - shift;
                s1 += a + bb;
                s2 = fmaf(a, a, fmaf(bb, bb, s2));
            }
        }
        const float inv_n = 1.f / (float)N;
        const float dm = s1 * inv_n;
        const float var = fmaxf(s2 * inv_n - dm * dm, 0.f);
        const float mean = shift + dm;
        const float rstd = rsqrtf(var + p.eps);
        const uint4 *xs = xv + (it.h * D) / 8;
        const float *g = p.gamma + it.h * D;
        const float *bt = p.beta + it.h * D;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 u = __ldg(xs + c);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
            uint32_t o4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = c * 8 + 2 * e;
                const float a = __uint_as_float(w[e] << 16);
                const float bb = __uint_as_float(w[e] & 0xFFFF0000u);
                const float ya = fmaf((a - mean) * rstd, __ldg(g + col), __ldg(bt + col));
                const float yb = fmaf((bb - mean) * rstd, __ldg(g + col + 1), __ldg(bt + col + 1));
                o4[e] = pack_bf16x2(ya, yb);
            }
            *reinterpret_cast<uint4 *>(dst_row_base + swz_off(t, c)) =
                make_uint4(o4[0], o4[1], o4[2], o4[3]);
        }
    } else {
#pragma unroll
        for (int c = 0; c < D / 8; ++c)
            *reinterpret_cast<uint4 *>(dst_row_base + swz_off(t, c)) = make_uint4(0, 0, 0, 0);
    }
}

// ---------------------------------------------------------------------------
// The attention kernel.  Persistent-capable: CTA c takes items c, c + grid,
// c + 2*grid, ...; all barrier phases run on counters that continue across
// items (g = key tiles so far, qi = items with work so far).
// ---------------------------------------------------------------------------
template <int D, bool PRENORM>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ AttnParams p) {
    using L = Layout<D>;
    constexpr int NH = L::NH;
    constexpr uint32_t TILE = L::kTile;

    // A bounded wait that expired earlier leaves g_status set; later launches
    // then return at once instead of timing out again.
    if (*reinterpret_cast<volatile unsigned int *>(&g_status) != 0u) return;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *base = smem_raw + pad;
    uint8_t *sQ = base + L::kQ;
    uint8_t *sK = base + L::kK;
    uint8_t *sV = base + L::kV;
    uint8_t *sO = base + L::kO;
    Bars *bars = reinterpret_cast<Bars *>(base + L::kBars);
    volatile int *abort = &bars->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->k_full[i], 1);
            mbar_init(&bars->v_full[i], 1);
            mbar_init(&bars->kv_empty[i], 1);
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->p_full[i], kSoftmaxThreads);
            mbar_init(&bars->pv_done[i], 1);
        }
        mbar_init(&bars->o_free, kSoftmaxThreads);
        mbar_init(&bars->wg_bar, kSoftmaxThreads);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        mbar_fence_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        if (!PRENORM) tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        tma_prefetch_desc(&p.tm_o);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == kProducerWarp) {
        // ----------------------------- TMA producer -----------------------------
        if (lane == 0) {
            uint32_t g = 0, qi = 0;
            int q_issued = -1;          // phase of the last Q load issued
            bool ok = true;
            for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
                const Item it = decode_item(p, item);
                if (it.n_kv == 0) continue;
                if (!PRENORM) {
                    if (qi > 0) ok = mbar_wait(&bars->q_empty, (qi - 1) & 1, kSiteQEmpty, abort);
                    if (!ok) break;
                    q_issued = (int)(qi & 1);
                    mbar_arrive_expect_tx(&bars->q_full, TILE);
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh)
                        tma_load_3d(sQ + hh * kHalfBytes, &p.tm_q, &bars->q_full, hh * 64, it.q0,
                                    it.bh);
                }
                for (int j = 0; j < it.n_kv; ++j, ++g) {
                    const uint32_t st = g & 1;
                    if (g >= 2) {
                        ok = mbar_wait(&bars->kv_empty[st], ((g >> 1) - 1) & 1, kSiteKvEmpty, abort);
                        if (!ok) break;
                    }
                    mbar_arrive_expect_tx(&bars->k_full[st], TILE);
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh)
                        tma_load_3d(sK + st * TILE + hh * kHalfBytes, &p.tm_k, &bars->k_full[st],
                                    hh * 64, j * kTileRows, it.bh);
                    mbar_arrive_expect_tx(&bars->v_full[st], TILE);
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh)
                        tma_load_3d(sV + st * TILE + hh * kHalfBytes, &p.tm_v, &bars->v_full[st],
                                    hh * 64, j * kTileRows, it.bh);
                }
                ++qi;
            }
            if (!ok) {
                // Let the loads already issued land before shared memory is released.
                volatile int no_abort = 0;
                for (uint32_t gg = (g >= 2 ? g - 2 : 0); gg < g; ++gg) {
                    mbar_wait(&bars->k_full[gg & 1], (gg >> 1) & 1, kSiteDrain, &no_abort);
                    mbar_wait(&bars->v_full[gg & 1], (gg >> 1) & 1, kSiteDrain, &no_abort);
                }
                if (q_issued >= 0) mbar_wait(&bars->q_full, (uint32_t)q_issued, kSiteDrain, &no_abort);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0, 0);   // Q K-major, K K-major
            constexpr uint32_t idPV = idesc_bf16_f32(128, D, 0, 1);    // P (TMEM), V N-major
            const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
            uint32_t g = 0, qi = 0;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
                const Item it = decode_item(p, item);
                if (it.n_kv == 0) continue;
                ok = mbar_wait(&bars->q_full, qi & 1, kSiteQFull, abort);
                if (!ok) break;
                // S_g = Q K_g^T into S buffer g & 1.
                auto issue_s = [&](uint32_t gs) -> bool {
                    const uint32_t st = gs & 1;
                    if (!mbar_wait(&bars->k_full[st], (gs >> 1) & 1, kSiteKFull, abort)) return false;
                    tc_fence_after();
                    const uint32_t dS = tmem + (st ? kColS1 : kColS0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        umma_ss(dS, desc_kmajor(sQa, kk), desc_kmajor(sKa + st * TILE, kk), idS,
                                kk > 0 ? 1u : 0u);
                    umma_commit(&bars->s_full[st]);
                    return true;
                };
                const uint32_t g0 = g;
                ok = issue_s(g0);
                for (int j = 0; ok && j < it.n_kv; ++j) {
                    const uint32_t gj = g0 + j;
                    const uint32_t sb = gj & 1;
                    if (j + 1 < it.n_kv) {
                        ok = issue_s(gj + 1);
                        if (!ok) break;
                    } else {
                        umma_commit(&bars->q_empty);      // Q tile no longer read
                    }
                    ok = mbar_wait(&bars->p_full[sb], (gj >> 1) & 1, kSitePFull, abort) &&
                         mbar_wait(&bars->v_full[sb], (gj >> 1) & 1, kSiteVFull, abort);
                    if (ok && j == 0 && qi > 0)
                        ok = mbar_wait(&bars->o_free, (qi - 1) & 1, kSiteOFree, abort);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t aP = tmem + (sb ? kColP1 : kColP0);
#pragma unroll
                    for (int kk = 0; kk < kTileRows / 16; ++kk)
                        umma_ts(tmem + kColO, aP + kk * 8, desc_mnmajor(sVa + sb * TILE, kk), idPV,
                                (j > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(&bars->kv_empty[sb]);
                    umma_commit(&bars->pv_done[sb]);
                }
                g = g0 + it.n_kv;
                ++qi;
            }
        }
    } else {
        // --------------------------- softmax warpgroup ---------------------------
        const int t = threadIdx.x;                    // row within the tile, TMEM lane
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        uint32_t g = 0, qi = 0, wg_phase = 0;
        bool ok = true;
        // Waits whose outcome the whole warp shares, so warp-collective
        // tcgen05 loads and stores never run with part of the warp gone.
        auto wwait = [&](uint64_t *bar, uint32_t parity, uint32_t site) -> bool {
            const bool r = mbar_wait(bar, parity, site, abort);
            return __all_sync(0xffffffffu, r);
        };
        // Bounded barrier of the softmax warpgroup (an mbarrier, so an abort
        // elsewhere cannot leave these warps blocked).
        auto wg_sync = [&]() -> bool {
            mbar_arrive(&bars->wg_bar);
            const bool r = wwait(&bars->wg_bar, wg_phase & 1, kSiteWg);
            ++wg_phase;
            return r;
        };
        for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
            const Item it = decode_item(p, item);
            const int row = it.q0 + t;
            if (PRENORM && it.n_kv > 0) {
                if (qi > 0) ok = wwait(&bars->q_empty, (qi - 1) & 1, kSiteQEmpty);
                if (!ok) break;
                prenorm_q_tile<D>(p, it, sQ, t);
                fence_proxy_async_smem();
                if (!(ok = wg_sync())) break;
                if (t == 0) mbar_arrive(&bars->q_full);
            }
            const int vis_end = p.causal ? min(it.len, row + 1) : it.len;
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < it.n_kv; ++j) {
                const uint32_t gj = g + j;
                const uint32_t sb = gj & 1;
                ok = wwait(&bars->s_full[sb], (gj >> 1) & 1, kSiteSFull);
                if (!ok) break;
                tc_fence_after();
                float s[kTileRows];
                {
                    const uint32_t src = tmem + lane_off + (sb ? kColS1 : kColS0);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t r[32];
                        tmem_ld32(src + c * 32, r);
#pragma unroll
                        for (int e = 0; e < 32; ++e) s[c * 32 + e] = u2f(r[e]);
                    }
                }
                const int lim = vis_end - j * kTileRows;   // visible keys of this row in the tile
                if (lim < kTileRows) {
#pragma unroll
                    for (int c = 0; c < kTileRows; ++c)
                        if (c >= lim) s[c] = -INFINITY;
                }
                float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
                for (int c = 4; c < kTileRows; c += 4) {
                    mx0 = fmaxf(mx0, s[c]);
                    mx1 = fmaxf(mx1, s[c + 1]);
                    mx2 = fmaxf(mx2, s[c + 2]);
                    mx3 = fmaxf(mx3, s[c + 3]);
                }
                const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * p.scale_log2;
                const bool need = m_tile > m_used + kRescaleThreshold;
                float alpha = 1.f;
                if (need) {
                    alpha = ex2_approx(m_used - m_tile);
                    m_used = m_tile;
                }
                const float msub = (m_used == -INFINITY) ? 0.f : m_used;
                float rs0 = 0.f, rs1 = 0.f;
                uint32_t pk[kTileRows / 2];
#pragma unroll
                for (int c = 0; c < kTileRows; c += 2) {
                    const float e0 = ex2_approx(fmaf(s[c], p.scale_log2, -msub));
                    const float e1 = ex2_approx(fmaf(s[c + 1], p.scale_log2, -msub));
                    rs0 += e0;
                    rs1 += e1;
                    pk[c >> 1] = pack_bf16x2(e0, e1);
                }
                l = fmaf(l, alpha, rs0 + rs1);
                // P buffer sb was last read by the P.V MMA of tile gj - 2.
                if (gj >= 2) {
                    ok = wwait(&bars->pv_done[sb], ((gj - 2) >> 1) & 1, kSitePvDone);
                    if (!ok) break;
                    tc_fence_after();
                }
                {
                    const uint32_t dst = tmem + lane_off + (sb ? kColP1 : kColP0);
                    uint32_t r[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = pk[e];
                    tmem_st32(dst, r);
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = pk[32 + e];
                    tmem_st32(dst + 32, r);
                    tmem_st_wait();
                }
                // Rescale O once the P.V of the previous tile has landed.
                if (j > 0 && __any_sync(0xffffffffu, need)) {
                    const uint32_t gp = gj - 1;
                    ok = wwait(&bars->pv_done[gp & 1], (gp >> 1) & 1, kSitePvDone);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t oa = tmem + lane_off + kColO;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(oa + c * 32, r);
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = f2u(u2f(r[e]) * alpha);
                        tmem_st32(oa + c * 32, r);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                mbar_arrive(&bars->p_full[sb]);
            }
            if (!ok) break;

            // ------------------------------- epilogue -------------------------------
            // sO is reused per item: the previous item's TMA store must have read it.
            if (t == 0) tma_store_wait_read();
            if (!(ok = wg_sync())) break;
            if (it.n_kv > 0) {
                const uint32_t gl = g + it.n_kv - 1;
                ok = wwait(&bars->pv_done[gl & 1], (gl >> 1) & 1, kSitePvDone);
                if (!ok) break;
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const uint32_t oa = tmem + lane_off + kColO;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(oa + c * 32, r);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 w;
                        w.x = pack_bf16x2(u2f(r[q4 * 8 + 0]) * inv, u2f(r[q4 * 8 + 1]) * inv);
                        w.y = pack_bf16x2(u2f(r[q4 * 8 + 2]) * inv, u2f(r[q4 * 8 + 3]) * inv);
                        w.z = pack_bf16x2(u2f(r[q4 * 8 + 4]) * inv, u2f(r[q4 * 8 + 5]) * inv);
                        w.w = pack_bf16x2(u2f(r[q4 * 8 + 6]) * inv, u2f(r[q4 * 8 + 7]) * inv);
                        *reinterpret_cast<uint4 *>(sO + swz_off(t, c * 4 + q4)) = w;
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars->o_free);
            } else {
#pragma unroll
                for (int c = 0; c < D / 8; ++c)
                    *reinterpret_cast<uint4 *>(sO + swz_off(t, c)) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            if (!(ok = wg_sync())) break;
            if (t == 0) {
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) {
                    if (PRENORM)
                        tma_store_3d(&p.tm_o, sO + hh * kHalfBytes, it.h * D + hh * 64, it.q0, it.b);
                    else
                        tma_store_3d(&p.tm_o, sO + hh * kHalfBytes, hh * 64, it.q0, it.bh);
                }
                tma_store_commit();
            }
            g += it.n_kv;
            if (it.n_kv > 0) ++qi;
        }
        if (t == 0) tma_store_wait_all();
    }

    // ------------------------------- teardown --------------------------------
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        if (*abort) {
            // Let MMAs still in flight finish before the columns are released.
            if (lane == 0) {
                volatile int no_abort = 0;
                umma_commit(&bars->drain);
                mbar_wait(&bars->drain, 0, kSiteDrain, &no_abort);
            }
            __syncwarp();
        }
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Descriptor self-test: one 128-row tcgen05 GEMM tile built from the same
// descriptor helpers the attention kernel uses.
// ---------------------------------------------------------------------------
struct SelftestParams {
    CUtensorMap tm_a;        // variants 0/1: A [128][K] bf16
    CUtensorMap tm_b;        // variant 0: B [128][K]; variants 1/2: B [128 keys][N]
    const uint32_t *a_raw;   // variant 2: A rows as packed bf16 pairs
    float *c;
    int variant;
    int kn;                  // K (variant 0) or N (variants 1/2)
};

__global__ void __launch_bounds__(128, 1) selftest_umma_kernel(const __grid_constant__ SelftestParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *sA = smem_raw + pad;
    uint8_t *sB = sA + 2 * kHalfBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + 2 * kHalfBytes);   // [0] full, [1] done
    uint32_t *tbase = reinterpret_cast<uint32_t *>(bars + 2);
    int *abort = reinterpret_cast<int *>(tbase + 1);
    const int warp = threadIdx.x >> 5, t = threadIdx.x;
    const int variant = p.variant, kn = p.kn;

    if (t == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        *abort = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(tbase, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tbase;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

    if (variant == 2) {
        // Row t of A into TMEM columns 128..191 as packed bf16 pairs.
        uint32_t r[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = p.a_raw[t * 64 + e];
        tmem_st32(tmem + lane_off + 128, r);
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = p.a_raw[t * 64 + 32 + e];
        tmem_st32(tmem + lane_off + 160, r);
        tmem_st_wait();
        tc_fence_before();
    }
    __syncthreads();

    bool ok = true;
    if (t == 0) {
        const int a_halves = variant == 0 ? kn / 64 : 2;
        const int b_halves = kn / 64;
        const uint32_t bytes = (variant == 2 ? 0 : a_halves * kHalfBytes) + b_halves * kHalfBytes;
        mbar_arrive_expect_tx(&bars[0], bytes);
        if (variant != 2)
            for (int hh = 0; hh < a_halves; ++hh)
                tma_load_3d(sA + hh * kHalfBytes, &p.tm_a, &bars[0], hh * 64, 0, 0);
        for (int hh = 0; hh < b_halves; ++hh)
            tma_load_3d(sB + hh * kHalfBytes, &p.tm_b, &bars[0], hh * 64, 0, 0);
        ok = mbar_wait(&bars[0], 0, kSiteSelftest, abort);
        if (ok) {
            tc_fence_after();
            const uint32_t sAa = smem_u32(sA), sBa = smem_u32(sB);
            if (variant == 0) {
                const uint32_t id = idesc_bf16_f32(128, 128, 0, 0);
                for (int kk = 0; kk < kn / 16; ++kk)
                    umma_ss(tmem, desc_kmajor(sAa, kk), desc_kmajor(sBa, kk), id, kk > 0);
            } else if (variant == 1) {
                const uint32_t id = idesc_bf16_f32(128, kn, 0, 1);
                for (int kk = 0; kk < 8; ++kk)
                    umma_ss(tmem, desc_kmajor(sAa, kk), desc_mnmajor(sBa, kk), id, kk > 0);
            } else {
                const uint32_t id = idesc_bf16_f32(128, kn, 0, 1);
                for (int kk = 0; kk < 8; ++kk)
                    umma_ts(tmem, tmem + 128 + kk * 8, desc_mnmajor(sBa, kk), id, kk > 0);
            }
            umma_commit(&bars[1]);
        }
    }
    __syncthreads();
    ok = !*reinterpret_cast<volatile int *>(abort);
    if (ok) ok = mbar_wait(&bars[1], 0, kSiteSelftest, abort);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
        tc_fence_after();
        const int ncols = variant == 0 ? 128 : kn;
        for (int c = 0; c < ncols / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_off + c * 32, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) p.c[t * ncols + c * 32 + e] = u2f(r[e]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ------------------------------ host side ----------------------------------
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 3-D bf16 tensor map over a dense [d2][d1][d0] array with a {64, 128, 1} box
// and the 128-byte swizzle; rows outside the array read as zero.
CUresult encode_bf16_3d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1,
                        uint64_t d2) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return CUDA_ERROR_NOT_SUPPORTED;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int g_grid_override = 0;

template <int D, bool PRENORM>
cudaError_t launch_attn(const AttnParams &p, cudaStream_t stream) {
    constexpr size_t smem = Layout<D>::kSmem;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(attn_fwd_bf16_kernel<D, PRENORM>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    int grid = p.n_items;
    if (g_grid_override > 0 && g_grid_override < grid) grid = g_grid_override;
    attn_fwd_bf16_kernel<D, PRENORM><<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

void set_bf16_grid_override(int ctas) { g_grid_override = ctas; }

cudaError_t read_device_status(uint32_t *bits, bool clear) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
    if (e != cudaSuccess) return e;
    if (bits) *bits = v;
    if (clear && v != 0) {
        const unsigned int z = 0;
        e = cudaMemcpyToSymbol(g_status, &z, sizeof(z));
    }
    return e;
}

cudaError_t launch_fwd_bf16(const Bf16Call &c, cudaStream_t stream, int *driver_err) {
    *driver_err = 0;
    AttnParams p;
    std::memset(&p, 0, sizeof(p));
    const bool prenorm = c.x != nullptr;
    const uint64_t BH = (uint64_t)c.B * c.H;
    CUresult r = CUDA_SUCCESS;
    if (!prenorm) r = encode_bf16_3d(&p.tm_q, c.q, c.D, c.Lq, BH);
    if (r == CUDA_SUCCESS) {
        // With no keys the K/V maps are never used; point them at a valid array.
        const bool has_k = c.Lk > 0;
        r = encode_bf16_3d(&p.tm_k, has_k ? c.k : c.out, c.D, has_k ? c.Lk : 1, has_k ? BH : 1);
        if (r == CUDA_SUCCESS)
            r = encode_bf16_3d(&p.tm_v, has_k ? c.v : c.out, c.D, has_k ? c.Lk : 1, has_k ? BH : 1);
    }
    if (r == CUDA_SUCCESS) {
        if (prenorm)
            r = encode_bf16_3d(&p.tm_o, c.out, (uint64_t)c.H * c.D, c.Lq, c.B);
        else
            r = encode_bf16_3d(&p.tm_o, c.out, c.D, c.Lq, BH);
    }
    if (r != CUDA_SUCCESS) {
        *driver_err = (int)r;
        return cudaErrorInvalidValue;
    }
    p.x = reinterpret_cast<const __nv_bfloat16 *>(c.x);
    p.gamma = c.gamma;
    p.beta = c.beta;
    p.eps = c.eps;
    p.kv_lengths = (c.mask_kind & 2) ? c.kv_lengths : nullptr;
    p.B = c.B;
    p.H = c.H;
    p.Lq = c.Lq;
    p.Lk = c.Lk;
    p.causal = (c.mask_kind & 1) ? 1 : 0;
    p.scale_log2 = c.scale * 1.4426950408889634f;
    p.n_qt = (c.Lq + kTileRows - 1) / kTileRows;
    p.n_items = (int)(BH * (uint64_t)p.n_qt);
    if (prenorm) return c.D == 64 ? launch_attn<64, true>(p, stream) : launch_attn<128, true>(p, stream);
    return c.D == 64 ? launch_attn<64, false>(p, stream) : launch_attn<128, false>(p, stream);
}

cudaError_t launch_selftest_umma(int variant, int kn, const void *a, const void *b, float *c,
                                 cudaStream_t stream, int *driver_err) {
    *driver_err = 0;
    SelftestParams p;
    std::memset(&p, 0, sizeof(p));
    CUresult r = CUDA_SUCCESS;
    if (variant == 0) {
        r = encode_bf16_3d(&p.tm_a, a, kn, 128, 1);
        if (r == CUDA_SUCCESS) r = encode_bf16_3d(&p.tm_b, b, kn, 128, 1);
    } else {
        if (variant == 1) r = encode_bf16_3d(&p.tm_a, a, 128, 128, 1);
        if (r == CUDA_SUCCESS) r = encode_bf16_3d(&p.tm_b, b, kn, 128, 1);
    }
    if (r != CUDA_SUCCESS) {
        *driver_err = (int)r;
        return cudaErrorInvalidValue;
    }
    p.a_raw = reinterpret_cast<const uint32_t *>(a);
    p.c = c;
    p.variant = variant;
    p.kn = kn;
    const size_t smem = 1024 + 4 * kHalfBytes + 64;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(selftest_umma_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    selftest_umma_kernel<<<1, 128, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace mha
