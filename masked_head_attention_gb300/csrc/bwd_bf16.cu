// bwd_bf16.cu -- backward pass of fused masked multi-head attention for bf16
// inputs on the sm_103a tensor cores (tcgen05 MMAs accumulating in TMEM,
// operands staged by TMA).
//
// The softmax weights are formed again from the forward's row log-sum-exp,
// p_ij = 2^(s_ij * scale * log2(e) - lse_i * log2(e)), and the softmax
// Jacobian of "Why attention must compute the max first" (gsyq.cn, section
// 3.3) is applied as dS_ij = p_ij (dP_ij - Delta_i), dP_ij = dout_i . v_j,
// Delta_i = dout_i . o_i (one row pass, shared with the CUDA-core backward).
// Two kinds of tile (bwd_tile<D, KV>), both run by one kernel launch, each
// CTA holding 128 rows of one (b, h) in TMEM lanes and streaming 64-row
// tiles of the other side:
//   KV = true  (key-stationary): rows = keys, stream query tiles.
//              S^T = K Q^T, dP^T = V dout^T; P^T and dS^T into TMEM;
//              dV += P^T dout, dK += dS^T Q  (dK scaled at the end).
//   KV = false (query-stationary): rows = queries, stream key tiles.
//              S = Q K^T, dP = dout V^T; dS into TMEM; dQ += dS K.
//              Q and dout sit in TMEM as the A operands of S and dP, so
//              those products read only the 64-row K / V tiles from shared
//              memory (with both operands in shared memory a 128 x 64 x 16
//              product is bound by the shared-memory port, not the math).
// No atomics: every gradient element is written once, the same on every run.
// The price is forming S and dP twice (seven products instead of five).
//
// CTA: the softmax warps (8 for D = 128: two per TMEM lane quadrant, each
// taking one 32-column half of a stream tile; 4 for D = 64), then a TMA
// producer warp and the MMA issuer / TMEM owner.  Stream tiles go through
// four shared-memory stages.  Per stream tile j the MMA warp issues S(j) and
// dP(j), waits for the softmax's P / dS, then the accumulating products,
// which read the stage and the P / dS columns before S(j + NB) overwrites
// them (NB = the number of S/dP buffers; the tensor pipe executes one
// thread's MMAs in order).
// TMEM: per S/dP buffer (two for D = 128, one for D = 64) S in its first 64
// columns and dP in the next 64; the packed bf16 pairs of P (KV) and dS
// overwrite the first 16 columns of each 32-column half of S and dP (KV: P
// over S, dS over dP; else dS over S).  The accumulators follow the buffers,
// then (query-stationary) Q and dout.
// With two buffers S(j + 1) and dP(j + 1) are issued before the products of
// tile j, so the softmax of a tile overlaps the products of its neighbours.
// All hand-offs are mbarriers; every wait is bounded.
#include <cstdint>
#include <cstring>
#include <type_traits>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kRowsB = 128;    // stationary rows per CTA
constexpr int kColsB = 64;     // rows of a stream tile
// Softmax warps: two per TMEM lane quadrant for D = 128 (each takes one
// 32-column half of a stream tile), one for D = 64 (both halves; two CTAs
// share an SM, which 320 threads of this size would not).  Then the TMA
// producer warp and the MMA warp.
template <int D>
constexpr int bwd_soft_warps() {
    return D == 128 ? 8 : 4;
}
template <int D>
constexpr int bwd_threads() {
    return 32 * (bwd_soft_warps<D>() + 2);
}
// Stream-tile stages (TMA runs up to three tiles ahead; a stage is released
// when the accumulating products of its tile have finished).  More stages
// (five, seven) measured no faster.
constexpr int kStagesB = 4;
// TMEM per S/dP buffer: S in columns [0, 64), dP in [64, 128) of the buffer.
constexpr uint32_t kColDpOff = 64;

struct BwdBf16Params {
    CUtensorMap tm_x, tm_y;     // stationary: KV: K, V; else Q, dout   (box rows 128)
    CUtensorMap tm_xs, tm_ys;   // stream:     KV: Q, dout; else K, V   (box rows 64)
    const float *lse;           // [B*H][Lq] natural log
    const float *delta;         // [B*H][Lq]
    const int32_t *kv_lengths;  // null unless the kv-length mask is on
    const __nv_bfloat16 *xa, *ya;   // query-stationary: Q and dout rows [B*H][Lq][D] (TMEM operands)
    __nv_bfloat16 *g1;          // KV: dK; else dQ     [B*H][rows][D]
    __nv_bfloat16 *g2;          // KV: dV; else unused
    int B, H, Lq, Lk;
    int causal;
    float scale, scale_log2;
};

struct __align__(8) BwdBars {
    uint64_t x_full, xa_full;   // stationary tile in shared memory (KV) / in TMEM (else)
    uint64_t st_full[kStagesB], st_empty[kStagesB];
    uint64_t s_full[2], p_full[2], acc_full, drain;   // s_full, p_full: per S/dP buffer
    uint32_t tmem_base;
    int abort;
};

template <int D, bool KV>
struct BwdBf16Cfg {
    static constexpr int NH = D / 64;                      // 64-column halves
    static constexpr uint32_t kHalfX = kRowsB * 128;       // 16 KB
    static constexpr uint32_t kHalfS = kColsB * 128;       // 8 KB
    static constexpr uint32_t kTileX = NH * kHalfX;
    static constexpr uint32_t kTileS = NH * kHalfS;
    // The key-stationary kernel keeps K and V in shared memory (the S and dP
    // products read both operands from there); the query-stationary kernel
    // keeps Q and dout in TMEM and needs no stationary tile here.
    static constexpr uint32_t kX = 0, kY = kTileX;
    static constexpr uint32_t kStage = KV ? 2 * kTileX : 0;  // stage s: xs at kStage + s*2*kTileS, ys after it
    // KV: per softmax warp, two slots of 64 (lse2, Delta) pairs (the current
    // and the next stream tile's query columns).
    static constexpr uint32_t kStat = kStage + 2 * kStagesB * kTileS;
    static constexpr uint32_t kBars = kStat + (KV ? 4 * 2 * 64 * 8 : 0);   // SW warps x 2 x (256 / SW) pairs
    static constexpr size_t kSmem = 1024 + kBars + sizeof(BwdBars);
};

// S/dP buffers in TMEM: two for D = 128 (the softmax of one stream tile
// overlaps the products of the next), one for D = 64 (two CTAs share an SM).
template <int D>
constexpr int bwd_sdp_buffers() {
    return D == 128 ? 2 : 1;
}
// TMEM columns: the S/dP buffers (128 each), then the accumulators: dV, dK
// (D columns each) for KV; else dQ (D columns) followed by Q and dout as MMA
// A operands (D / 2 columns each, bf16 pairs).  2D after the buffers either
// way; a power of two.
template <int D, bool KV>
constexpr uint32_t bwd_tmem_cols() {
    return (128 * bwd_sdp_buffers<D>() + 2 * D) <= 256 ? 256u : 512u;
}

// K-major descriptor of K-step kk (16 bf16 along the row) of a tile stored as
// 64-column halves of `half` bytes in the 128-byte swizzled layout.
__device__ __forceinline__ uint64_t desc_k(uint32_t tile, int kk, uint32_t half) {
    return sdesc_sw128(tile + (kk >> 2) * half + (kk & 3) * 32, 16, 1024);
}
// MN-major descriptor of K-step kk (16 rows) of a [rows][D] tile used as the
// B operand with N = D (64-column halves `half` bytes apart).
__device__ __forceinline__ uint64_t desc_mn(uint32_t tile, int kk, uint32_t half) {
    return sdesc_sw128(tile + kk * 2048, half, 1024);
}

// One 128-row stationary tile: rank tr of n_tiles on its side (heaviest
// first), problem bh.
template <int D, bool KV>
__device__ __forceinline__ void bwd_tile(const BwdBf16Params &p, int tr, int n_tiles, int bh) {
    using C = BwdBf16Cfg<D, KV>;
    constexpr int NH = C::NH;
    constexpr int NS = kStagesB;
    constexpr int SW = bwd_soft_warps<D>();
    constexpr int kProdWarpB = SW, kMmaWarpB = SW + 1;
    if (wait_expired_before()) return;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *base = smem_raw + pad;
    BwdBars *bars = reinterpret_cast<BwdBars *>(base + C::kBars);
    volatile int *abort = &bars->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // This CTA's stationary tile and the stream tiles it visits.  Ranks run
    // heaviest first: under the causal rule the first key tiles see the most
    // queries, the last query tiles the most keys.
    const int tile = (KV || !p.causal) ? tr : n_tiles - 1 - tr;
    const int b = bh / p.H;
    const int r0 = tile * kRowsB;
    int len = p.Lk;
    if (p.kv_lengths) len = max(0, min((int)p.kv_lengths[b], p.Lk));
    int j0, j1;   // stream tiles [j0, j1)
    if (KV) {
        // Query tiles that see a key of [r0, r0 + 128): none past the length;
        // under the causal rule only queries >= r0.
        j0 = p.causal ? r0 / kColsB : 0;
        j1 = r0 < len ? (p.Lq + kColsB - 1) / kColsB : j0;
    } else {
        int kend = len;
        if (p.causal) kend = min(kend, r0 + kRowsB);
        j0 = 0;
        j1 = (kend + kColsB - 1) / kColsB;
    }
    const int n = max(0, j1 - j0);

    // Start-up work that needs no other role goes out before the CTA-wide
    // barrier: the query-stationary softmax threads issue their row loads of
    // Q and dout (stored to TMEM after it), and the producer lane prefetches
    // the tensor maps, sets up the barriers (nothing else touches them before
    // the CTA-wide barrier) and starts the stationary tile and the first
    // stream stages.
    constexpr int NG = 2 / (SW / 4);   // query-stationary: operands per softmax warp (Q, dout)
    uint32_t xa_w[KV ? 1 : NG][KV ? 1 : D / 2];
    if (!KV && warp < SW && n > 0) {
        const int row = r0 + 32 * (warp & 3) + lane;
        const bool have_row = row < p.Lq;
        const size_t off = ((size_t)bh * p.Lq + (have_row ? row : 0)) * D;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const uint4 *src = reinterpret_cast<const uint4 *>(((warp >> 2) * NG + g == 0 ? p.xa : p.ya) + off);
#pragma unroll
            for (int u = 0; u < (KV ? 0 : D / 8); ++u) {
                const uint4 v = have_row ? __ldg(src + u) : make_uint4(0u, 0u, 0u, 0u);
                xa_w[g][4 * u] = v.x;
                xa_w[g][4 * u + 1] = v.y;
                xa_w[g][4 * u + 2] = v.z;
                xa_w[g][4 * u + 3] = v.w;
            }
        }
    }
    int pre_issued = 0;   // stream stages the producer lane started before the barrier
    if (warp == kProdWarpB && lane == 0) {
        tma_prefetch_desc(&p.tm_xs);
        tma_prefetch_desc(&p.tm_ys);
        if (KV) {
            tma_prefetch_desc(&p.tm_x);
            tma_prefetch_desc(&p.tm_y);
        }
        mbar_init(&bars->x_full, 1);
        mbar_init(&bars->xa_full, SW);   // one arrival per softmax warp
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars->st_full[s], 1);
            mbar_init(&bars->st_empty[s], 1);
        }
        for (int bb = 0; bb < 2; ++bb) {
            mbar_init(&bars->s_full[bb], 1);
            mbar_init(&bars->p_full[bb], SW);   // one arrival per softmax warp
        }
        mbar_init(&bars->acc_full, 1);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        mbar_fence_init();
        if (n > 0) {
            if (KV) {
                mbar_arrive_expect_tx(&bars->x_full, 2 * C::kTileX);
                for (int hh = 0; hh < NH; ++hh) {
                    tma_load_3d(base + C::kX + hh * C::kHalfX, &p.tm_x, &bars->x_full, hh * 64, r0, bh);
                    tma_load_3d(base + C::kY + hh * C::kHalfX, &p.tm_y, &bars->x_full, hh * 64, r0, bh);
                }
            }
            for (; pre_issued < NS && pre_issued < n; ++pre_issued) {
                uint8_t *st = base + C::kStage + pre_issued * 2 * C::kTileS;
                const int c0 = (j0 + pre_issued) * kColsB;
                mbar_arrive_expect_tx(&bars->st_full[pre_issued], 2 * C::kTileS);
                for (int hh = 0; hh < NH; ++hh) {
                    tma_load_3d(st + hh * C::kHalfS, &p.tm_xs, &bars->st_full[pre_issued], hh * 64, c0, bh);
                    tma_load_3d(st + C::kTileS + hh * C::kHalfS, &p.tm_ys, &bars->st_full[pre_issued], hh * 64,
                                c0, bh);
                }
            }
        }
    }
    constexpr uint32_t kTmemCols = bwd_tmem_cols<D, KV>();
    if (warp == kMmaWarpB) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    auto wwait = [&](uint64_t *bar, uint32_t parity, uint32_t site) -> bool {
        const bool r = mbar_wait(bar, parity, site, abort);
        return __all_sync(0xffffffffu, r);
    };

    if (warp == kProdWarpB) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0 && n > 0) {
            bool ok = true;
            int issued = pre_issued;   // the stationary tile and stages [0, pre_issued) went out above
            for (int j = pre_issued; ok && j < n; ++j) {
                const int s = j % NS;
                if (j >= NS)
                    ok = mbar_wait(&bars->st_empty[s], ((j / NS) - 1) & 1, kSiteKvEmpty, abort);
                if (!ok) break;
                uint8_t *st = base + C::kStage + s * 2 * C::kTileS;   // s = j % NS
                const int c0 = (j0 + j) * kColsB;
                mbar_arrive_expect_tx(&bars->st_full[s], 2 * C::kTileS);
                for (int hh = 0; hh < NH; ++hh) {
                    tma_load_3d(st + hh * C::kHalfS, &p.tm_xs, &bars->st_full[s], hh * 64, c0, bh);
                    tma_load_3d(st + C::kTileS + hh * C::kHalfS, &p.tm_ys, &bars->st_full[s], hh * 64, c0,
                                bh);
                }
                issued = j + 1;
            }
            // Loads already issued must land before shared memory is released.
            volatile int no_abort = 0;
            if (KV) mbar_wait(&bars->x_full, 0, kSiteDrain, &no_abort);
            for (int j = max(0, issued - NS); j < issued; ++j)
                mbar_wait(&bars->st_full[j % NS], (j / NS) & 1, kSiteDrain, &no_abort);
        }
    } else if (warp == kMmaWarpB) {
        // ------------------------------- MMA issuer -------------------------------
        constexpr uint32_t idS = idesc_bf16_f32(128, kColsB, 0, 0);   // both operands K-major
        constexpr uint32_t idAcc = idesc_bf16_f32(128, D, 0, 1);      // A from TMEM, B MN-major
        constexpr int NB = bwd_sdp_buffers<D>();
        constexpr uint32_t kAcc = 128 * NB;                           // first accumulator column
        constexpr uint32_t kXa = kAcc + D, kYa = kXa + D / 2;         // query-stationary: Q, dout
        bool ok = n > 0, issued = false;
        // Under a test's short wait limit: a wait that must expire (the drain
        // phase completes only at teardown).
        if (ok && wait_limit_is_test()) ok = wwait(&bars->drain, 0, kSiteTest);
        if (ok) ok = KV ? wwait(&bars->x_full, 0, kSiteQFull) : wwait(&bars->xa_full, 0, kSiteQFull);
        const uint32_t sx = smem_u32(base + C::kX), sy = smem_u32(base + C::kY);
        // S(j) = X Xs^T and dP(j) = Y Ys^T (128 x 64 each, K = D) into buffer
        // j % NB; the caller has waited for stage j and commits s_full.
        auto issue_sdp = [&](int j) {
            const uint32_t sxs = smem_u32(base + C::kStage + (j % NS) * 2 * C::kTileS);
            const uint32_t sys = sxs + C::kTileS;
            const uint32_t cs = (uint32_t)(j % NB) * 128;
            if (KV) {   // K and V from shared memory
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    if (elect_one())
                        umma_ss(tmem + cs, desc_k(sx, kk, C::kHalfX), desc_k(sxs, kk, C::kHalfS), idS, kk > 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    if (elect_one())
                        umma_ss(tmem + cs + kColDpOff, desc_k(sy, kk, C::kHalfX), desc_k(sys, kk, C::kHalfS),
                                idS, kk > 0);
            } else {    // Q and dout from TMEM (8 columns per K-step of 16)
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    if (elect_one()) umma_ts(tmem + cs, tmem + kXa + kk * 8, desc_k(sxs, kk, C::kHalfS), idS, kk > 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    if (elect_one())
                        umma_ts(tmem + cs + kColDpOff, tmem + kYa + kk * 8, desc_k(sys, kk, C::kHalfS), idS,
                                kk > 0);
            }
            issued = true;
        };
        auto commit_s = [&](int j) {
            if (elect_one()) umma_commit(&bars->s_full[j % NB]);
            __syncwarp();
        };
        // Accumulating products of tile j over its 64 rows (4 K-steps of 16;
        // P / dS as packed bf16 pairs, 8 TMEM columns per K-step, the pairs of
        // each 32-row half at the start of that half's 32 columns); the caller
        // has waited for the softmax.  Then the stage is released.
        auto pcol = [](int kk) -> uint32_t { return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8); };
        auto issue_acc = [&](int j) {
            const uint32_t sxs = smem_u32(base + C::kStage + (j % NS) * 2 * C::kTileS);
            const uint32_t sys = sxs + C::kTileS;
            const uint32_t cs = (uint32_t)(j % NB) * 128;
            if (KV) {
#pragma unroll
                for (int kk = 0; kk < kColsB / 16; ++kk)
                    if (elect_one())   // dV += P^T dout
                        umma_ts(tmem + kAcc, tmem + cs + pcol(kk), desc_mn(sys, kk, C::kHalfS), idAcc,
                                (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < kColsB / 16; ++kk)
                    if (elect_one())   // dK += dS^T Q
                        umma_ts(tmem + kAcc + D, tmem + cs + kColDpOff + pcol(kk), desc_mn(sxs, kk, C::kHalfS),
                                idAcc, (j > 0 || kk > 0) ? 1u : 0u);
            } else {
#pragma unroll
                for (int kk = 0; kk < kColsB / 16; ++kk)
                    if (elect_one())   // dQ += dS K
                        umma_ts(tmem + kAcc, tmem + cs + pcol(kk), desc_mn(sxs, kk, C::kHalfS), idAcc,
                                (j > 0 || kk > 0) ? 1u : 0u);
            }
            if (elect_one()) {
                umma_commit(&bars->st_empty[j % NS]);
                if (j == n - 1) umma_commit(&bars->acc_full);
            }
            __syncwarp();
        };
        // Tensor-pipe order: S/dP(0) (and S/dP(1) with two buffers), then per
        // tile j its products followed by S/dP(j + NB), which overwrites the
        // buffer those products read just before it (one thread's MMAs execute
        // in order).  With two buffers the softmax of tile j + 1 overlaps the
        // products of j and S/dP(j + 2).
        // A wait of this warp placed after a commit returns only once every
        // product issued before that commit has finished, so the waits of a
        // tile come before its issues.  (Holding the S/dP commit back past the
        // next wait keeps the pipe busier but delays the softmax by this
        // warp's reaction time; measured slower.)
        for (int j = 0; ok && j < NB && j < n; ++j) {
            ok = wwait(&bars->st_full[j % NS], (j / NS) & 1, kSiteKFull);
            if (ok) {
                tc_fence_after();
                issue_sdp(j);
                commit_s(j);
            }
        }
        for (int j = 0; ok && j < n; ++j) {
            const int jn = j + NB;
            ok = wwait(&bars->p_full[j % NB], (j / NB) & 1, kSitePFull);
            if (ok && jn < n) ok = wwait(&bars->st_full[jn % NS], (jn / NS) & 1, kSiteKFull);
            if (!ok) break;
            tc_fence_after();
            issue_acc(j);
            if (jn < n) {
                issue_sdp(jn);
                commit_s(jn);
            }
        }
        if (issued) {
            volatile int no_abort = 0;
            if (elect_one()) umma_commit(&bars->drain);
            __syncwarp();
            mbar_wait(&bars->drain, 0, kSiteDrain, &no_abort);
            __syncwarp();
        }
    } else {
        // --------------------------------- softmax --------------------------------
        // Warp w owns TMEM lane quadrant w % 4 (rows 32 (w % 4) + lane) and,
        // with two warps per quadrant, the 32-column half w / 4 of each tile.
        constexpr int G = SW / 4;          // warps per quadrant
        constexpr int HPW = 2 / G;         // 32-column halves per warp
        const int gi = warp >> 2;          // this warp's group within the quadrant
        const int h0 = gi * HPW;           // first half this warp handles
        const int t = 32 * (warp & 3) + lane;   // stationary row within the tile = TMEM lane
        const int row = r0 + t;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const float *lse_bh = p.lse + (size_t)bh * p.Lq;
        const float *dl_bh = p.delta + (size_t)bh * p.Lq;
        constexpr float kLog2e = 1.4426950408889634f;
        // dQ kernel: the row's own statistics.
        float lse2_row = 0.f, dl_row = 0.f;
        if (!KV && row < p.Lq) {
            lse2_row = lse_bh[row] * kLog2e;
            dl_row = dl_bh[row];
        }
        // KV: this warp's copies of its query columns' (lse2, Delta) pairs,
        // two slots: the next tile's are fetched while the current one is
        // used.  (One copy shared by all warps needs a barrier per tile, which
        // measured slower.)
        constexpr int kWCols = 32 * HPW;   // columns per warp
        float2 *stw = reinterpret_cast<float2 *>(base + C::kStat) + warp * 2 * kWCols;
        auto fetch_stats = [&](int jj, float2 (&v)[HPW]) {
            const int cb = (j0 + jj) * kColsB + 32 * h0;
#pragma unroll
            for (int u = 0; u < HPW; ++u) {
                const int qc = cb + lane + 32 * u;
                v[u] = qc < p.Lq ? make_float2(lse_bh[qc] * kLog2e, dl_bh[qc]) : make_float2(0.f, 0.f);
            }
        };
        // Query-stationary: the row's Q and dout into TMEM (bf16 pairs, the
        // A-operand layout of the S and dP products; zeros past Lq); with two
        // warps per quadrant each writes one of the two.  One memory round
        // trip: every load was issued before the first store.
        if constexpr (!KV) {
          if (n > 0) {
            constexpr uint32_t kXa = 128 * bwd_sdp_buffers<D>() + D;
            // The rows were loaded before the CTA-wide barrier (xa_w).
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                const uint32_t dst = tmem + lane_off + kXa + (gi * NG + g) * (D / 2);
                if constexpr (D == 128) {
                    tmem_st64(dst, *reinterpret_cast<uint32_t(*)[64]>(xa_w[g]));
                } else {
                    tmem_st32(dst, *reinterpret_cast<uint32_t(*)[32]>(xa_w[g]));
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->xa_full);
          }
        }
        float2 nxt[HPW];
        if (KV && n > 0) fetch_stats(0, nxt);
        bool ok = true;
        for (int j = 0; ok && j < n; ++j) {
            const int c0 = (j0 + j) * kColsB;
            float2 *cur = stw + (j & 1) * kWCols;
            if (KV) {
                // Slot j & 1 was last read for tile j - 2, before this warp's
                // tile j - 1 work; the lanes are converged here.
                __syncwarp();
#pragma unroll
                for (int u = 0; u < HPW; ++u) cur[lane + 32 * u] = nxt[u];
                __syncwarp();
                if (j + 1 < n) fetch_stats(j + 1, nxt);   // in flight during this tile
            }
            constexpr int NB = bwd_sdp_buffers<D>();
            const uint32_t cs = (uint32_t)(j % NB) * 128;   // this tile's S/dP buffer
            ok = wwait(&bars->s_full[j % NB], (j / NB) & 1, kSiteSFull);
            if (!ok) break;
            tc_fence_after();
            // A tile every position of which is visible (inside the length, the
            // query range and the causal triangle) skips the element test.
            const bool interior =
                KV ? (r0 + kRowsB <= len && c0 + kColsB <= p.Lq && (!p.causal || r0 + kRowsB - 1 <= c0))
                   : (c0 + kColsB <= len && r0 + kRowsB <= p.Lq && (!p.causal || c0 + kColsB - 1 <= r0));
            const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
            // The visible columns of this row form one range [vlo, vhi) relative
            // to the tile: KV (row = key): queries from the key on (causal) up to
            // Lq, none for a key past the length; else (row = query): keys
            // below the length and up to the query (causal), none past Lq.
            int vlo, vhi;
            if (KV) {
                vlo = (p.causal ? row : 0) - c0;
                vhi = row < len ? p.Lq - c0 : vlo;
            } else {
                vlo = -c0;
                vhi = row < p.Lq ? (p.causal ? min(len, row + 1) : len) - c0 : vlo;
            }
            // The element loop in two compiled forms, chosen by a warp-uniform
            // test: without the visibility test (a straight line the compiler
            // schedules across columns) and with it.  Half h covers columns
            // [32h, 32h + 32) of S and dP; its P and dS (packed bf16 pairs) go to
            // the first 16 of those columns of S and of dP, read by this warp.
            auto tile_math = [&](auto masked_tag) {
                constexpr bool kMasked = decltype(masked_tag)::value;
#pragma unroll
                for (int hu = 0; hu < HPW; ++hu) {
                    const int half = h0 + hu;
                    const uint32_t hc = (uint32_t)(32 * half);
                    const int lo = vlo - 32 * half, hi = vhi - 32 * half;   // relative to the half
                    uint32_t sr[32], dr[32], pk[16], dk[16];
                    tmem_ld32_pair(tmem + lane_off + cs + hc, sr, tmem + lane_off + cs + kColDpOff + hc, dr);
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        // Statistics of the two columns (KV: per query column; else the row's).
                        float2 nl2, ndl;
                        if (KV) {
                            const float4 st = *reinterpret_cast<const float4 *>(cur + 32 * hu + c);   // (l2, dl) x 2
                            nl2 = make_float2(-st.x, -st.z);
                            ndl = make_float2(-st.y, -st.w);
                        } else {
                            nl2 = make_float2(-lse2_row, -lse2_row);
                            ndl = make_float2(-dl_row, -dl_row);
                        }
                        const float2 x =
                            __ffma2_rn(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, nl2);
                        float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                        if (kMasked) {
                            pr.x = (c >= lo && c < hi) ? pr.x : 0.f;
                            pr.y = (c + 1 >= lo && c + 1 < hi) ? pr.y : 0.f;
                        }
                        const float2 dd =
                            __fadd2_rn(make_float2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])), ndl);
                        const float2 ds = __fmul2_rn(pr, dd);
                        pk[c >> 1] = pack_bf16x2(pr.x, pr.y);
                        dk[c >> 1] = pack_bf16x2(ds.x, ds.y);
                    }
                    if (KV) {
                        tmem_st16(tmem + lane_off + cs + hc, pk);               // P^T over S
                        tmem_st16(tmem + lane_off + cs + kColDpOff + hc, dk);   // dS^T over dP
                    } else {
                        tmem_st16(tmem + lane_off + cs + hc, dk);               // dS over S
                    }
                }
            };
            if (interior)
                tile_math(std::false_type{});
            else
                tile_math(std::true_type{});
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full[j % NB]);
        }
        // Epilogue: the accumulators (scaled) as bf16, one row per thread (its
        // share of the 32-column chunks).  The wait and the TMEM loads are
        // warp-collective, so every lane runs them; only the stores depend on
        // the row.
        const int rows_valid = KV ? p.Lk : p.Lq;
        bool have = false;
        if (ok && n > 0) {
            have = wwait(&bars->acc_full, 0, kSitePvDone);   // warp-uniform
            if (have) tc_fence_after();
        }
        if (ok && (n == 0 || have)) {
            const bool store = row < rows_valid;
            constexpr int kChunks = (D / 32) / G;   // 32-column chunks per warp and accumulator
#pragma unroll
            for (int ai = 0; ai < (KV ? 2 : 1); ++ai) {
                // KV: ai 0 = dV (first accumulator), ai 1 = dK (after it, scaled);
                // else dQ (scaled).
                __nv_bfloat16 *dst = (KV && ai == 0 ? p.g2 : p.g1) +
                                     ((size_t)bh * rows_valid + (store ? row : 0)) * D;
                const float sc = (KV && ai == 0) ? 1.f : p.scale;
#pragma unroll
                for (int cu = 0; cu < kChunks; ++cu) {
                    const int ch = gi * kChunks + cu;
                    uint32_t a[32];
                    if (have) {
                        tmem_ld32(tmem + lane_off + 128 * bwd_sdp_buffers<D>() + (KV && ai == 1 ? D : 0) +
                                      ch * 32, a);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) a[e] = 0u;
                    }
                    if (store) {
#pragma unroll
                        for (int e = 0; e < 32; e += 8) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(a[e]) * sc, __uint_as_float(a[e + 1]) * sc);
                            w.y = pack_bf16x2(__uint_as_float(a[e + 2]) * sc, __uint_as_float(a[e + 3]) * sc);
                            w.z = pack_bf16x2(__uint_as_float(a[e + 4]) * sc, __uint_as_float(a[e + 5]) * sc);
                            w.w = pack_bf16x2(__uint_as_float(a[e + 6]) * sc, __uint_as_float(a[e + 7]) * sc);
                            *reinterpret_cast<uint4 *>(dst + ch * 32 + e) = w;
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarpB) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Both halves of the backward in one launch: the key-stationary tiles (dK,
// dV) and the query-stationary tiles (dQ) are independent, so one grid holds
// both, interleaved by rank (key tile rank r, then query tile rank r, each
// for every (b, h)), heaviest first.  Neither half's last wave then leaves
// SMs idle while the other waits to start.
struct BwdBf16Launch {
    BwdBf16Params kv, q;   // key-stationary and query-stationary parameters
    int n_kv, n_q;         // 128-row tiles on each side (0: that half is absent)
    int BH;
};

template <int D>
__global__ void __launch_bounds__(bwd_threads<D>(), 1)
    attn_bwd_bf16_kernel(const __grid_constant__ BwdBf16Launch L) {
    pdl_wait();      // the stream's previous kernel has completed; its writes are visible
    pdl_trigger();   // the next kernel may be scheduled
    const int idx = (int)blockIdx.x, BH = L.BH;
    const int m = min(L.n_kv, L.n_q);
    int r, bh;
    bool kv;
    if (idx < 2 * m * BH) {
        r = idx / (2 * BH);
        kv = ((idx / BH) & 1) == 0;
        bh = idx % BH;
    } else {
        const int i2 = idx - 2 * m * BH;
        r = m + i2 / BH;
        kv = L.n_kv > L.n_q;
        bh = i2 % BH;
    }
    if (kv)
        bwd_tile<D, true>(L.kv, r, L.n_kv, bh);
    else
        bwd_tile<D, false>(L.q, r, L.n_q, bh);
}

template <int D>
cudaError_t launch_bwd_bf16_tc(const BwdBf16Launch &L, cudaStream_t stream) {
    // Shared memory requested so that the CTAs resident on one SM never ask
    // for more than its 512 TMEM columns together (an allocation would
    // otherwise wait for another CTA to finish): 512 / columns per CTA (the
    // same for both halves).
    static_assert(bwd_tmem_cols<D, true>() == bwd_tmem_cols<D, false>(), "one TMEM size");
    constexpr uint32_t per_sm = 512u / bwd_tmem_cols<D, true>();
    constexpr size_t floor_smem = (228u * 1024u) / (per_sm + 1) + 1024u;
    constexpr size_t need = BwdBf16Cfg<D, true>::kSmem > BwdBf16Cfg<D, false>::kSmem
                                ? BwdBf16Cfg<D, true>::kSmem
                                : BwdBf16Cfg<D, false>::kSmem;
    constexpr size_t smem = need > floor_smem ? need : floor_smem;
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(attn_bwd_bf16_kernel<D>), smem);
    if (e != cudaSuccess) return e;
    const uint64_t blocks = ((uint64_t)L.n_kv + (uint64_t)L.n_q) * (uint64_t)L.BH;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffull) return cudaErrorInvalidConfiguration;
    return launch_kernel(attn_bwd_bf16_kernel<D>, dim3((unsigned)blocks), dim3(bwd_threads<D>()), smem,
                         stream, nullptr, L);
}

}  // namespace

cudaError_t launch_bwd_bf16_tensor(const void *q, const void *k, const void *v, const void *dout,
                                   const float *lse, const float *delta, const int32_t *kv_lengths,
                                   void *dq, void *dk, void *dv, int B, int H, int Lq, int Lk, int D,
                                   int mask_kind, float scale, cudaStream_t stream, int *driver_err) {
    *driver_err = 0;
    const uint64_t BH = (uint64_t)B * H;
    if (BH > 0x7fffffffull) return cudaErrorInvalidConfiguration;
    BwdBf16Launch L;
    std::memset(&L, 0, sizeof(L));
    L.BH = (int)BH;
    BwdBf16Params &pk = L.kv, &pq = L.q;
    pk.lse = lse;
    pk.delta = delta;
    pk.kv_lengths = (mask_kind & 2) ? kv_lengths : nullptr;
    pk.B = B;
    pk.H = H;
    pk.Lq = Lq;
    pk.Lk = Lk;
    pk.causal = (mask_kind & 1) ? 1 : 0;
    pk.scale = scale;
    pk.scale_log2 = scale * 1.4426950408889634f;
    pq = pk;
    CUresult r = CUDA_SUCCESS;
    // Key-stationary: dK, dV (every key row written, zeros where no query sees it).
    if (Lk > 0) {
        const bool has_q = Lq > 0;
        r = encode_bf16_3d(&pk.tm_x, k, D, Lk, BH, kRowsB);
        if (r == CUDA_SUCCESS) r = encode_bf16_3d(&pk.tm_y, v, D, Lk, BH, kRowsB);
        if (r == CUDA_SUCCESS) r = encode_bf16_3d(&pk.tm_xs, has_q ? q : k, D, has_q ? Lq : Lk, BH, kColsB);
        if (r == CUDA_SUCCESS) r = encode_bf16_3d(&pk.tm_ys, has_q ? dout : v, D, has_q ? Lq : Lk, BH, kColsB);
        if (r != CUDA_SUCCESS) {
            *driver_err = (int)r;
            return cudaErrorInvalidValue;
        }
        pk.g1 = static_cast<__nv_bfloat16 *>(dk);
        pk.g2 = static_cast<__nv_bfloat16 *>(dv);
        L.n_kv = (Lk + kRowsB - 1) / kRowsB;
    }
    // Query-stationary: dQ.
    if (Lq > 0) {
        const bool has_k = Lk > 0;
        // Q and dout go to TMEM row by row (plain loads); K and V stream by TMA.
        pq.xa = static_cast<const __nv_bfloat16 *>(q);
        pq.ya = static_cast<const __nv_bfloat16 *>(dout);
        r = encode_bf16_3d(&pq.tm_xs, has_k ? k : q, D, has_k ? Lk : Lq, BH, kColsB);
        if (r == CUDA_SUCCESS) r = encode_bf16_3d(&pq.tm_ys, has_k ? v : dout, D, has_k ? Lk : Lq, BH, kColsB);
        if (r != CUDA_SUCCESS) {
            *driver_err = (int)r;
            return cudaErrorInvalidValue;
        }
        pq.g1 = static_cast<__nv_bfloat16 *>(dq);
        pq.g2 = nullptr;
        L.n_q = (Lq + kRowsB - 1) / kRowsB;
    }
    const cudaError_t e = D == 64 ? launch_bwd_bf16_tc<64>(L, stream) : launch_bwd_bf16_tc<128>(L, stream);
    return e;
}

cudaError_t status_ctl_bwd_bf16(int op, uint64_t value, uint32_t *bits) {
    return unit_status_ctl(op, value, bits);
}

}  // namespace mha
