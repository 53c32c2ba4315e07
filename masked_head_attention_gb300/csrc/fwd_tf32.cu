// fwd_tf32.cu -- fused masked multi-head attention forward for fp32 inputs on
// the sm_103a tensor cores, at fp32-level accuracy through a three-term TF32
// split: every fp32 operand x is written as
//     x = hi + lo,   hi = x truncated to tf32,   lo = x - hi
// (tf32 keeps 10 explicit mantissa bits; x - hi is exact in fp32; the tensor
// core itself truncates an fp32 word to tf32, so x is passed as hi and lo's
// low bits are dropped below 2^-20 |x|), and each product as
//     a b ~= a_hi b_hi + a_lo b_hi + a_hi b_lo
// where the dropped a_lo b_lo is below 2^-20 |a b|.  S = Q K^T and O += P V
// are each three tcgen05 kind::tf32 MMAs per K-step, accumulating in fp32 in
// TMEM.  The softmax is the same online form as the other kernels.
//
// Head dimension 64.  Work item = one 128-row query tile of one (b, h); key
// tiles of 64.  CTA = 10 warps, persistent over items (one CTA per SM):
//   warps 0-3  softmax: thread t owns query row t (TMEM lane t).  It loads
//              its S row (64 keys) from TMEM, masks it from (row, col,
//              length), keeps the running max and rescaled running sum, and
//              writes P as tf32 hi over its S columns and tf32 lo into a
//              column block of its own.  At the end it divides its O row by
//              the row sum and stores it (and the row's log-sum-exp when
//              asked).
//   warps 4-7  converters: the Q tile's rows, times scale * log2(e), into
//              hi / lo TMEM columns (the A operand of S, read from TMEM, so S
//              arrives in the base-2 domain); each K tile's lo beside it in
//              shared memory (the raw tile is its hi); each V tile into
//              transposed hi / lo tiles (the B operand of P V, K-major: row =
//              feature, 64 keys along the row), so every MMA operand is
//              K-major.
//   warp 8     TMA producer: the Q tile per item, K and V tiles of 64 keys
//              through two stages; key tiles past the causal limit or the
//              valid length are never loaded.
//   warp 9     MMA issuer (elected lane) and TMEM owner.  Per item:
//                  S(0), S(1), PV(0), S(2), PV(1), ..., PV(n-1)
//              so the softmax of tile j overlaps S(j+1) and the P V of the
//              previous tile.
// TMEM columns: Q hi 0-63, Q lo 64-127, S/P-hi buffers 128-191 and 192-255,
// P-lo buffers 256-319 and 320-383, O 384-447.
// All hand-offs are mbarriers; every wait is bounded.
//
// Page sections this follows: "Why attention must compute the max first"
// (gsyq.cn) 2.3-2.4 and 3.1 (online softmax with the max shift, fused between
// QK^T and PV, scores kept on chip); "masked multi head attention" CUDA
// article (2kiu.com) 2 and 3.1 (skip fully masked tiles, mask in-kernel as
// -infinity before the softmax).
#include <cstdint>
#include <cstring>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kD = 64;                 // head dimension of this kernel
constexpr int kRows = 128;             // query rows per item
constexpr int kKeys = 64;              // keys per key tile
constexpr int kThreads = 320;
constexpr int kConvWarp0 = 4;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQh = 0, kColQl = 64, kColS = 128, kColPl = 256, kColO = 384;
constexpr float kRescaleThreshold = 8.0f;   // P stays <= 256 between rescales

// Shared memory (offsets from a 1024-byte aligned base).  A "box" is one
// TMA box of 32 fp32 columns (128 bytes per row, 128-byte swizzle).
constexpr uint32_t kQBox = kRows * 128;             // 16 KB: 128 rows x 32 columns
constexpr uint32_t kKBox = kKeys * 128;             // 8 KB: 64 rows x 32 columns
constexpr uint32_t kQ = 0;                          // raw Q tile: 2 boxes
constexpr uint32_t kStage0 = 2 * kQBox;
constexpr uint32_t kKh = 0;                         // K raw, then hi in place: 2 boxes
constexpr uint32_t kKl = 2 * kKBox;                 // K lo
constexpr uint32_t kVr = 4 * kKBox;                 // V raw
constexpr uint32_t kVh = 6 * kKBox;                 // V^T hi: 2 halves of [64 features][32 keys]
constexpr uint32_t kVl = 8 * kKBox;                 // V^T lo
constexpr uint32_t kStageBytes = 10 * kKBox;        // 80 KB
// O staging for the TMA-store epilogue: per softmax warp two boxes of 32
// rows x 32 columns (4 KB each).
constexpr uint32_t kOBox = 32 * 128;
constexpr uint32_t kO = kStage0 + 2 * kStageBytes;
constexpr uint32_t kBarsOff = kO + 4 * 2 * kOBox;
// Batches ordered by visible length (longest first) for the item order,
// when the kv-length mask is on and B is at most this.
constexpr int kMaxSortB = 128;

struct Tf32Params {
    CUtensorMap tm_q;     // Q [B*H][Lq][64] fp32, box {32, 128, 1}
    CUtensorMap tm_k;     // K [B*H][Lk][64], box {32, 64, 1}
    CUtensorMap tm_v;     // V [B*H][Lk][64], box {32, 64, 1}
    CUtensorMap tm_o;     // O [B*H][Lq][64], box {32, 32, 1} (one warp's rows)
    float *out;           // [B*H][Lq][64]
    float *lse;           // [B*H][Lq] or null
    const int32_t *kv_lengths;   // null unless the kv-length mask is on
    int B, H, Lq, Lk;
    int causal;
    float scale_log2;
    int n_qt;             // 128-row query tiles per (b, h)
    int n_items;          // B * H * n_qt
};

struct __align__(8) Bars {
    uint64_t q_raw, q_raw_free, q_ready, q_free;
    uint64_t k_raw[2], k_ready[2], k_empty[2];
    uint64_t v_raw[2], v_ready[2], v_empty[2];
    uint64_t s_full[2], p_full[2], pv_done, o_full, o_free;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int sorted;               // batch order below is in use
    int ord[kMaxSortB];       // batch at length rank r
    int len[kMaxSortB];       // clamped visible length of batch b
};

constexpr size_t kSmem = 1024 + kBarsOff + sizeof(Bars);
static_assert(kSmem <= 232448, "shared memory over the per-block limit");

struct Item {
    int b, bh, q0;
    int len;   // visible keys of batch b (clamped)
    int n;     // key tiles of 64 the query tile visits
};

// Item order, heaviest first.  With kv lengths (and B <= kMaxSortB): batches
// by visible length, longest first, then latest query tiles, then heads.
// Otherwise latest (for causal masks the heaviest) query tiles first, (b, h)
// fastest.
__device__ __forceinline__ Item decode_item(const Tf32Params &p, const Bars *bars, int item) {
    Item it;
    int len = p.Lk;
    if (bars->sorted) {
        const int per_b = p.n_qt * p.H;
        const int r = item / per_b, rem = item - r * per_b;
        const int qt = p.n_qt - 1 - rem / p.H;
        it.b = bars->ord[r];
        it.bh = it.b * p.H + rem % p.H;
        it.q0 = qt * kRows;
        len = bars->len[it.b];
    } else {
        const int BH = p.B * p.H;
        const int qt = p.n_qt - 1 - item / BH;
        it.bh = item % BH;
        it.b = it.bh / p.H;
        it.q0 = qt * kRows;
        if (p.kv_lengths) len = max(0, min((int)p.kv_lengths[it.b], p.Lk));
    }
    it.len = len;
    int kend = len;
    if (p.causal) kend = min(kend, it.q0 + kRows);
    it.n = (kend + kKeys - 1) / kKeys;
    return it;
}

// Persistent walk: rounds of gridDim.x items, forward in even rounds and
// backward in odd ones.
struct ItemIter {
    int r = 0, idx = -1;
    __device__ __forceinline__ bool next(int n_items) {
        const int G = gridDim.x, c = blockIdx.x;
        for (;;) {
            if ((long long)r * G >= n_items) return false;
            idx = (r & 1) ? (r + 1) * G - 1 - c : r * G + c;
            ++r;
            if (idx < n_items) return true;
        }
    }
};

// Byte offset of element (row, col) (col < 32) inside one 128-byte-swizzled box.
__device__ __forceinline__ uint32_t box_off(int row, int col) {
    return (uint32_t)(row * 128 + ((((col >> 2) ^ (row & 7)) & 7) << 4) + (col & 3) * 4);
}

// x = hi + lo with hi = x's top 11 significant bits (its low 13 mantissa
// bits cleared: a tf32 value) and lo = x - hi, exact in fp32 (x and hi share
// their exponent and top bits).  The tensor core reads a tf32 operand from an
// fp32 word by ignoring its low 13 mantissa bits -- measured on GB300 for
// operands in shared memory and in TMEM: 8192 of 8192 products of random fp32
// values equal the products of their truncations -- so x itself is passed as
// hi, and lo's own bits beyond 11 are dropped by the same rule: |lo| < 2^-10
// |x|, so that costs below 2^-20 |x|.  Done on pairs: two bit masks and one
// packed fp32x2 FMA (x - hi formed as fma(hi, -1, x), one exact rounding).
// The _rn intrinsic is never contracted into other FMAs.
__device__ __forceinline__ void split_tf32x2(float2 v, uint32_t &hi0, uint32_t &hi1, uint32_t &lo0,
                                             uint32_t &lo1) {
    hi0 = __float_as_uint(v.x);
    hi1 = __float_as_uint(v.y);
    const float2 h = make_float2(__uint_as_float(hi0 & 0xFFFFE000u), __uint_as_float(hi1 & 0xFFFFE000u));
    const float2 l = __ffma2_rn(h, make_float2(-1.f, -1.f), v);   // v - hi, exact
    lo0 = __float_as_uint(l.x);
    lo1 = __float_as_uint(l.y);
}

__device__ __forceinline__ float row_lse2(float m2, float l) {
    if (m2 == -INFINITY || !(l > 0.f)) return -INFINITY;
    return 0.69314718055994531f * (m2 + log2f(l));
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tf32x3_kernel(const __grid_constant__ Tf32Params p) {
    pdl_wait();      // the stream's previous kernel has completed; its writes are visible
    pdl_trigger();   // the next kernel may be scheduled
    if (wait_expired_before()) return;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *base = smem_raw + pad;
    Bars *bars = reinterpret_cast<Bars *>(base + kBarsOff);
    volatile int *abort = &bars->abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_raw, 1);
        mbar_init(&bars->q_raw_free, 4);   // one arrival per converter warp
        mbar_init(&bars->q_ready, 4);
        mbar_init(&bars->q_free, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->k_raw[s], 1);
            mbar_init(&bars->k_ready[s], 4);
            mbar_init(&bars->k_empty[s], 1);
            mbar_init(&bars->v_raw[s], 1);
            mbar_init(&bars->v_ready[s], 4);
            mbar_init(&bars->v_empty[s], 1);
            mbar_init(&bars->s_full[s], 1);
            mbar_init(&bars->p_full[s], 4);   // one arrival per softmax warp
        }
        mbar_init(&bars->pv_done, 1);
        mbar_init(&bars->o_full, 1);
        mbar_init(&bars->o_free, 4);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        mbar_fence_init();
    }
    // Batch order by visible length (rank = number of batches before it).
    const bool sorted = p.kv_lengths != nullptr && p.B > 1 && p.B <= kMaxSortB;
    if (threadIdx.x == 0) bars->sorted = sorted ? 1 : 0;
    if (sorted) {
        for (int b = threadIdx.x; b < p.B; b += kThreads)
            bars->len[b] = max(0, min((int)p.kv_lengths[b], p.Lk));
        __syncthreads();
        for (int b = threadIdx.x; b < p.B; b += kThreads) {
            const int lb = bars->len[b];
            int rank = 0;
            for (int u = 0; u < p.B; ++u) {
                const int lu = bars->len[u];
                rank += (lu > lb || (lu == lb && u < b)) ? 1 : 0;
            }
            bars->ord[rank] = b;
        }
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&p.tm_q);
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

    // Warp-uniform bounded wait (a warp-collective tcgen05 op may follow).
    auto wwait = [&](uint64_t *bar, uint32_t parity, uint32_t site) -> bool {
        const bool r = mbar_wait(bar, parity, site, abort);
        return __all_sync(0xffffffffu, r);
    };

    if (warp == kProducerWarp) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            uint32_t g = 0, k = 0;
            uint32_t gk = 0, gv = 0;   // K / V tiles whose loads were issued
            int q_pending = -1;
            bool ok = true;
            ItemIter iter;
            while (ok && iter.next(p.n_items)) {
                const Item it = decode_item(p, bars, iter.idx);
                if (it.n == 0) continue;
                if (k > 0) ok = mbar_wait(&bars->q_raw_free, (k - 1) & 1, kSiteQEmpty, abort);
                if (!ok) break;
                mbar_arrive_expect_tx(&bars->q_raw, 2 * kQBox);
                for (int hh = 0; hh < 2; ++hh)
                    tma_load_3d(base + kQ + hh * kQBox, &p.tm_q, &bars->q_raw, hh * 32, it.q0, it.bh);
                q_pending = (int)(k & 1);
                for (int j = 0; ok && j < it.n; ++j) {
                    const uint32_t st = g & 1;
                    uint8_t *stage = base + kStage0 + st * kStageBytes;
                    if (g >= 2) ok = mbar_wait(&bars->k_empty[st], ((g >> 1) - 1) & 1, kSiteKvEmpty, abort);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&bars->k_raw[st], 2 * kKBox);
                    for (int hh = 0; hh < 2; ++hh)
                        tma_load_3d(stage + kKh + hh * kKBox, &p.tm_k, &bars->k_raw[st], hh * 32,
                                    j * kKeys, it.bh);
                    ++gk;
                    if (g >= 2) ok = mbar_wait(&bars->v_empty[st], ((g >> 1) - 1) & 1, kSiteKvEmpty, abort);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&bars->v_raw[st], 2 * kKBox);
                    for (int hh = 0; hh < 2; ++hh)
                        tma_load_3d(stage + kVr + hh * kKBox, &p.tm_v, &bars->v_raw[st], hh * 32,
                                    j * kKeys, it.bh);
                    ++gv;
                    ++g;
                }
                ++k;
            }
            if (!ok) {
                // Let the loads already issued land before shared memory is released.
                volatile int no_abort = 0;
                for (uint32_t gg = (gk >= 2u ? gk - 2 : 0); gg < gk; ++gg)
                    mbar_wait(&bars->k_raw[gg & 1], (gg >> 1) & 1, kSiteDrain, &no_abort);
                for (uint32_t gg = (gv >= 2u ? gv - 2 : 0); gg < gv; ++gg)
                    mbar_wait(&bars->v_raw[gg & 1], (gg >> 1) & 1, kSiteDrain, &no_abort);
                if (q_pending >= 0)
                    mbar_wait(&bars->q_raw, (uint32_t)q_pending, kSiteDrain, &no_abort);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------- MMA issuer -------------------------------
        constexpr uint32_t idS = idesc_tf32_f32(128, kKeys);   // S: N = 64 keys
        constexpr uint32_t idPV = idesc_tf32_f32(128, kD);     // O: N = 64 features
        const uint64_t d0 = sdesc_sw128(smem_u32(base + kStage0), 16, 1024);
        const uint32_t dlo = (uint32_t)d0, dhi = (uint32_t)(d0 >> 32);
        constexpr uint32_t kStageU = kStageBytes >> 4, kBoxU = kKBox >> 4;
        uint32_t g = 0, k = 0;
        bool ok = true;
        bool issued = false;
        // Under a test's short wait limit: a wait that must expire (the drain
        // phase completes only at teardown).
        if (wait_limit_is_test()) ok = wwait(&bars->drain, 0, kSiteTest);
        // Three MMAs per K-step (hi.hi, lo.hi, hi.lo) into `dcol`; A from TMEM
        // columns a_hi / a_lo (8 columns per K-step), B from the K-major tiles
        // b_hi / b_lo (descriptor low words; 64 rows, two 128-byte halves).
        // The whole (converged) warp walks the fully unrolled sequence and one
        // elected lane -- the same lane every time -- issues each MMA (elect
        // and MMA in one predicated block, about five instructions per MMA:
        // this warp shares its scheduler with a softmax and a converter warp,
        // and a 128 x 64 x 8 MMA retires every 32 cycles).
        auto mma3 = [&](uint32_t dcol, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo,
                        uint32_t idesc, bool fresh) {
            const uint32_t d = tmem + dcol, ah = tmem + a_hi, al = tmem + a_lo;
#pragma unroll
            for (int ps = 0; ps < 3; ++ps) {
                const uint32_t a = ps == 1 ? al : ah;
                const uint32_t b = ps == 2 ? b_lo : b_hi;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (uint32_t)((kk >> 2) * kBoxU + (kk & 3) * 2);
                    umma_ts_tf32_elect(d, a + kk * 8, b + off, dhi, idesc,
                                       (ps == 0 && kk == 0) ? (fresh ? 0u : 1u) : 1u);
                }
            }
        };
        ItemIter iter;
        while (ok && iter.next(p.n_items)) {
            const Item it = decode_item(p, bars, iter.idx);
            if (it.n == 0) continue;
            ok = wwait(&bars->q_ready, k & 1, kSiteQFull);
            // Issue order S(0), S(1), PV(0), S(2), PV(1), ...: S(j) goes out once
            // PV(j - 2) has, so the S/P buffer it overwrites is free by the
            // in-order execution of the tensor pipe.
            int js = 0, jp = 0;
            while (ok && jp < it.n) {
                const bool do_s = js < it.n && js <= jp + 1;
                const int j = do_s ? js : jp;
                const uint32_t gg = g + j, st = gg & 1;
                const uint32_t sb = dlo + st * kStageU;
                if (do_s) {
                    ok = wwait(&bars->k_ready[st], (gg >> 1) & 1, kSiteKFull);
                    if (!ok) break;
                    tc_fence_after();
                    mma3(kColS + (gg & 1) * 64, kColQh, kColQl, sb + (kKh >> 4), sb + (kKl >> 4), idS,
                         true);
                    if (elect_one()) {
                        umma_commit(&bars->s_full[gg & 1]);
                        umma_commit(&bars->k_empty[st]);
                        if (j == it.n - 1) umma_commit(&bars->q_free);
                    }
                    __syncwarp();
                    ++js;
                } else {
                    ok = wwait(&bars->v_ready[st], (gg >> 1) & 1, kSiteVFull);
                    if (ok && j == 0 && k > 0) ok = wwait(&bars->o_free, (k - 1) & 1, kSiteOFree);
                    if (ok) ok = wwait(&bars->p_full[gg & 1], (gg >> 1) & 1, kSitePFull);
                    if (!ok) break;
                    tc_fence_after();
                    mma3(kColO, kColS + (gg & 1) * 64, kColPl + (gg & 1) * 64, sb + (kVh >> 4),
                         sb + (kVl >> 4), idPV, j == 0);
                    if (elect_one()) {
                        umma_commit(&bars->pv_done);
                        umma_commit(&bars->v_empty[st]);
                        if (j == it.n - 1) umma_commit(&bars->o_full);
                    }
                    __syncwarp();
                    ++jp;
                }
                issued = true;
            }
            g += it.n;
            ++k;
        }
        if (issued) {
            // Every MMA must have finished before TMEM is released.
            volatile int no_abort = 0;
            if (elect_one()) umma_commit(&bars->drain);
            __syncwarp();
            mbar_wait(&bars->drain, 0, kSiteDrain, &no_abort);
            __syncwarp();
        }
    } else if (warp >= kConvWarp0) {
        // ------------------------------- converters -------------------------------
        const int c = threadIdx.x - 32 * kConvWarp0;   // 0..127: Q row / TMEM lane
        const int cw = c >> 5;
        const uint32_t lane_off = (uint32_t)(cw * 32) << 16;
        uint32_t g = 0, k = 0;
        bool ok = true;
        ItemIter iter;
        while (ok && iter.next(p.n_items)) {
            const Item it = decode_item(p, bars, iter.idx);
            if (it.n == 0) continue;
            ok = wwait(&bars->q_raw, k & 1, kSiteQFull);
            if (ok && k > 0) ok = wwait(&bars->q_free, (k - 1) & 1, kSiteQEmpty);
            if (!ok) break;
            {
                // Row c of Q -> hi into TMEM columns 0-63, lo into 64-127.
                uint32_t hi[64], lo[64];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const float4 x = *reinterpret_cast<const float4 *>(
                            base + kQ + hh * kQBox + box_off(c, ch * 4));
                        const int e = hh * 32 + ch * 4;
                        // The logit scale (times log2 e) is folded into Q here,
                        // so S arrives in the base-2 domain.
                        const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
                        split_tf32x2(__fmul2_rn(make_float2(x.x, x.y), c2), hi[e], hi[e + 1], lo[e],
                                     lo[e + 1]);
                        split_tf32x2(__fmul2_rn(make_float2(x.z, x.w), c2), hi[e + 2], hi[e + 3],
                                     lo[e + 2], lo[e + 3]);
                    }
                tmem_st64(tmem + lane_off + kColQh, hi);
                tmem_st64(tmem + lane_off + kColQl, lo);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars->q_ready);
                    mbar_arrive(&bars->q_raw_free);
                }
            }
            for (int j = 0; ok && j < it.n; ++j) {
                const uint32_t st = g & 1;
                uint8_t *stage = base + kStage0 + st * kStageBytes;
                // K: the raw tile serves as hi in place; lo beside it (same
                // swizzled positions).
                ok = wwait(&bars->k_raw[st], (g >> 1) & 1, kSiteKFull);
                if (!ok) break;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 *ph = reinterpret_cast<const float4 *>(stage + kKh) + c + 128 * i;
                    float4 *pl = reinterpret_cast<float4 *>(stage + kKl) + c + 128 * i;
                    const float4 x = *ph;
                    uint4 h, l;
                    split_tf32x2(make_float2(x.x, x.y), h.x, h.y, l.x, l.y);
                    split_tf32x2(make_float2(x.z, x.w), h.z, h.w, l.z, l.w);
                    *reinterpret_cast<uint4 *>(pl) = l;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->k_ready[st]);
                // V: thread (feature d, key half kh) reads 32 keys of column d
                // and writes row d of the transposed hi / lo halves kh.
                ok = wwait(&bars->v_raw[st], (g >> 1) & 1, kSiteVFull);
                if (!ok) break;
                {
                    const int d = (cw & 1) * 32 + lane, kh = cw >> 1;
                    const uint8_t *vbox = stage + kVr + (cw & 1) * kKBox;
                    uint32_t hi[32], lo[32];
#pragma unroll
                    for (int kk = 0; kk < 32; kk += 2) {
                        const float x0 =
                            *reinterpret_cast<const float *>(vbox + box_off(kh * 32 + kk, lane));
                        const float x1 =
                            *reinterpret_cast<const float *>(vbox + box_off(kh * 32 + kk + 1, lane));
                        split_tf32x2(make_float2(x0, x1), hi[kk], hi[kk + 1], lo[kk], lo[kk + 1]);
                    }
                    uint8_t *th = stage + kVh + kh * kKBox;
                    uint8_t *tl = stage + kVl + kh * kKBox;
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const uint32_t o = box_off(d, cc * 4);
                        *reinterpret_cast<uint4 *>(th + o) =
                            make_uint4(hi[4 * cc], hi[4 * cc + 1], hi[4 * cc + 2], hi[4 * cc + 3]);
                        *reinterpret_cast<uint4 *>(tl + o) =
                            make_uint4(lo[4 * cc], lo[4 * cc + 1], lo[4 * cc + 2], lo[4 * cc + 3]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->v_ready[st]);
                ++g;
            }
            ++k;
        }
    } else {
        // --------------------------------- softmax --------------------------------
        const int t = threadIdx.x;   // query row within the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        uint8_t *stg = base + kO + warp * 2 * kOBox;   // this warp's 32 x 64 O staging
        uint32_t g = 0, k = 0;
        bool ok = true;
        // Row (lane) of this warp's 32-row slice, scaled by `inv`, into the
        // staging boxes, then one TMA store per box (rows past Lq clipped).
        auto store_rows = [&](const Item &it, const uint32_t (&o)[64], float inv) {
            if (lane == 0) tma_store_wait_read();   // the previous store has read the staging
            __syncwarp();
            // The row's elements are summed on the side: a NaN or infinite
            // element makes the sum non-finite (|O| <= max |V|, so finite rows
            // cannot overflow it).
            float2 rsum = make_float2(0.f, 0.f);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const int e = hh * 32 + ch * 4;
                    const float4 v4 =
                        make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                                    __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                    rsum = __fadd2_rn(rsum, __fadd2_rn(make_float2(v4.x, v4.y), make_float2(v4.z, v4.w)));
                    *reinterpret_cast<float4 *>(stg + hh * kOBox + box_off(lane, ch * 4)) = v4;
                }
            report_flag(!finite_f(rsum.x + rsum.y) && it.q0 + warp * 32 + lane < p.Lq, kFlagNonFinite);
            fence_proxy_async_smem();
            __syncwarp();
            const int r0 = it.q0 + warp * 32;
            if (lane == 0 && r0 < p.Lq) {
                tma_store_3d(&p.tm_o, stg, 0, r0, it.bh);
                tma_store_3d(&p.tm_o, stg + kOBox, 32, r0, it.bh);
                tma_store_commit();
            }
        };
        ItemIter iter;
        while (ok && iter.next(p.n_items)) {
            const Item it = decode_item(p, bars, iter.idx);
            const int row = it.q0 + t;
            if (it.n == 0) {
                // No visible key: zeros (and -inf log-sum-exp).
                uint32_t z[64];
#pragma unroll
                for (int e = 0; e < 64; ++e) z[e] = 0u;
                store_rows(it, z, 0.f);
                if (p.lse && row < p.Lq) p.lse[(size_t)it.bh * p.Lq + row] = -INFINITY;
                continue;
            }
            const int vis_end = p.causal ? min(it.len, row + 1) : it.len;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; ok && j < it.n; ++j) {
                const uint32_t gg = g + j;
                const uint32_t colS = kColS + (gg & 1) * 64;
                ok = wwait(&bars->s_full[gg & 1], (gg >> 1) & 1, kSiteSFull);
                if (!ok) break;
                tc_fence_after();
                uint32_t r[64];
                tmem_ld64(tmem + lane_off + colS, r);
                const int k0 = j * kKeys;
                const bool edge = (k0 + kKeys > it.len) || (p.causal && k0 + kKeys - 1 > it.q0);
                float x[64];
                float mx[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    float v = __uint_as_float(r[e]);
                    if (edge && k0 + e >= vis_end) v = -INFINITY;
                    x[e] = v;
                }
#pragma unroll
                for (int e = 0; e < 64; e += 8) {
#pragma unroll
                    for (int u = 0; u < 8; u += 2) mx[u >> 1] = max3f(mx[u >> 1], x[e + u], x[e + u + 1]);
                }
                const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                const float m_new = fmaxf(m, mt);
                // Rescale O and l only when the max grew by more than the
                // threshold and O already holds a contribution (l > 0).
                const bool need = j > 0 && l > 0.f && m_new > m + kRescaleThreshold;
                if (__any_sync(0xffffffffu, need)) {
                    ok = wwait(&bars->pv_done, (gg - 1) & 1, kSitePvDone);
                    if (!ok) break;
                    tc_fence_after();
                    const float alpha = need ? ex2_approx(m - m_new) : 1.f;
                    uint32_t o[64];
                    tmem_ld64(tmem + lane_off + kColO, o);
#pragma unroll
                    for (int e = 0; e < 64; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st64(tmem + lane_off + kColO, o);
                    if (need) l *= alpha;
                }
                if (j == 0 || l == 0.f || m_new > m + kRescaleThreshold) m = m_new;
                const float msub = (m == -INFINITY) ? 0.f : m;
                const float2 negm = make_float2(-msub, -msub);
                float2 rs0 = make_float2(0.f, 0.f), rs1 = make_float2(0.f, 0.f);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    // P = 2^(x - m) for 32 keys, split into tf32 hi (over the S
                    // columns) and lo (the P-lo buffer).
                    uint32_t hi[32], lo[32];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const int f = half * 32 + e;
                        const float2 d0 = __fadd2_rn(make_float2(x[f], x[f + 1]), negm);
                        const float2 d1 = __fadd2_rn(make_float2(x[f + 2], x[f + 3]), negm);
                        const float2 p01 = make_float2(ex2_approx(d0.x), ex2_approx(d0.y));
                        const float2 p23 = make_float2(ex2_approx(d1.x), ex2_approx(d1.y));
                        rs0 = __fadd2_rn(rs0, p01);
                        rs1 = __fadd2_rn(rs1, p23);
                        split_tf32x2(p01, hi[e], hi[e + 1], lo[e], lo[e + 1]);
                        split_tf32x2(p23, hi[e + 2], hi[e + 3], lo[e + 2], lo[e + 3]);
                    }
                    tmem_st32(tmem + lane_off + colS + half * 32, hi);
                    tmem_st32(tmem + lane_off + kColPl + (gg & 1) * 64 + half * 32, lo);
                }
                l += (rs0.x + rs0.y) + (rs1.x + rs1.y);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_full[gg & 1]);
            }
            if (!ok) break;
            // Epilogue: O / l (zeros for a row that saw no visible key).
            ok = wwait(&bars->o_full, k & 1, kSiteQFull);
            if (!ok) break;
            tc_fence_after();
            uint32_t o[64];
            tmem_ld64(tmem + lane_off + kColO, o);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->o_free);
            const float inv = l > 0.f ? 1.f / l : 0.f;
            // The sum is 0 for a row with no visible key and at least 1
            // otherwise, unless an input was not finite.
            report_flag(row < p.Lq && !finite_f(l), kFlagSum);
            store_rows(it, o, inv);
            if (p.lse && row < p.Lq) p.lse[(size_t)it.bh * p.Lq + row] = row_lse2(m, l);
            g += it.n;
            ++k;
        }
        // Output stores must finish before the CTA's shared memory is released.
        if (lane == 0) tma_store_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// 3-D fp32 tensor map over a dense [d2][d1][64] array with a {32, box_rows, 1}
// box and the 128-byte swizzle; rows outside the array read as zero.
CUresult encode_f32_3d(CUtensorMap *map, const void *ptr, uint64_t d1, uint64_t d2,
                       uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return CUDA_ERROR_NOT_SUPPORTED;
    const cuuint64_t dims[3] = {(cuuint64_t)kD, d1, d2};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * 4, (cuuint64_t)kD * d1 * 4};
    const cuuint32_t box[3] = {32, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(ptr), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

bool tf32x3_applies(int D) { return D == kD; }

cudaError_t launch_fwd_tf32x3(const float *q, const float *k, const float *v,
                              const int32_t *kv_lengths, float *out, float *lse, int B, int H,
                              int Lq, int Lk, int D, int mask_kind, float scale,
                              cudaStream_t stream, int *driver_err) {
    *driver_err = 0;
    if (D != kD) return cudaErrorInvalidValue;
    Tf32Params p;
    std::memset(&p, 0, sizeof(p));
    const uint64_t BH = (uint64_t)B * H;
    CUresult r = encode_f32_3d(&p.tm_q, q, Lq, BH, kRows);
    const bool has_k = Lk > 0;
    if (r == CUDA_SUCCESS)
        r = encode_f32_3d(&p.tm_k, has_k ? (const void *)k : (const void *)q, has_k ? Lk : Lq, BH, kKeys);
    if (r == CUDA_SUCCESS)
        r = encode_f32_3d(&p.tm_v, has_k ? (const void *)v : (const void *)q, has_k ? Lk : Lq, BH, kKeys);
    if (r == CUDA_SUCCESS) r = encode_f32_3d(&p.tm_o, out, Lq, BH, 32);
    if (r != CUDA_SUCCESS) {
        *driver_err = (int)r;
        return cudaErrorInvalidValue;
    }
    p.out = out;
    p.lse = lse;
    p.kv_lengths = (mask_kind & 2) ? kv_lengths : nullptr;
    p.B = B;
    p.H = H;
    p.Lq = Lq;
    p.Lk = Lk;
    p.causal = (mask_kind & 1) ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.n_qt = (Lq + kRows - 1) / kRows;
    p.n_items = (int)(BH * (uint64_t)p.n_qt);
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(attn_fwd_tf32x3_kernel), kSmem);
    if (e != cudaSuccess) return e;
    int grid = device_info().sms;
    if (grid > p.n_items) grid = p.n_items;
    if (grid < 1) return cudaSuccess;
    return launch_kernel(attn_fwd_tf32x3_kernel, dim3(grid), dim3(kThreads), kSmem, stream, nullptr,
                         p);
}

cudaError_t status_ctl_fwd_tf32(int op, uint64_t value, uint32_t *bits) {
    return unit_status_ctl(op, value, bits);
}

}  // namespace mha
