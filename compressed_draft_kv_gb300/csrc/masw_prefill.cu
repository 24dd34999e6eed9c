// Draft prefill under the structured write mask ([EN] §3.3 Algorithm 2
// with the mask of §3.2 Algorithm 1): one layer of attention over a whole
// prefix of T raw tokens with the M = m(T) memory-slot tokens interleaved, then
// the resulting memory M_0 is stored in the pool.
//
// Query rows: raw token i (1-based) reads the sink, raw tokens of its window
// [max(S+1, i-W+1), i], and the slots materialised before it (tau_m < i); slot
// token g_m reads the sink, the window at tau_m and slots 1..m-1.  Key rows come
// from the caller's raw and slot K/V arrays ([T, Hkv, D], [M, Hkv, D]).  For one
// tile of query rows the visible keys are a few contiguous ranges (sink, window
// band, slot prefix), and for one row each range is a single interval, so the
// mask of a 64-key block is one or two intervals of columns (a bit mask per
// row, skipped for blocks every row sees whole).  With S <= 8 the sink and a
// slot prefix of up to 56 slots share one block.
//
// Query tiles cover the T + M rows in that interleaved order (slot token g_m
// right after raw token tau_m): a slot row has the mask of raw row tau_m, so it
// shares that tile's key ranges.
//
// Fifth-generation tensor cores, one CTA per (128-row query tile, query head),
// two CTAs per SM:
//   * the four softmax warps load their rows of Q once and store them in tensor
//     memory, where S = Q K^T reads them as the A operand (no shared-memory
//     re-reads of Q);
//   * lane 0 of a fifth warp issues TMA tiled loads (128-byte swizzle) of K
//     blocks of 64 keys into three stages, two blocks ahead, and S = Q K^T
//     (tcgen05.mma, M = 128, N = 64, accumulator in tensor memory); lane 0 of a
//     sixth warp does the same for V and O += P V (M = 128, N = 128, V read
//     MN-major).  Two issuing threads keep both MMA streams moving: a single
//     thread spends most of its time on MMA issue and commit round trips;
//   * thread t of the softmax warps owns query row t (TMEM lane t): it reads its
//     64 scores with tcgen05.ld, applies the mask and the online softmax, and
//     writes its row of P (bf16) into shared memory in the swizzled K-major
//     layout the PV MMA reads;
//   * the running max only moves when a row's maximum grows by more than 2^8,
//     so the O rescale (tcgen05.ld / st of the row) is rare; the final
//     normalisation uses the same max, so the result is exact;
//   * the roles hand off through mbarriers (S done, S read, P written, PV done),
//     every wait is bounded and one timed-out wait stops the CTA and the grid.
// 112 KB of shared memory and 256 TMEM columns (O, S, Q) per CTA.
#include "masw_internal.cuh"
#include "masw_tc.cuh"

#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

namespace masw {

namespace tcp {

using namespace tc;

constexpr int kBM = 128;                         // query rows per CTA = TMEM lanes
constexpr int kBN = 64;                          // keys per block
constexpr int kD = 128;                          // head_dim
constexpr int kStages = 3;                       // K and V stages
constexpr uint32_t kKVBytes = kBN * kD * 2;      // 2 panels of 64 rows x 128 B
constexpr uint32_t kPBytes = kBM * kBN * 2;      // 1 panel of 128 rows x 128 B
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kStages * kKVBytes;
constexpr uint32_t kOffP = kOffV + kStages * kKVBytes;
constexpr uint32_t kOffBar = kOffP + kPBytes;    // mbarriers, the TMEM address, an abort flag
constexpr uint32_t kSmem = kOffBar + 160;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 0;                    // O: columns [0, 128)
constexpr uint32_t kColS = 128;                  // S: columns [128, 192)
constexpr uint32_t kColQ = 192;                  // Q (bf16 pairs, the A operand of S): [192, 256)
// instruction descriptors (kind::f16): f32 accumulator, bf16 A and B, M = 128;
// S: N = 64, A (Q, tensor memory) and B (K) K-major; O: N = 128, B (V) MN-major
constexpr uint32_t kIdescBase = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBM >> 4) << 24);
constexpr uint32_t kIdescS = kIdescBase | ((uint32_t)(kBN >> 3) << 17);
constexpr uint32_t kIdescO = kIdescBase | (1u << 16) | ((uint32_t)(kD >> 3) << 17);

}  // namespace tcp

struct PrefillParams {
    CUtensorMap tm_k_raw;    // [T][Hkv][128] bf16, box 64 x 1 x 64
    CUtensorMap tm_v_raw;
    CUtensorMap tm_k_slot;   // [M][Hkv][128]
    CUtensorMap tm_v_slot;
    CUtensorMap tm_k_sink;   // raw K/V, box 8 x 1 x 64: the first 8 rows of a merged sink + slot block
    CUtensorMap tm_v_sink;
    CUtensorMap tm_k_slot56; // slot K/V, box 56 x 1 x 64: its other 56 rows
    CUtensorMap tm_v_slot56;
    const __nv_bfloat16* q_raw;    // [T][Hq][128]
    const __nv_bfloat16* q_slot;   // [M][Hq][128]
    float* o_raw;            // [T][Hq][128]
    float* lse_raw;          // [T][Hq] or null
    float* o_slot;           // [M][Hq][128]
    float* lse_slot;         // [M][Hq] or null
    int* d_err;
    int T, M, S, W, r, Hq, Hkv, self_attend;
    int merge_ok;            // 1: S <= 8 and the merged-block maps exist
    float scale_log2;
};

// bits [lo, hi) of a 64-column block (0 <= lo, hi <= 64; empty when hi <= lo)
__device__ __forceinline__ uint64_t col_bits(int lo, int hi) {
    const uint64_t a = hi >= 64 ? ~0ull : ((1ull << hi) - 1ull);
    const uint64_t b = lo >= 64 ? ~0ull : ((1ull << lo) - 1ull);
    return a & ~b;
}

// mbarriers of one CTA
__device__ __forceinline__ constexpr int bar_k(int s) { return s; }        // K stage landed (TMA)
__device__ __forceinline__ constexpr int bar_v(int s) { return 3 + s; }    // V stage landed (TMA)
constexpr int kBarS = 6;       // S = Q K^T done (MMA commit)
constexpr int kBarSFree = 7;   // the four softmax warps have read S (4 arrivals)
constexpr int kBarP = 8;       // the four softmax warps have written P and rescaled O (4 arrivals)
constexpr int kBarO = 9;       // O += P V done (MMA commit)
constexpr int kBarQ = 10;      // the four softmax warps have stored Q in tensor memory (4 arrivals)
constexpr int kBarDone = 11;   // every S MMA done (early exit only)
constexpr int kBarDoneV = 12;  // every PV MMA done (early exit only)
constexpr int kNumBars = 13;

// Warp roles: warps 0-3 own query rows 0-127 (TMEM lanes), stage Q into tensor
// memory and run the softmax; lane 0 of warp 4 loads K and issues S = Q K^T,
// lane 0 of warp 5 loads V and issues O += P V.  They hand off through mbarriers
// only.  Two CTAs per SM.
__global__ void __launch_bounds__(192, 2) prefill_kernel(const __grid_constant__ PrefillParams p) {
    using namespace tcp;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sb = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * kNumBars + 4);
    auto bar_at = [&](int i) { return sb + kOffBar + 8u * (uint32_t)i; };

    const int G = p.Hq / p.Hkv;
    const int hq = (int)blockIdx.y, kvh = hq / G;                // query head and its kv head
    const int S = p.S, W = p.W, r = p.r;
    // The CTA's rows [q0, q1) of the interleaved order of the T + M query rows.
    // A slot row g_m has the mask of raw row tau_m (the sink, the window at
    // tau_m, slots 1..m-1), so slot rows ride in the raw tiles with tau_m as
    // their position.
    const int q0 = (int)blockIdx.x * kBM, q1 = imin(p.T + p.M, q0 + kBM);
    const bool live = tid < kBM && q0 + tid < q1;
    auto eff = [&](int x) { return x > 0 ? x : S + W + (-x) * r; };
    const int xr = live ? interleaved_row(q0 + tid, S, W, r, p.M) : 1;   // this row: raw token (> 0) or slot (< 0)

    // visible key ranges of the CTA: 0 = sink and 1 = window band (raw rows),
    // 2 = slot prefix (slot rows), each [a_k, b_k) possibly empty; this thread's
    // row sees the interval [lo_k, hi_k) of range k.  Kept in scalars (no
    // dynamically indexed arrays) so that nothing spills to local memory.
    const int i_first = eff(interleaved_row(q0, S, W, r, p.M)), i_last = eff(interleaved_row(q1 - 1, S, W, r, p.M));
    const int b0 = imin(S, i_last);
    const int a1 = imax(S + 1, i_first - W + 1) - 1;
    const int b1 = imax(a1, i_last);
    // slots with tau < i_last (a slot row with self-attention also sees itself)
    const int b2 = slot_count(p.self_attend ? i_last : i_last - 1, S, W, r);
    const int i = eff(xr);
    const int lo1 = imax(S + 1, i - W + 1) - 1;
    int hi0 = 0, hi1 = 0, hi2 = 0;
    if (live) {
        hi0 = imin(S, i);
        hi1 = i;
        hi2 = xr > 0 ? slot_count(i - 1, S, W, r) : (p.self_attend ? -xr : -xr - 1);
    }
    // The sink (S <= 8 keys) and a slot prefix of at most 56 slots share one
    // block when both are present: rows 0..7 of the stage come from the raw
    // arrays, rows 8..63 from the slot arrays, and a row sees columns
    // [0, hi0) and [8, 8 + hi2) of it.  It saves the tile a block of 64 keys.
    const bool merged = p.merge_ok && b0 > 0 && b2 > 0 && b2 <= kBN - 8;
    const int bs1 = (b0 + kBN - 1) / kBN;
    const int bs2 = bs1 + (b1 - a1 + kBN - 1) / kBN;
    const int nblk = bs2 + (merged ? 0 : (b2 + kBN - 1) / kBN);
    // range index and first key of block blk
    auto block_of = [&](int blk, int& k, int& key0) {
        k = (blk >= bs1 ? 1 : 0) + (blk >= bs2 ? 1 : 0);
        key0 = k == 0 ? blk * kBN : (k == 1 ? a1 + (blk - bs1) * kBN : (blk - bs2) * kBN);
    };

    pdl_wait();
    pdl_trigger();
    // this thread's Q row (softmax threads): all 16 loads in flight while the
    // CTA allocates tensor memory and initialises its barriers
    uint4 qreg[16];
    if (warp < 4) {
        const __nv_bfloat16* qsrc = xr > 0 ? p.q_raw + (size_t)(xr - 1) * p.Hq * kD : p.q_slot + (size_t)(-xr - 1) * p.Hq * kD;
        const uint4* qp = reinterpret_cast<const uint4*>(qsrc + (size_t)hq * kD);
#pragma unroll
        for (int c = 0; c < 16; ++c) qreg[c] = live ? __ldg(qp + c) : make_uint4(0u, 0u, 0u, 0u);
    }
    // the swizzled layouts need a 1024-byte aligned base; after a timed-out wait
    // anywhere in the grid the remaining CTAs skip their work
    const bool misaligned = (sb & 1023u) != 0u;
    if (__syncthreads_or(tid == 0 && (misaligned || *reinterpret_cast<volatile int*>(p.d_err) == MASW_ETIMEOUT))) {
        if (misaligned && tid == 0) atomicExch(p.d_err + 2, 1);
        return;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b)
            mbar_init(bars + b, (b == kBarSFree || b == kBarP || b == kBarQ) ? 4 : 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp >= 4) {
        // ------- warp 4 lane 0: K loads and S = Q K^T; warp 5 lane 0: V loads and O += P V -------
        // (two issuing threads: each waits on its own inputs, so neither MMA
        // stream stalls behind the other's waits)
        if (lane == 0 && nblk > 0) {
            const bool is_v = warp == 5;
            // blocks whose load was issued / waited: [0, li) / [0, lw)
            int li = 0, lw = 0;
            auto load = [&](int blk) {
                int k, key0;
                block_of(blk, k, key0);
                const CUtensorMap* m =
                    k == 2 ? (is_v ? &p.tm_v_slot : &p.tm_k_slot) : (is_v ? &p.tm_v_raw : &p.tm_k_raw);
                const int st = blk % kStages;
                const int bi = is_v ? bar_v(st) : bar_k(st);
                const uint32_t dst = sb + (is_v ? kOffV : kOffK) + st * kKVBytes;
                mbar_expect_tx(bars + bi, kKVBytes);
                if (merged && k == 0) {
                    // 8 raw rows (1 KB per 64-column panel) then 56 slot rows at
                    // the next 1024-byte boundary: the same bytes and swizzle
                    // phase as one 64-row box
                    const CUtensorMap* ms = is_v ? &p.tm_v_sink : &p.tm_k_sink;
                    const CUtensorMap* mg = is_v ? &p.tm_v_slot56 : &p.tm_k_slot56;
#pragma unroll
                    for (int pn = 0; pn < 2; ++pn) {
                        tma_load_3d(dst + pn * (kKVBytes / 2), ms, 64 * pn, kvh, 0, bar_at(bi));
                        tma_load_3d(dst + pn * (kKVBytes / 2) + 1024, mg, 64 * pn, kvh, 0, bar_at(bi));
                    }
                } else {
                    tma_load_3d(dst, m, 0, kvh, key0, bar_at(bi));
                    tma_load_3d(dst + kKVBytes / 2, m, 64, kvh, key0, bar_at(bi));
                }
                li = blk + 1;
            };
            for (int b = 0; b < imin(2, nblk); ++b) load(b);
            bool ok = true;
            if (!is_v) {
                ok = wait_or_abort(bars + kBarQ, 0, abort_flag, p.d_err);
                for (int j = 0; ok && j < nblk; ++j) {
                    const int st = j % kStages;
                    ok = wait_or_abort(bars + bar_k(st), (uint32_t)(j / kStages) & 1u, abort_flag, p.d_err);
                    if (ok) lw = j + 1;
                    // single S buffer: the softmax must have read S(j-1)
                    if (ok && j >= 1) ok = wait_or_abort(bars + kBarSFree, (uint32_t)(j - 1) & 1u, abort_flag, p.d_err);
                    if (!ok) break;
                    tc_fence_after();
                    // descriptor of the stage once; k-step kk adds a compile-time
                    // offset to the start-address field (addresses stay < 256 KB)
                    const uint64_t bd0 = sw128_desc(sb + kOffK + st * kKVBytes, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk)
                        umma_bf16_ts(tmem + kColS, tmem + kColQ + kk * 8,
                                     bd0 + (uint64_t)(((kk >> 2) * (kKVBytes / 2) + (kk & 3) * 32) >> 4), kIdescS,
                                     kk > 0 ? 1u : 0u);
                    umma_commit(bar_at(kBarS));
                    // K(j+2) takes the stage of K(j-1), whose S the softmax has read
                    if (j + 2 < nblk) load(j + 2);
                }
            } else {
                for (int j = 0; ok && j < nblk; ++j) {
                    const int st = j % kStages;
                    ok = wait_or_abort(bars + kBarP, (uint32_t)j & 1u, abort_flag, p.d_err);
                    if (ok) {
                        ok = wait_or_abort(bars + bar_v(st), (uint32_t)(j / kStages) & 1u, abort_flag, p.d_err);
                        if (ok) lw = j + 1;
                    }
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t a0 = sw128_desc(sb + kOffP, 16, 1024);
                    const uint64_t v0 = sw128_desc(sb + kOffV + st * kKVBytes, kKVBytes / 2, 1024);
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        umma_bf16(tmem + kColO, a0 + (uint64_t)((kk * 32) >> 4), v0 + (uint64_t)((kk * 2048) >> 4),
                                  kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(bar_at(kBarO));
                    // P(j) written means the softmax saw PV(j-1) complete:
                    // V(j+2) takes the stage of V(j-1)
                    if (j + 2 < nblk) load(j + 2);
                }
            }
            if (!ok) {
                // early exit: let this thread's MMAs and loads in flight finish
                // before the CTA releases its tensor and shared memory
                *abort_flag = 1;
                const int done = is_v ? kBarDoneV : kBarDone;
                umma_commit(bar_at(done));
                mbar_wait(bars + done, 0, nullptr);
                for (int blk = lw; blk < li; ++blk)
                    mbar_wait(bars + (is_v ? bar_v(blk % kStages) : bar_k(blk % kStages)),
                              (uint32_t)(blk / kStages) & 1u, nullptr);
            }
        }
        __syncwarp();
    } else {
        // ---------------- softmax warps: thread tid owns query row tid ----------------
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const uint32_t t_o = tmem + kColO + lane_off;
        // Q row -> tensor memory (zeros past the last row), the A operand of S
        {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t qv[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 w = qreg[h * 8 + c];
                    qv[4 * c] = w.x;
                    qv[4 * c + 1] = w.y;
                    qv[4 * c + 2] = w.z;
                    qv[4 * c + 3] = w.w;
                }
                tmem_st32(tmem + kColQ + lane_off + h * 32, qv);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_at(kBarQ));
        }
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < nblk; ++j) {
            if (!__all_sync(0xffffffffu, wait_or_abort(bars + kBarS, (uint32_t)j & 1u, abort_flag, p.d_err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[2][32];
            tmem_ld32(tmem + kColS + lane_off, sv[0]);
            tmem_ld32(tmem + kColS + lane_off + 32, sv[1]);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_at(kBarSFree));

            int k, key0;
            block_of(j, k, key0);
            const int lo_k = k == 1 ? lo1 : 0;
            const int hi_k = k == 0 ? hi0 : (k == 1 ? hi1 : hi2);
            // visible columns of this block for this row: [e_lo, e_hi)
            const int e_lo = imin(kBN, imax(0, lo_k - key0)), e_hi = imin(kBN, imax(0, hi_k - key0));
            float x[64];
#pragma unroll
            for (int e = 0; e < 64; ++e) x[e] = __uint_as_float(sv[e >> 5][e & 31]);
            // visible columns as a bit mask: [e_lo, e_hi), or in the merged
            // block the sink columns [0, hi0) and the slot columns [8, 8 + hi2)
            const uint64_t vis = (merged && k == 0) ? (col_bits(0, hi0) | col_bits(8, 8 + hi2)) : col_bits(e_lo, e_hi);
            if (vis != ~0ull) {
                const uint32_t v_lo = (uint32_t)vis, v_hi = (uint32_t)(vis >> 32);
#pragma unroll
                for (int e = 0; e < 64; ++e)
                    x[e] = (((e < 32 ? v_lo : v_hi) >> (e & 31)) & 1u) ? x[e] : -INFINITY;
            }
            // row max of the raw scores (scale > 0 commutes with max): 3-input
            // max in four chains
            float mx4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
            for (int e = 4; e < 64; e += 8) {
#pragma unroll
                for (int c = 0; c < 4; ++c) mx4[c] = fmax3(mx4[c], x[e + 2 * c], x[e + 2 * c + 1]);
            }
            const float mx = fmax3(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3], mx4[3]);
            float alpha = 1.f;
            const float m_new = fmaxf(m_run, mx * p.scale_log2);
            if (m_new > m_run + 8.f) {
                alpha = ex2_approx(m_run - m_new);
                m_run = m_new;
            }
            const float nmref = m_run == -INFINITY ? 0.f : -m_run;
            // p = 2^(x * scale_log2 - m): packed FMA for the arguments, packed
            // adds for the row sum (four f32x2 chains)
            const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nm2 = f2_pack(nmref, nmref);
            uint32_t pk[32];
            uint64_t sum2[4] = {0, 0, 0, 0};
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                float a0, a1v;
                f2_unpack(f2_fma(f2_pack(x[2 * e], x[2 * e + 1]), sc2, nm2), a0, a1v);
                const float p0 = ex2_approx(a0), p1 = ex2_approx(a1v);
                sum2[e & 3] = f2_add(sum2[e & 3], f2_pack(p0, p1));
                pk[e] = pack_bf16(p0, p1);
            }
            float sum_lo, sum_hi;
            f2_unpack(f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3])), sum_lo, sum_hi);
            const float sum = sum_lo + sum_hi;
            const bool resc = alpha != 1.f && l_run > 0.f;
            l_run = l_run * alpha + sum;

            // PV(j-1) must be complete before O is rescaled and P is overwritten
            if (j > 0) {
                if (!__all_sync(0xffffffffu,
                                wait_or_abort(bars + kBarO, (uint32_t)(j - 1) & 1u, abort_flag, p.d_err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(t_o + c * 32, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                    tmem_st32(t_o + c * 32, ov);
                }
                tmem_wait_st();
            }
            // row tid of P: 64 bf16 = one 128-byte swizzled row
            const uint32_t prow = sb + kOffP + (uint32_t)tid * 128u;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                st_shared_v4(prow + ((uint32_t)(c ^ (tid & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                             pk[4 * c + 3]);
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_at(kBarP));
        }
        // last PV, then O / l for this row
        if (ok && nblk > 0)
            ok = __all_sync(0xffffffffu,
                            wait_or_abort(bars + kBarO, (uint32_t)(nblk - 1) & 1u, abort_flag, p.d_err));
        tc_fence_after();
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        // O / l through a swizzled 32 x 32 tile per warp in the (now idle) K
        // stages: thread `lane` writes 32 columns of its row, then each store
        // instruction writes 128-byte pieces of 4 rows (the rows are Hq*512
        // bytes apart in global memory, so one row per thread would scatter)
        if (ok && nblk > 0) {
            const uint32_t tile = sb + kOffK + (uint32_t)warp * 4096u;
            float* rowp[8];                              // global row of tile row 4 i + lane / 8, or null
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int tl = i * 4 + (lane >> 3);     // row warp * 32 + tl, owned by lane tl
                const int x = __shfl_sync(0xffffffffu, xr, tl);
                const bool lv = q0 + warp * 32 + tl < q1;
                rowp[i] = !lv ? nullptr
                              : (x > 0 ? p.o_raw + ((size_t)(x - 1) * p.Hq + hq) * kD
                                       : p.o_slot + ((size_t)(-x - 1) * p.Hq + hq) * kD);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t ov[32];
                tmem_ld32(t_o + c * 32, ov);
                tmem_wait_ld();
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4)
                    st_shared_v4(tile + (uint32_t)lane * 128u + ((uint32_t)(e4 ^ (lane & 7)) << 4),
                                 __float_as_uint(__uint_as_float(ov[4 * e4]) * inv),
                                 __float_as_uint(__uint_as_float(ov[4 * e4 + 1]) * inv),
                                 __float_as_uint(__uint_as_float(ov[4 * e4 + 2]) * inv),
                                 __float_as_uint(__uint_as_float(ov[4 * e4 + 3]) * inv));
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rr = i * 4 + (lane >> 3), e4 = lane & 7;
                    const float4 v = ld_shared_v4f(tile + (uint32_t)rr * 128u + ((uint32_t)(e4 ^ (rr & 7)) << 4));
                    if (rowp[i]) *reinterpret_cast<float4*>(rowp[i] + c * 32 + e4 * 4) = v;
                }
                __syncwarp();
            }
        }
        float* lp = xr > 0 ? (p.lse_raw ? p.lse_raw + (size_t)(xr - 1) * p.Hq + hq : nullptr)
                           : (p.lse_slot ? p.lse_slot + (size_t)(-xr - 1) * p.Hq + hq : nullptr);
        if (live && lp) *lp = l_run > 0.f ? (m_run + __log2f(l_run)) * 0.6931471805599453f : -INFINITY;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// Store the prefill's memory M_0 of one (layer, sequence): sink rows, the last
// W+R raw tokens in their ring rows, the slot chain, the full-KV cache, the
// per-head counters and the slot position ids.
struct StoreParams {
    const uint8_t* k_raw;   // [T][Hkv][rowb]
    const uint8_t* v_raw;
    const uint8_t* k_slot;  // [M][Hkv][rowb]
    const uint8_t* v_slot;
    uint8_t* pool_k;
    uint8_t* pool_v;
    uint8_t* full_k;
    uint8_t* full_v;
    int* d_t;
    int* d_m;
    int* d_pos;
    int lb, T, M, S, W, r, Wc, C, Hkv, rowb, Tmax, M_max;
};

__global__ void prefill_store_kernel(const __grid_constant__ StoreParams p) {
    pdl_wait();
    pdl_trigger();
    // grid-stride over (source row, head, 16-byte chunk) of raw then slot rows
    const int vpr = p.rowb / 16;
    const size_t nraw = (size_t)p.T * p.Hkv * vpr, nslot = (size_t)p.M * p.Hkv * vpr;
    const int ring_from = imax(p.S + 1, p.T - p.Wc + 1);   // oldest raw token kept in the ring
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < nraw + nslot;
         idx += (size_t)gridDim.x * blockDim.x) {
        const bool is_slot = idx >= nraw;
        const size_t li = is_slot ? idx - nraw : idx;
        const int cc = (int)(li % vpr);
        const int hh = (int)((li / vpr) % p.Hkv);
        const int row = (int)(li / ((size_t)vpr * p.Hkv));
        const size_t src = ((size_t)row * p.Hkv + hh) * p.rowb + cc * 16;
        const size_t blk = ((size_t)p.lb * p.Hkv + hh);
        if (is_slot) {
            const size_t dst = (blk * p.C + p.S + p.Wc + row) * p.rowb + cc * 16;
            *reinterpret_cast<uint4*>(p.pool_k + dst) = *reinterpret_cast<const uint4*>(p.k_slot + src);
            *reinterpret_cast<uint4*>(p.pool_v + dst) = *reinterpret_cast<const uint4*>(p.v_slot + src);
            continue;
        }
        const uint4 kv = *reinterpret_cast<const uint4*>(p.k_raw + src);
        const uint4 vv = *reinterpret_cast<const uint4*>(p.v_raw + src);
        const int i = row + 1;
        int prow = -1;
        if (i <= p.S) prow = i - 1;
        else if (i >= ring_from) prow = p.S + ring_row(i, p.S, p.Wc);
        if (prow >= 0) {
            const size_t dst = (blk * p.C + prow) * p.rowb + cc * 16;
            *reinterpret_cast<uint4*>(p.pool_k + dst) = kv;
            *reinterpret_cast<uint4*>(p.pool_v + dst) = vv;
        }
        if (p.full_k) {
            const size_t dst = (blk * p.Tmax + row) * p.rowb + cc * 16;
            *reinterpret_cast<uint4*>(p.full_k + dst) = kv;
            *reinterpret_cast<uint4*>(p.full_v + dst) = vv;
        }
    }
    if (blockIdx.x == 0) {
        for (int hh = threadIdx.x; hh < p.Hkv; hh += blockDim.x) {
            p.d_t[(size_t)p.lb * p.Hkv + hh] = p.T;
            p.d_m[(size_t)p.lb * p.Hkv + hh] = p.M;
        }
        for (int j = threadIdx.x; j < p.M; j += blockDim.x)
            p.d_pos[(size_t)p.lb * p.M_max + j] = p.S + p.W + (j + 1) * p.r;
    }
}

}  // namespace masw

using namespace masw;

// [rows][heads][128] bf16 as a 3-d tensor (head_dim innermost), boxes of
// 64 x 1 x box_rows elements with the 128-byte swizzle the MMA descriptors use
static bool make_map(CUtensorMap* map, const void* base, int rows, int heads, int box_rows) {
    const cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {256, (cuuint64_t)heads * 256};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    return tma_encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

extern "C" int masw_prefill(masw_mem_t* mem, int layer, int seq, int T, const void* q_raw, const void* k_raw,
                            const void* v_raw, const void* q_slot, const void* k_slot, const void* v_slot,
                            int n_q_heads, float* o_raw, float* lse_raw, float* o_slot, float* lse_slot,
                            masw_stream_t stream) {
    if (!mem) return masw_set_error(nullptr, MASW_EINVAL, "prefill: NULL handle");
    if (layer < 0 || layer >= mem->L || seq < 0 || seq >= mem->B)
        return masw_set_error(mem, MASW_EINVAL, "prefill: layer or seq out of range");
    if (mem->dtype != MASW_BF16 || mem->D != tcp::kD)
        return masw_set_error(mem, MASW_EINVAL, "prefill: bf16 pools with head_dim 128 only");
    if (n_q_heads < mem->Hkv || n_q_heads % mem->Hkv) return masw_set_error(mem, MASW_EINVAL, "prefill: bad n_q_heads");
    if (T < 1 || T > mem->max_seq_len) return masw_set_error(mem, MASW_ECAPACITY, "prefill: T out of range");
    const int M = slot_count(T, mem->S, mem->W, mem->r);
    if (M > mem->M_max) return masw_set_error(mem, MASW_ECAPACITY, "prefill: slot chain too short");
    if (!q_raw || !k_raw || !v_raw || !o_raw || (M > 0 && (!q_slot || !k_slot || !v_slot || !o_slot)))
        return masw_set_error(mem, MASW_EINVAL, "prefill: NULL pointer");
    if (((uintptr_t)q_raw | (uintptr_t)k_raw | (uintptr_t)v_raw | (uintptr_t)q_slot | (uintptr_t)k_slot |
         (uintptr_t)v_slot) & 15)
        return masw_set_error(mem, MASW_EINVAL, "prefill: inputs must be 16-byte aligned");
    if (((uintptr_t)o_raw | (uintptr_t)o_slot) & 7 || ((uintptr_t)lse_raw | (uintptr_t)lse_slot) & 3)
        return masw_set_error(mem, MASW_EINVAL, "prefill: outputs must be 8-byte (O) / 4-byte (LSE) aligned");
    if (n_q_heads > 65535) return masw_set_error(mem, MASW_EINVAL, "prefill: too many heads");
    if (!tma_encode_fn()) return masw_set_error(mem, MASW_ECUDA, "prefill: cuTensorMapEncodeTiled is unavailable");
    PrefillParams p;
    std::memset(&p, 0, sizeof(p));
    const int Hkv = mem->Hkv;
    bool maps = make_map(&p.tm_k_raw, k_raw, T, Hkv, tcp::kBN) &&
                make_map(&p.tm_v_raw, v_raw, T, Hkv, tcp::kBN);
    if (M > 0)
        maps = maps && make_map(&p.tm_k_slot, k_slot, M, Hkv, tcp::kBN) && make_map(&p.tm_v_slot, v_slot, M, Hkv, tcp::kBN);
    if (!maps) return masw_set_error(mem, MASW_EINVAL, "prefill: cannot describe the inputs as TMA tensors");
    // maps of the merged sink + slot block (8 raw rows, then 56 slot rows)
    if (M > 0 && mem->S >= 1 && mem->S <= 8)
        p.merge_ok = make_map(&p.tm_k_sink, k_raw, T, Hkv, 8) && make_map(&p.tm_v_sink, v_raw, T, Hkv, 8) &&
                     make_map(&p.tm_k_slot56, k_slot, M, Hkv, tcp::kBN - 8) &&
                     make_map(&p.tm_v_slot56, v_slot, M, Hkv, tcp::kBN - 8);
    p.q_raw = (const __nv_bfloat16*)q_raw;
    p.q_slot = (const __nv_bfloat16*)q_slot;
    p.o_raw = o_raw;
    p.lse_raw = lse_raw;
    p.o_slot = o_slot;
    p.lse_slot = lse_slot;
    p.d_err = mem->d_err;
    p.T = T;
    p.M = M;
    p.S = mem->S;
    p.W = mem->W;
    p.r = mem->r;
    p.Hq = n_q_heads;
    p.Hkv = Hkv;
    p.self_attend = mem->self_attend;
    p.scale_log2 = mem->scale * 1.4426950408889634f;
    // 128-row tiles of the T + M query rows in interleaved order
    const int tiles = (T + M + tcp::kBM - 1) / tcp::kBM;
    cudaStream_t st = (cudaStream_t)stream;
    static std::atomic<bool> configured[64];   // per device, set once (idempotent)
    if (!configured[mem->device & 63].load(std::memory_order_acquire)) {
        MASW_CUDA_TRY(mem, cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tcp::kSmem));
        MASW_CUDA_TRY(mem, cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                cudaSharedmemCarveoutMaxShared));
        configured[mem->device & 63].store(true, std::memory_order_release);
    }
    masw_note_launch(mem, (void*)st, layer);   // the store kernel below writes this layer's rows
    MASW_CUDA_TRY(mem, masw_launch(prefill_kernel, dim3(tiles, n_q_heads), dim3(192), tcp::kSmem, st, 1, p));
    StoreParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.k_raw = (const uint8_t*)k_raw;
    sp.v_raw = (const uint8_t*)v_raw;
    sp.k_slot = (const uint8_t*)k_slot;
    sp.v_slot = (const uint8_t*)v_slot;
    sp.pool_k = (uint8_t*)mem->pool_k;
    sp.pool_v = (uint8_t*)mem->pool_v;
    sp.full_k = (uint8_t*)mem->full_k;
    sp.full_v = (uint8_t*)mem->full_v;
    sp.d_t = mem->d_t;
    sp.d_m = mem->d_m;
    sp.d_pos = mem->d_pos;
    sp.lb = layer * mem->B + seq;
    sp.T = T;
    sp.M = M;
    sp.S = mem->S;
    sp.W = mem->W;
    sp.r = mem->r;
    sp.Wc = mem->Wc;
    sp.C = mem->C;
    sp.Hkv = mem->Hkv;
    sp.rowb = mem->D * (int)mem->esize;
    sp.Tmax = mem->max_seq_len;
    sp.M_max = mem->M_max;
    const size_t vecs = (size_t)(T + M) * mem->Hkv * (sp.rowb / 16);
    const int blocks = (int)std::min<size_t>((vecs + 255) / 256, (size_t)mem->num_sms * 8);
    MASW_CUDA_TRY(mem, masw_launch(prefill_store_kernel, dim3(imax(1, blocks)), dim3(256), 0, st, 1, sp));
    mem->h_t[(size_t)layer * mem->B + seq] = T;
    mem->h_m[(size_t)layer * mem->B + seq] = M;
    return MASW_OK;
}
