// Draft prefill under the structured write mask ([EN] §3.3 Algorithm 2 step 2
// with the mask of §3.2 Algorithm 1 step 2): one layer of attention over a whole
// prefix of T raw tokens with the M = m(T) memory-slot tokens interleaved, then
// the resulting memory M_0 is stored in the pool.
//
// Query rows: raw token i (1-based) reads the sink, raw tokens of its window
// [max(S+1, i-W+1), i], and the slots materialised before it (tau_m < i); slot
// token g_m reads the sink, the window at tau_m and slots 1..m-1.  Key rows come
// from the caller's raw and slot K/V arrays ([T, Hkv, D], [M, Hkv, D]).  For one
// tile of query rows the visible keys are a few contiguous ranges (sink, window
// band, slot prefix), and for one row each range is a single interval, so the
// mask is two compares per score.
//
// Fifth-generation tensor cores, one CTA per (128-row query tile, query head):
//   * TMA tiled loads (128-byte swizzle) bring Q (resident), and K and V blocks
//     of 64 keys into two stages each;
//   * thread 0 issues S = Q K^T (tcgen05.mma, M = 128, N = 64, accumulator in
//     tensor memory) and O += P V (M = 128, N = 128, V read MN-major);
//   * thread t owns query row t (TMEM lane t): it reads its 64 scores with
//     tcgen05.ld, applies the mask and the online softmax, and writes its row of
//     P (bf16) into shared memory in the swizzled K-major layout the next MMA
//     reads;
//   * the running max only moves when a row's maximum grows by more than 2^8,
//     so the O rescale (tcgen05.ld / st of the row) is rare; the final
//     normalisation uses the same max, so the result is exact.
// 112 KB of shared memory and 256 TMEM columns per CTA: two CTAs per SM, whose
// softmax and MMA phases overlap.
#include "masw_internal.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

namespace masw {

namespace tcp {

constexpr int kBM = 128;                         // query rows per CTA = TMEM lanes
constexpr int kBN = 64;                          // keys per block
constexpr int kD = 128;                          // head_dim
constexpr uint32_t kQBytes = kBM * kD * 2;       // 2 panels of 128 rows x 128 B
constexpr uint32_t kKVBytes = kBN * kD * 2;      // 2 panels of 64 rows x 128 B
constexpr uint32_t kPBytes = kBM * kBN * 2;      // 1 panel of 128 rows x 128 B
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffV = kOffK + 2 * kKVBytes;
constexpr uint32_t kOffP = kOffV + 2 * kKVBytes;
constexpr uint32_t kOffBar = kOffP + kPBytes;    // 9 mbarriers + the TMEM address
constexpr uint32_t kSmem = kOffBar + 80;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 0;                    // O: columns [0, 128)
constexpr uint32_t kColS = 128;                  // S: two buffers, columns [128, 192) and [192, 256)
// instruction descriptors (kind::f16): f32 accumulator, bf16 A and B, M = 128;
// S: N = 64, both operands K-major; O: N = 128, B (V) MN-major
constexpr uint32_t kIdescBase = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBM >> 4) << 24);
constexpr uint32_t kIdescS = kIdescBase | ((uint32_t)(kBN >> 3) << 17);
constexpr uint32_t kIdescO = kIdescBase | (1u << 16) | ((uint32_t)(kD >> 3) << 17);

// shared-memory matrix descriptor, 128-byte swizzle (atoms of 8 rows x 128 B)
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// 2^x by the MUFU instruction (inputs of -inf give 0)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

#define MASW_R8(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), "=r"(v[i + 4]), "=r"(v[i + 5]), \
                   "=r"(v[i + 6]), "=r"(v[i + 7])
#define MASW_W8(i) "r"(v[i]), "r"(v[i + 1]), "r"(v[i + 2]), "r"(v[i + 3]), "r"(v[i + 4]), "r"(v[i + 5]), \
                   "r"(v[i + 6]), "r"(v[i + 7])
// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : MASW_R8(0), MASW_R8(8), MASW_R8(16), MASW_R8(24)
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        MASW_W8(0), MASW_W8(8), MASW_W8(16), MASW_W8(24)
        : "memory");
}
#undef MASW_R8
#undef MASW_W8
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

}  // namespace tcp

struct PrefillParams {
    CUtensorMap tm_q_raw;    // [T][Hq][128] bf16, box 64 x 1 x 128
    CUtensorMap tm_k_raw;    // [T][Hkv][128] bf16, box 64 x 1 x 64
    CUtensorMap tm_v_raw;
    CUtensorMap tm_q_slot;   // [M][Hq][128] (unused when M = 0)
    CUtensorMap tm_k_slot;   // [M][Hkv][128]
    CUtensorMap tm_v_slot;
    float* o_raw;            // [T][Hq][128]
    float* lse_raw;          // [T][Hq] or null
    float* o_slot;           // [M][Hq][128]
    float* lse_slot;         // [M][Hq] or null
    int* d_err;
    int T, M, S, W, r, Hq, Hkv, self_attend;
    int raw_tiles;           // tiles of raw query rows (the rest are slot tiles)
    int slot_rows;           // slot query rows per slot tile
    float scale_log2;
};

__global__ void __launch_bounds__(128, 2) prefill_kernel(const __grid_constant__ PrefillParams p) {
    using namespace tcp;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t sb = smem_u32(smem);
    // mbarriers: q, k0, k1, v0, v1, s0, s1, o, done
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffBar + 72);
    const uint32_t bar_q = sb + kOffBar, bar_o = bar_q + 56, bar_done = bar_q + 64;

    const int hq = blockIdx.y, G = p.Hq / p.Hkv, kvh = hq / G;
    const bool slot_tile = (int)blockIdx.x >= p.raw_tiles;
    const int q0 = slot_tile ? ((int)blockIdx.x - p.raw_tiles) * p.slot_rows : (int)blockIdx.x * kBM;
    const int nq = slot_tile ? p.M : p.T;
    const int q1 = imin(nq, q0 + (slot_tile ? p.slot_rows : kBM));
    const int S = p.S, W = p.W, r = p.r;

    // visible key ranges of the tile: 0 = sink and 1 = window band (raw rows),
    // 2 = slot prefix (slot rows), each [a_k, b_k) possibly empty; this thread's
    // row sees the interval [lo_k, hi_k) of range k.  Kept in scalars (no
    // dynamically indexed arrays) so that nothing spills to local memory.
    const int qrow = q0 + tid;
    const bool live = qrow < q1;
    int a0 = 0, b0 = 0, a1 = 0, b1 = 0, b2 = 0;
    int lo1 = 0, hi0 = 0, hi1 = 0, hi2 = 0;
    if (!slot_tile) {
        const int i0 = q0 + 1, i1 = q1, i = qrow + 1;   // 1-based raw positions
        b0 = imin(S, i1);
        a1 = imax(S + 1, i0 - W + 1) - 1;
        b1 = imax(a1, i1);
        b2 = slot_count(i1 - 1, S, W, r);
        lo1 = imax(S + 1, i - W + 1) - 1;
        if (live) {
            hi0 = imin(S, i);
            hi1 = i;
            hi2 = slot_count(i - 1, S, W, r);
        }
    } else {
        const int m0 = q0 + 1, m1 = q1, m = qrow + 1;   // 1-based slot indices
        const int tau0 = S + W + m0 * r, tau1 = S + W + m1 * r, tau = S + W + m * r;
        b0 = S;
        a1 = imax(S, tau0 - W);
        b1 = tau1;
        b2 = imax(0, p.self_attend ? m1 : m1 - 1);
        lo1 = tau - W;
        if (live) {
            hi0 = S;
            hi1 = tau;
            hi2 = p.self_attend ? m : m - 1;
        }
    }
    (void)a0;
    const int bs1 = (b0 + kBN - 1) / kBN;
    const int bs2 = bs1 + (b1 - a1 + kBN - 1) / kBN;
    const int nblk = bs2 + (b2 + kBN - 1) / kBN;
    // range index and first key of block blk
    auto block_of = [&](int blk, int& k, int& key0) {
        k = (blk >= bs1 ? 1 : 0) + (blk >= bs2 ? 1 : 0);
        key0 = k == 0 ? blk * kBN : (k == 1 ? a1 + (blk - bs1) * kBN : (blk - bs2) * kBN);
    };

    pdl_wait();
    pdl_trigger();
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
        for (int b = 0; b < 9; ++b) mbar_init(bars + b, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t t_o = tmem + kColO;

    // thread 0: TMA producer and MMA issuer
    // per stage: loads issued and phases waited (thread 0's bookkeeping, for the
    // drain on an early exit); bit-packed counters, stage st in bits 16*st
    uint32_t issued_k = 0, issued_v = 0, waited_k = 0, waited_v = 0;
    auto load_kv = [&](int blk, bool is_v) {
        int k, key0;
        block_of(blk, k, key0);
        const CUtensorMap* m = k == 2 ? (is_v ? &p.tm_v_slot : &p.tm_k_slot) : (is_v ? &p.tm_v_raw : &p.tm_k_raw);
        const int st = blk & 1;
        const uint32_t dst = sb + (is_v ? kOffV : kOffK) + st * kKVBytes;
        const uint32_t bar = sb + kOffBar + 8 * ((is_v ? 3 : 1) + st);
        mbar_expect_tx(bars + (is_v ? 3 : 1) + st, kKVBytes);
        tma_load_3d(dst, m, 0, kvh, key0, bar);
        tma_load_3d(dst + kKVBytes / 2, m, 64, kvh, key0, bar);
        (is_v ? issued_v : issued_k) += 1u << (16 * st);
    };
    bool ok = true;
    // S(blk) = Q K(blk)^T into TMEM buffer blk & 1 (thread 0; commits even when
    // a wait failed so that the waiting threads move on)
    auto issue_s = [&](int blk) {
        const int st = blk & 1;
        if (ok) {
            ok = mbar_wait(bars + 1 + st, (uint32_t)(blk >> 1) & 1u, p.d_err);
            waited_k += ok ? 1u << (16 * st) : 0u;
        }
        tc_fence_after();
        if (ok) {
            const uint32_t qa = sb + kOffQ, kb = sb + kOffK + st * kKVBytes;
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
                const uint64_t a = sw128_desc(qa + (kk >> 2) * (kQBytes / 2) + (kk & 3) * 32, 16, 1024);
                const uint64_t b = sw128_desc(kb + (kk >> 2) * (kKVBytes / 2) + (kk & 3) * 32, 16, 1024);
                umma_bf16(tmem + kColS + 64 * st, a, b, kIdescS, kk > 0 ? 1u : 0u);
            }
        }
        umma_commit(sb + kOffBar + 8 * (5 + st));
    };
    if (tid == 0) {
        const CUtensorMap* mq = slot_tile ? &p.tm_q_slot : &p.tm_q_raw;
        mbar_expect_tx(bars + 0, kQBytes);
        tma_load_3d(sb + kOffQ, mq, 0, hq, q0, bar_q);
        tma_load_3d(sb + kOffQ + kQBytes / 2, mq, 64, hq, q0, bar_q);
        for (int b = 0; b < imin(2, nblk); ++b) {
            load_kv(b, false);
            load_kv(b, true);
        }
        if (nblk > 0) ok = mbar_wait(bars + 0, 0, p.d_err);
        for (int b = 0; b < imin(2, nblk); ++b) issue_s(b);
    }
    __syncwarp();

    // Block j: S(j) was issued two blocks ahead.  While the threads run the
    // softmax of block j the tensor cores run PV(j-1) and S(j+1).
    float m_run = -INFINITY, l_run = 0.f;
    bool aborted = false;
    for (int j = 0; j < nblk; ++j) {
        const int st = j & 1;
        const uint32_t ph = (uint32_t)(j >> 1) & 1u;
        ok = mbar_wait(bars + 5 + st, ph, p.d_err) && ok;
        tc_fence_after();
        uint32_t sv[2][32];
        tmem_ld32(tmem + kColS + 64 * st + lane_off, sv[0]);
        tmem_ld32(tmem + kColS + 64 * st + lane_off + 32, sv[1]);
        tmem_wait_ld();
        // S(j) is done with K stage st: refill it two blocks ahead
        if (tid == 0 && ok && j + 2 < nblk) load_kv(j + 2, false);

        int k, key0;
        block_of(j, k, key0);
        const int lo_k = k == 1 ? lo1 : 0;
        const int hi_k = k == 0 ? hi0 : (k == 1 ? hi1 : hi2);
        // visible columns of this block for this row: [e_lo, e_hi)
        const int e_lo = imin(kBN, imax(0, lo_k - key0)), e_hi = imin(kBN, imax(0, hi_k - key0));
        float x[64];
#pragma unroll
        for (int e = 0; e < 64; ++e) x[e] = __uint_as_float(sv[e >> 5][e & 31]);
        if (e_lo > 0 || e_hi < kBN) {
#pragma unroll
            for (int e = 0; e < 64; ++e) x[e] = (e >= e_lo && e < e_hi) ? x[e] : -INFINITY;
        }
        // row max of the raw scores (scale > 0 commutes with max), 8 chains
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = x[e];
#pragma unroll
        for (int e = 8; e < 64; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], x[e]);
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        float alpha = 1.f;
        const float m_new = fmaxf(m_run, mx * p.scale_log2);
        if (m_new > m_run + 8.f) {
            alpha = ex2_approx(m_run - m_new);
            m_run = m_new;
        }
        const float nmref = m_run == -INFINITY ? 0.f : -m_run;
        uint32_t pk[32];
        float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const float p0 = ex2_approx(fmaf(x[2 * e], p.scale_log2, nmref));
            const float p1 = ex2_approx(fmaf(x[2 * e + 1], p.scale_log2, nmref));
            sum8[e & 7] += p0 + p1;
            pk[e] = pack_bf16(p0, p1);
        }
        const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
        const bool resc = alpha != 1.f && l_run > 0.f;
        l_run = l_run * alpha + sum;

        // PV(j-1) must be complete before O is rescaled and P is overwritten
        if (j > 0) ok = mbar_wait(bars + 7, (uint32_t)(j - 1) & 1u, p.d_err) && ok;
        tc_fence_after();
        // ... and it released V stage (j+1)&1
        if (tid == 0 && ok && j >= 1 && j + 1 < nblk) load_kv(j + 1, true);
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t ov[32];
                tmem_ld32(t_o + lane_off + c * 32, ov);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                tmem_st32(t_o + lane_off + c * 32, ov);
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
        if (__syncthreads_or(!ok)) {
            aborted = true;   // PV(j) not issued; S(j+1) may still be in flight
            break;
        }
        if (tid == 0) {
            tc_fence_after();
            ok = mbar_wait(bars + 3 + st, ph, p.d_err);
            waited_v += ok ? 1u << (16 * st) : 0u;
            if (ok) {
                const uint32_t vb = sb + kOffV + st * kKVBytes;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t a = sw128_desc(sb + kOffP + kk * 32, 16, 1024);
                    const uint64_t b = sw128_desc(vb + kk * 2048, kKVBytes / 2, 1024);
                    umma_bf16(t_o, a, b, kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
                }
            }
            umma_commit(bar_o);
            // every thread has read S(j): its buffer takes S(j+2)
            if (j + 2 < nblk) issue_s(j + 2);
        }
        __syncwarp();
    }
    // last PV (every committed phase of bar_o is waited here or in the loop)
    if (nblk > 0 && !aborted) ok = mbar_wait(bars + 7, (uint32_t)(nblk - 1) & 1u, p.d_err) && ok;
    tc_fence_after();
    float* obase = slot_tile ? p.o_slot : p.o_raw;
    float* lbase = slot_tile ? p.lse_slot : p.lse_raw;
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    float* orow = obase + ((size_t)(live ? qrow : q0) * p.Hq + hq) * kD;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t ov[32];
        tmem_ld32(t_o + lane_off + c * 32, ov);
        tmem_wait_ld();
        if (live && nblk > 0) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4*>(orow + c * 32 + e) =
                    make_float4(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv,
                                __uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
        }
    }
    if (live && lbase)
        lbase[(size_t)qrow * p.Hq + hq] = l_run > 0.f ? (m_run + __log2f(l_run)) * 0.6931471805599453f : -INFINITY;
    // on an early exit, let the MMAs and loads still in flight finish before the
    // CTA ends (one commit covers every MMA this thread issued)
    if (tid == 0 && (aborted || !ok)) {
        umma_commit(bar_done);
        mbar_wait(bars + 8, 0, nullptr);
        for (int st = 0; st < 2; ++st) {
            const uint32_t sh = 16 * st;
            for (uint32_t n = (waited_k >> sh) & 0xFFFFu; n < ((issued_k >> sh) & 0xFFFFu); ++n)
                mbar_wait(bars + 1 + st, n & 1u, nullptr);
            for (uint32_t n = (waited_v >> sh) & 0xFFFFu; n < ((issued_v >> sh) & 0xFFFFu); ++n)
                mbar_wait(bars + 3 + st, n & 1u, nullptr);
        }
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

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

// [rows][heads][128] bf16 as a 3-d tensor (head_dim innermost), boxes of
// 64 x 1 x box_rows elements with the 128-byte swizzle the MMA descriptors use
static bool make_map(CUtensorMap* map, const void* base, int rows, int heads, int box_rows) {
    const cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {256, (cuuint64_t)heads * 256};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
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
    if (!encode_fn()) return masw_set_error(mem, MASW_ECUDA, "prefill: cuTensorMapEncodeTiled is unavailable");
    PrefillParams p;
    std::memset(&p, 0, sizeof(p));
    const int Hkv = mem->Hkv;
    bool maps = make_map(&p.tm_q_raw, q_raw, T, n_q_heads, tcp::kBM) && make_map(&p.tm_k_raw, k_raw, T, Hkv, tcp::kBN) &&
                make_map(&p.tm_v_raw, v_raw, T, Hkv, tcp::kBN);
    if (M > 0)
        maps = maps && make_map(&p.tm_q_slot, q_slot, M, n_q_heads, tcp::kBM) &&
               make_map(&p.tm_k_slot, k_slot, M, Hkv, tcp::kBN) && make_map(&p.tm_v_slot, v_slot, M, Hkv, tcp::kBN);
    if (!maps) return masw_set_error(mem, MASW_EINVAL, "prefill: cannot describe the inputs as TMA tensors");
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
    p.raw_tiles = (T + tcp::kBM - 1) / tcp::kBM;
    // slot rows per tile: extra rows widen the tile's window band by r keys
    // each, worth it while that stays below the keys every slot row reads anyway
    p.slot_rows = imin(tcp::kBM, imax(1, (mem->S + mem->W + M / 2) / mem->r + 1));
    p.scale_log2 = mem->scale * 1.4426950408889634f;
    const int tiles = p.raw_tiles + (M + p.slot_rows - 1) / p.slot_rows;
    cudaStream_t st = (cudaStream_t)stream;
    static bool configured[64] = {};
    if (!configured[mem->device & 63]) {
        MASW_CUDA_TRY(mem, cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tcp::kSmem));
        MASW_CUDA_TRY(mem, cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                cudaSharedmemCarveoutMaxShared));
        configured[mem->device & 63] = true;
    }
    MASW_CUDA_TRY(mem, masw_launch(prefill_kernel, dim3(tiles, n_q_heads), dim3(128), tcp::kSmem, st, 1, p));
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
