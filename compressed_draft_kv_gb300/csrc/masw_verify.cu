// Target verify attention over an uncompressed cache ([EN] §3.3 Algorithm 2):
// Lq query positions per sequence, causal inside the block, GQA.
//
// Like the draft prefill this is a dense contraction (the Lq*G query rows of a
// kv head share every K/V row: 24 flop per byte at Lq = 6, G = 4), so it runs
// on the fifth-generation tensor cores with TMA and tensor memory (the
// prefill's machinery): per (key split, kv head, sequence) one CTA streams its
// keys in blocks of 64 and keeps S, O and Q in tensor memory; splits over the
// key axis are merged by split_epilogue.
#include "masw_internal.cuh"
#include "masw_splits.h"
#include "masw_tc.cuh"

#include <atomic>

#include <cstring>

namespace masw {

constexpr int kVD = 128;             // head_dim
constexpr int kVMaxSplit = 64;       // key splits per (sequence, kv head) at most
constexpr int kVMaxNQ = 32;          // query rows (Lq * G) per (sequence, kv head) at most

// ---------------------------------------------------------------------------
// Verify on fifth-generation tensor cores.  One CTA per (key split, kv head,
// sequence), 192 threads.  The pair's NQ = Lq * G <= 32 query rows (row n is
// position n / G, head h * G + n % G) are stored four times in tensor memory,
// at lanes 32 w + n for w = 0..3, so S = Q K^T (M = 128, N = 64 keys) yields
// every score four times, once in each warp's lane quarter.  Softmax warp w
// handles only columns 16 w .. 16 w + 15 of each block: its rows of P are zero
// elsewhere, so the one O += P V MMA (N = 128) accumulates four partial
// outputs over disjoint keys, each with its own running max and sum, merged
// at the end.  This spreads the exponentials over the four SM sub-partitions
// (a single softmax warp holding all 64 columns left three of them idle).
// Lane 0 of warp 4 loads K (TMA) and issues S; lane 0 of warp 5 loads V and
// issues P V.  The split partials are merged by split_epilogue.  One CTA per SM
// (256 tensor-memory columns, 192 KB of shared memory): five K and five V stages
// keep four blocks of each in flight, and two P buffers let the softmax of
// block j+1 write its P while P V of block j still reads the other (fewer,
// deeper streams measured faster than two CTAs per SM with three stages).
// ---------------------------------------------------------------------------
namespace vtc {
using namespace tc;
constexpr int kBM = 128;                         // MMA rows = tensor-memory lanes
constexpr int kBN = 64;                          // keys per block
constexpr int kD = 128;                          // head_dim
constexpr int kStages = 5;                       // K and V stages (one CTA per SM)
constexpr uint32_t kKVBytes = kBN * kD * 2;      // 2 panels of 64 rows x 128 B
constexpr uint32_t kPBytes = kBM * kBN * 2;      // a P buffer: 1 panel of 128 rows x 128 B
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kStages * kKVBytes;
constexpr uint32_t kOffP = kOffV + kStages * kKVBytes;
constexpr uint32_t kSmem = kOffP + 2 * kPBytes;  // two P buffers; the barriers are static shared memory
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 0;                    // O: columns [0, 128)
constexpr uint32_t kColS = 128;                  // S: columns [128, 192)
constexpr uint32_t kColQ = 192;                  // Q (bf16 pairs, the A operand of S): [192, 256)
// instruction descriptors (kind::f16): f32 accumulator, bf16 A and B, M = 128;
// S: N = 64, A (Q, tensor memory) and B (K) K-major; O: N = 128, B (V) MN-major
constexpr uint32_t kIdescBase = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBM >> 4) << 24);
constexpr uint32_t kIdescS = kIdescBase | ((uint32_t)(kBN >> 3) << 17);
constexpr uint32_t kIdescO = kIdescBase | (1u << 16) | ((uint32_t)(kD >> 3) << 17);
__device__ __forceinline__ constexpr int bar_k(int s) { return s; }             // K stage landed (TMA)
__device__ __forceinline__ constexpr int bar_v(int s) { return kStages + s; }   // V stage landed (TMA)
constexpr int kBarS = 2 * kStages;   // S = Q K^T done (MMA commit)
constexpr int kBarSFree = kBarS + 1; // the four softmax warps have read S (4 arrivals)
constexpr int kBarQ = kBarS + 2;     // the four softmax warps have stored Q in tensor memory (4 arrivals)
constexpr int kBarDone = kBarS + 3;  // every S MMA done (early exit only)
constexpr int kBarDoneV = kBarS + 4; // every PV MMA done (early exit only)
// P buffer b written and O rescaled (4 arrivals); the PV MMA that read it done (commit)
__device__ __forceinline__ constexpr int bar_pfull(int b) { return kBarS + 5 + b; }
__device__ __forceinline__ constexpr int bar_pfree(int b) { return kBarS + 7 + b; }
constexpr int kNumBars = kBarS + 9;
// merge layout in the idle stage buffers after the loop: four partial O rows
// per query row, their (max, sum), the merged rows and (max, sum)
constexpr uint32_t kOffPartO = 0;                                  // [4][kVMaxNQ][128] f32
constexpr uint32_t kOffPartML = kOffPartO + 4 * kVMaxNQ * kD * 4;  // [2][4][kVMaxNQ] f32
constexpr uint32_t kOffML = kOffPartML + 2 * 4 * kVMaxNQ * 4;      // [2][kVMaxNQ] f32
constexpr uint32_t kOffCO = kOffP;                                 // [kVMaxNQ][128] f32
static_assert(kOffML + 2 * kVMaxNQ * 4 <= kOffP && kVMaxNQ * kD * 4 <= kPBytes, "merge does not fit");
}  // namespace vtc

struct VerifyTcParams {
    CUtensorMap tm_k;         // K cache as [B*Hkv][Tmax][128] bf16, boxes of 64 x 64 x 1
    CUtensorMap tm_v;
    const __nv_bfloat16* q;   // [B][Lq][Hq][128]
    const int* kv_len;        // [B]
    float* o;                 // [B][Lq][Hq][128]
    float* lse;               // [B][Lq][Hq] or null
    float* part;              // [B*Hkv][n_split][NQ][D+2]
    unsigned* tickets;        // [B*Hkv]
    int* status;              // MASW_ETIMEOUT if a bounded wait gave up
    int B, Lq, Hq, Hkv, G, NQ, Tmax, n_split;
    float scale_log2;
};

__global__ void __launch_bounds__(192, 1) verify_tc_kernel(const __grid_constant__ VerifyTcParams p) {
    using namespace vtc;
    extern __shared__ __align__(1024) uint8_t vsmem[];
    __shared__ uint64_t bars[kNumBars];
    __shared__ uint32_t tslot;
    __shared__ int abort_store;
    volatile int* abort_flag = &abort_store;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sb = smem_u32(vsmem);
    auto bar_at = [&](int i) { return smem_u32(bars + i); };
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int G = p.G, NQ = p.NQ;

    pdl_wait();
    pdl_trigger();
    const int n_keys = p.kv_len[b];
    const int chunk = ((n_keys + p.n_split - 1) / p.n_split + kBN - 1) / kBN * kBN;
    const int k0 = imin(n_keys, split * chunk);
    const int k1 = imin(n_keys, k0 + chunk);
    const int nblk = (k1 - k0 + kBN - 1) / kBN;
    const int head_row = b * p.Hkv + h;          // third coordinate of the cache tensor maps

    // softmax warps 0-3: this lane's query row (copy `warp`) and the first key
    // it may not see
    const bool live = warp < 4 && lane < NQ;
    const int jpos = lane / G;
    const int lim = live ? imin(k1, n_keys - p.Lq + 1 + jpos) : k0;
    uint4 qreg[16];
    if (warp < 4) {
        const uint4* qp = reinterpret_cast<const uint4*>(
            p.q + (((size_t)b * p.Lq + (live ? jpos : 0)) * p.Hq + (size_t)h * G + (live ? lane % G : 0)) * kD);
#pragma unroll
        for (int c = 0; c < 16; ++c) qreg[c] = live ? __ldg(qp + c) : make_uint4(0u, 0u, 0u, 0u);
    }
    const bool misaligned = (sb & 1023u) != 0u;
    if (__syncthreads_or(tid == 0 && misaligned)) {
        if (tid == 0) atomicExch(p.status, MASW_EINVAL);
        return;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tslot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i)
            mbar_init(bars + i, (i == kBarSFree || i == bar_pfull(0) || i == bar_pfull(1) || i == kBarQ) ? 4 : 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;

    if (warp >= 4) {
        if (lane == 0 && nblk > 0) {
            const bool is_v = warp == 5;
            int li = 0, lw = 0;   // blocks whose load was issued / waited
            auto load = [&](int blk) {
                const int st = blk % kStages;
                const int bi = is_v ? bar_v(st) : bar_k(st);
                const uint32_t dst = sb + (is_v ? kOffV : kOffK) + st * kKVBytes;
                const CUtensorMap* m = is_v ? &p.tm_v : &p.tm_k;
                mbar_expect_tx(bars + bi, kKVBytes);
                tma_load_3d(dst, m, 0, k0 + blk * kBN, head_row, bar_at(bi));
                tma_load_3d(dst + kKVBytes / 2, m, 64, k0 + blk * kBN, head_row, bar_at(bi));
                li = blk + 1;
            };
            for (int blk = 0; blk < imin(kStages - 1, nblk); ++blk) load(blk);
            bool ok = true;
            if (!is_v) {
                ok = wait_or_abort(bars + kBarQ, 0, abort_flag, p.status);
                for (int j = 0; ok && j < nblk; ++j) {
                    const int st = j % kStages;
                    ok = wait_or_abort(bars + bar_k(st), (uint32_t)(j / kStages) & 1u, abort_flag, p.status);
                    if (ok) lw = j + 1;
                    // single S buffer: the softmax must have read S(j-1)
                    if (ok && j >= 1) ok = wait_or_abort(bars + kBarSFree, (uint32_t)(j - 1) & 1u, abort_flag, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t bd0 = sw128_desc(sb + kOffK + st * kKVBytes, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk)
                        umma_bf16_ts(tmem + kColS, tmem + kColQ + kk * 8,
                                     bd0 + (uint64_t)(((kk >> 2) * (kKVBytes / 2) + (kk & 3) * 32) >> 4), kIdescS,
                                     kk > 0 ? 1u : 0u);
                    umma_commit(bar_at(kBarS));
                    // K(j+kStages-1) takes the stage of K(j-1), whose S the softmax has read
                    if (j + kStages - 1 < nblk) load(j + kStages - 1);
                }
            } else {
                for (int j = 0; ok && j < nblk; ++j) {
                    const int st = j % kStages, pb = j & 1;
                    ok = wait_or_abort(bars + bar_pfull(pb), (uint32_t)(j >> 1) & 1u, abort_flag, p.status);
                    if (ok) {
                        ok = wait_or_abort(bars + bar_v(st), (uint32_t)(j / kStages) & 1u, abort_flag, p.status);
                        if (ok) lw = j + 1;
                    }
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t a0 = sw128_desc(sb + kOffP + pb * kPBytes, 16, 1024);
                    const uint64_t v0 = sw128_desc(sb + kOffV + st * kKVBytes, kKVBytes / 2, 1024);
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        umma_bf16(tmem + kColO, a0 + (uint64_t)((kk * 32) >> 4), v0 + (uint64_t)((kk * 2048) >> 4),
                                  kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(bar_at(bar_pfree(pb)));
                    // V(j+kStages-1) takes the stage of V(j-1) once PV(j-1) is done
                    // (the next completion of that P buffer needs P(j+1): no phase is skipped)
                    if (j + kStages - 1 < nblk) {
                        if (j >= 1)
                            ok = wait_or_abort(bars + bar_pfree(pb ^ 1), (uint32_t)((j - 1) >> 1) & 1u, abort_flag,
                                               p.status);
                        if (!ok) break;
                        load(j + kStages - 1);
                    }
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
        // ------- softmax warp w: lane n owns copy w of query row n, columns 16 w .. 16 w + 15 -------
        const int w = warp;
        const uint32_t lane_off = (uint32_t)(w * 32) << 16;
        const uint32_t t_o = tmem + kColO + lane_off;
        // Q row -> tensor memory (zeros for lanes past NQ), the A operand of S
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            uint32_t qv[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 x = qreg[hh * 8 + c];
                qv[4 * c] = x.x;
                qv[4 * c + 1] = x.y;
                qv[4 * c + 2] = x.z;
                qv[4 * c + 3] = x.w;
            }
            tmem_st32(tmem + kColQ + lane_off + hh * 32, qv);
        }
        // this row's P outside the warp's 16 columns stays zero: written once per buffer
        const uint32_t prow = sb + kOffP + (uint32_t)(w * 32 + lane) * 128u;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            if ((c >> 1) != w) {
                st_shared_v4(prow + ((uint32_t)(c ^ (lane & 7)) << 4), 0u, 0u, 0u, 0u);
                st_shared_v4(prow + kPBytes + ((uint32_t)(c ^ (lane & 7)) << 4), 0u, 0u, 0u, 0u);
            }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(kBarQ));
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < nblk; ++j) {
            if (!__all_sync(0xffffffffu, wait_or_abort(bars + kBarS, (uint32_t)j & 1u, abort_flag, p.status))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[16];
            tmem_ld16(tmem + kColS + lane_off + w * 16, sv);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_at(kBarSFree));

            // visible columns of this warp's 16 for this row: [0, e_hi) (causal limit)
            const int key0 = k0 + j * kBN + w * 16;
            const int e_hi = imin(16, imax(0, lim - key0));
            float x[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) x[e] = e < e_hi ? __uint_as_float(sv[e]) : -INFINITY;
            const float mx = fmax3(fmax3(fmax3(x[0], x[1], x[2]), fmax3(x[3], x[4], x[5]), fmax3(x[6], x[7], x[8])),
                                   fmax3(x[9], x[10], x[11]), fmax3(fmax3(x[12], x[13], x[14]), x[15], x[15]));
            // the running max moves only when it grows by more than 2^8, so the O
            // rescale is rare (exact: the partial is relative to m_run)
            float alpha = 1.f;
            const float m_new = fmaxf(m_run, mx * p.scale_log2);
            if (m_new > m_run + 8.f) {
                alpha = ex2_approx(m_run - m_new);
                m_run = m_new;
            }
            const float nmref = m_run == -INFINITY ? 0.f : -m_run;
            const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nm2 = f2_pack(nmref, nmref);
            uint32_t pk[8];
            uint64_t sum2[2] = {0, 0};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float a0, a1v;
                f2_unpack(f2_fma(f2_pack(x[2 * e], x[2 * e + 1]), sc2, nm2), a0, a1v);
                const float p0 = ex2_approx(a0), p1 = ex2_approx(a1v);
                sum2[e & 1] = f2_add(sum2[e & 1], f2_pack(p0, p1));
                pk[e] = pack_bf16(p0, p1);
            }
            float sum_lo, sum_hi;
            f2_unpack(f2_add(sum2[0], sum2[1]), sum_lo, sum_hi);
            const bool resc = alpha != 1.f && l_run > 0.f;
            l_run = l_run * alpha + (sum_lo + sum_hi);

            // P buffer j&1 is free once PV(j-2) is done; O is rescaled only after
            // PV(j-1) (the next completion of either buffer needs a P not yet written)
            const int pb = j & 1;
            if (j >= 2) {
                if (!__all_sync(0xffffffffu, wait_or_abort(bars + bar_pfree(pb), (uint32_t)((j - 2) >> 1) & 1u,
                                                           abort_flag, p.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            const bool any_resc = __any_sync(0xffffffffu, resc);
            if (any_resc && j >= 1) {
                if (!__all_sync(0xffffffffu, wait_or_abort(bars + bar_pfree(pb ^ 1), (uint32_t)((j - 1) >> 1) & 1u,
                                                           abort_flag, p.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (any_resc) {
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
            // this warp's two 16-byte chunks of the row (128-byte swizzle)
            const uint32_t pr = prow + pb * kPBytes;
            st_shared_v4(pr + ((uint32_t)((2 * w) ^ (lane & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
            st_shared_v4(pr + ((uint32_t)((2 * w + 1) ^ (lane & 7)) << 4), pk[4], pk[5], pk[6], pk[7]);
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_at(bar_pfull(pb)));
        }
        if (ok && nblk > 0)
            ok = __all_sync(0xffffffffu, wait_or_abort(bars + bar_pfree((nblk - 1) & 1),
                                                       (uint32_t)((nblk - 1) >> 1) & 1u, abort_flag, p.status));
        tc_fence_after();
        // this copy's partial O row and (max, sum) -> the stage buffers (idle now)
        float* po = reinterpret_cast<float*>(vsmem + kOffPartO) + ((size_t)w * kVMaxNQ + lane) * kD;
        float* pml = reinterpret_cast<float*>(vsmem + kOffPartML);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t ov[32];
            if (nblk > 0) {
                tmem_ld32(t_o + c * 32, ov);
                tmem_wait_ld();
            }
            if (live) {
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(po + c * 32 + e) =
                        nblk > 0 ? make_float4(__uint_as_float(ov[e]), __uint_as_float(ov[e + 1]),
                                               __uint_as_float(ov[e + 2]), __uint_as_float(ov[e + 3]))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if (live) {
            pml[w * kVMaxNQ + lane] = m_run;
            pml[(4 + w) * kVMaxNQ + lane] = l_run;
        }
    }
    tc_fence_before();
    // every thread reads the flag: one that set it counts itself in
    const bool aborted = __syncthreads_or(*abort_flag != 0);
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    if (aborted) return;   // outputs of this call are undefined; p.status says why
    // merge the four copies of each row: M = max_w m_w, weights 2^(m_w - M)
    const float* pml = reinterpret_cast<const float*>(vsmem + kOffPartML);
    const float* po = reinterpret_cast<const float*>(vsmem + kOffPartO);
    float* cm = reinterpret_cast<float*>(vsmem + kOffML);
    float* cl = cm + kVMaxNQ;
    float* co = reinterpret_cast<float*>(vsmem + kOffCO);
    for (int i = tid; i < NQ * kD; i += blockDim.x) {
        const int n = i / kD, d = i % kD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, pml[w * kVMaxNQ + n]);
        float a = 0.f, l = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float mw = pml[w * kVMaxNQ + n];
            const float e = mw == -INFINITY ? 0.f : ex2_approx(mw - M);
            a += e * po[((size_t)w * kVMaxNQ + n) * kD + d];
            l += e * pml[(4 + w) * kVMaxNQ + n];
        }
        co[i] = a;
        if (d == 0) {
            cm[n] = M;
            cl[n] = l;
        }
    }
    __syncthreads();
    EpiOut out;
    out.o = p.o + ((size_t)b * p.Lq * p.Hq + (size_t)h * G) * kD;
    out.lse = p.lse ? p.lse + (size_t)b * p.Lq * p.Hq + (size_t)h * G : nullptr;
    out.rows_per_group = G;
    out.o_row_stride = kD;
    out.o_group_stride = p.Hq * kD;
    out.lse_row_stride = 1;
    out.lse_group_stride = p.Hq;
    out.o_alt = nullptr;
    out.lse_alt = nullptr;
    out.alt_from = -1;
    float* part = p.part + (size_t)head_row * p.n_split * NQ * (kD + 2);
    split_epilogue<kD>(NQ, cm, cl, co, out, part, p.tickets + head_row, split, p.n_split, nullptr);
}

// Resident tensor-core verify CTAs per SM: the occupancy query, and the bound
// from the kernel's attributes (shared memory with the per-block reserve), at
// most two (256 tensor-memory columns each); one with the current stages.
static int verify_tc_occupancy() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (!cache[dev].load(std::memory_order_acquire)) {
        int n = 0;
        if (cudaFuncSetAttribute(verify_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, vtc::kSmem) !=
                cudaSuccess ||
            cudaFuncSetAttribute(verify_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, verify_tc_kernel, 192, vtc::kSmem) != cudaSuccess) {
            cudaGetLastError();
            n = 1;
        }
        cudaFuncAttributes fa;
        int smem_sm = 0, smem_rsv = 0;
        if (cudaFuncGetAttributes(&fa, verify_tc_kernel) == cudaSuccess &&
            cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev) == cudaSuccess) {
            const long long per = (long long)vtc::kSmem + fa.sharedSizeBytes + smem_rsv;
            n = imax(n, (int)(smem_sm / per));
        } else {
            cudaGetLastError();
        }
        cache[dev].store(imax(1, imin(n, 2)), std::memory_order_release);
    }
    return cache[dev].load(std::memory_order_acquire);
}

// Split count shared by the launcher and the workspace query: one wave of the
// resident CTA slots, at least 256 keys per split (masw_splits.h).
static int verify_splits(int B, int Hkv, int Tmax, int num_sms) {
    return verify_split_plan(B * Hkv, verify_tc_occupancy() * num_sms, Tmax, kVMaxSplit);
}

static int num_sms_current(int* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MASW_ECUDA;
    if (cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MASW_ECUDA;
    return MASW_OK;
}

static size_t verify_part_bytes(int B, int Hkv, int NQ, int n_split) {
    return verify_partial_bytes(B * Hkv, NQ, kVD, n_split);
}

}  // namespace masw

using namespace masw;

static int verify_check(int B, int Lq, int Hq, int Hkv, int D, int Tmax) {
    if (B < 1 || Lq < 1 || Hq < 1 || Hkv < 1 || Tmax < Lq) return MASW_EINVAL;
    if (D != kVD) return MASW_EINVAL;
    if (Hq % Hkv) return MASW_EINVAL;
    if ((Hq / Hkv) * Lq > kVMaxNQ) return MASW_EINVAL;
    if (B > 65535 || Hkv > 65535) return MASW_EINVAL;
    return MASW_OK;
}

extern "C" int masw_verify_workspace_bytes(int B, int Lq, int Hq, int Hkv, int D, int Tmax, size_t* bytes) {
    if (!bytes) return masw_set_error(nullptr, MASW_EINVAL, "bytes is NULL");
    int rc = verify_check(B, Lq, Hq, Hkv, D, Tmax);
    if (rc) return masw_set_error(nullptr, rc, "unsupported verify sizes (D must be 128, Lq*Hq/Hkv <= 32)");
    int sms = 0;
    if (num_sms_current(&sms)) return masw_set_error(nullptr, MASW_ECUDA, "cannot query the current device");
    const int NQ = (Hq / Hkv) * Lq;
    const int n_split = verify_splits(B, Hkv, Tmax, sms);
    *bytes = verify_part_bytes(B, Hkv, NQ, n_split) + (size_t)B * Hkv * sizeof(unsigned) + 16;
    return MASW_OK;
}

// K or V cache [B][Hkv][Tmax][128] bf16 as a 3-d tensor [B*Hkv][Tmax][128]
// (head_dim innermost), boxes of 64 x 64 x 1 with the 128-byte swizzle the MMA
// descriptors use; rows past Tmax read as zeros
static bool make_cache_map(CUtensorMap* map, const void* base, int Tmax, int heads_total) {
    const cuuint64_t dims[3] = {128, (cuuint64_t)Tmax, (cuuint64_t)heads_total};
    const cuuint64_t strides[2] = {256, (cuuint64_t)Tmax * 256};
    const cuuint32_t box[3] = {64, 64, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return tma_encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor-core verify kernel on (q, caches, scratch); scratch = [partials
// (part_bytes)][tickets, one per (sequence, kv head)][status word].
static int launch_verify_tc(const void* q, const void* k_cache, const void* v_cache, const int* kv_len, int B,
                            int Lq, int Hq, int Hkv, int Tmax, float scale_log2, float* o, float* lse, void* scratch,
                            size_t part_bytes, int n_split, cudaStream_t st, const char* who) {
    if (!tma_encode_fn()) return masw_set_error(nullptr, MASW_ECUDA, std::string(who) + ": cuTensorMapEncodeTiled is unavailable");
    if ((long long)B * Hkv > 0x7fffffff || (long long)Tmax * 256 >= (1ll << 40))
        return masw_set_error(nullptr, MASW_EINVAL, std::string(who) + ": cache too large for a tensor map");
    VerifyTcParams prm;
    std::memset(&prm, 0, sizeof(prm));
    if (!make_cache_map(&prm.tm_k, k_cache, Tmax, B * Hkv) || !make_cache_map(&prm.tm_v, v_cache, Tmax, B * Hkv))
        return masw_set_error(nullptr, MASW_EINVAL, std::string(who) + ": cannot describe the caches as TMA tensors");
    prm.q = (const __nv_bfloat16*)q;
    prm.kv_len = kv_len;
    prm.o = o;
    prm.lse = lse;
    prm.part = (float*)scratch;
    prm.tickets = (unsigned*)((uint8_t*)scratch + part_bytes);
    prm.status = (int*)(prm.tickets + (size_t)B * Hkv);
    prm.B = B;
    prm.Lq = Lq;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.G = Hq / Hkv;
    prm.NQ = prm.G * Lq;
    prm.Tmax = Tmax;
    prm.n_split = n_split;
    prm.scale_log2 = scale_log2;
    verify_tc_occupancy();   // sets the kernel's shared-memory attributes once per device
    const cudaError_t e =
        masw_launch(verify_tc_kernel, dim3(n_split, Hkv, B), dim3(192), vtc::kSmem, st, 1, prm);
    if (e != cudaSuccess) return masw_set_error(nullptr, MASW_ECUDA, std::string(who) + ": " + cudaGetErrorString(e));
    return MASW_OK;
}

extern "C" int masw_verify_attn(const void* q, const void* k_cache, const void* v_cache, const int* kv_len, int B,
                                int Lq, int Hq, int Hkv, int D, int Tmax, int dtype, float scale, float* o,
                                float* lse, void* workspace, size_t workspace_bytes, masw_stream_t stream) {
    if (!q || !k_cache || !v_cache || !kv_len || !o || !workspace)
        return masw_set_error(nullptr, MASW_EINVAL, "verify: NULL pointer");
    if (dtype != MASW_BF16) return masw_set_error(nullptr, MASW_EINVAL, "verify: only MASW_BF16 is supported");
    int rc = verify_check(B, Lq, Hq, Hkv, D, Tmax);
    if (rc) return masw_set_error(nullptr, rc, "verify: unsupported sizes (D must be 128, Lq*Hq/Hkv <= 32)");
    if (((uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache | (uintptr_t)workspace) & 15)
        return masw_set_error(nullptr, MASW_EINVAL, "verify: q, caches and workspace must be 16-byte aligned");
    if (((uintptr_t)o | (uintptr_t)lse | (uintptr_t)kv_len) & 3)
        return masw_set_error(nullptr, MASW_EINVAL, "verify: o, lse and kv_len must be 4-byte aligned");
    int sms = 0;
    if (num_sms_current(&sms)) return masw_set_error(nullptr, MASW_ECUDA, "verify: cannot query the device");
    const int G = Hq / Hkv, NQ = G * Lq;
    const int n_split = verify_splits(B, Hkv, Tmax, sms);
    const size_t partb = verify_part_bytes(B, Hkv, NQ, n_split);
    if (workspace_bytes < partb + (size_t)B * Hkv * sizeof(unsigned) + 16)
        return masw_set_error(nullptr, MASW_EINVAL, "verify: workspace too small");
    // the tickets are zero on entry (zero-filled workspace, reset by the last
    // CTA of each pair in every call): no memset node between calls, so
    // consecutive verify launches keep their programmatic overlap
    const float sl2 = (scale > 0.f ? scale : 1.0f / sqrtf((float)D)) * 1.4426950408889634f;
    return launch_verify_tc(q, k_cache, v_cache, kv_len, B, Lq, Hq, Hkv, Tmax, sl2, o, lse, workspace, partb, n_split,
                            (cudaStream_t)stream, "verify");
}

// ---------------------------------------------------------------------------
// Verify attention that allocates nothing.
//
// masw_verify_attn needs a workspace from its caller.  Some callers cannot
// provide one: code that only ever receives input and output pointers (a
// plugin slot in another engine, say), code whose device memory is all owned
// by a framework's own allocator, or a latency-critical loop where a
// cudaMalloc -- which can synchronise the whole device -- is not acceptable.
// For them the split partials and tickets live in the array below, which is
// part of the library image: every GPU that loads the library holds these
// 4 MiB + 16 KiB until the process exits.
//
// Limits: B * Hkv <= kNoAllocMaxPairs.  The partials of the usual split count
// fit in kNoAllocPartBytes on any GPU with up to about 250 SMs (the split count
// stops at one CTA per SM, and NQ <= 32 rows of 130 floats per split): on a
// 152-SM GB300 they take at most ~2.5 MB.  The loop that lowers the split count
// when they would not fit is a guard for larger devices.
// All calls share the array and each leaves its partials in it; the tickets
// and the status word are cleared on the stream at the start of every call,
// and the status word can be copied out to the caller after the kernel.  Two
// calls that overlap on the GPU (different streams, or different host threads)
// race on the array and give wrong results: serialise them.
// ---------------------------------------------------------------------------
namespace masw {
constexpr size_t kNoAllocPartBytes = (size_t)4 << 20;
constexpr int kNoAllocMaxPairs = 4096;
constexpr size_t kNoAllocBytes = kNoAllocPartBytes + (size_t)kNoAllocMaxPairs * sizeof(unsigned) + 16;
}  // namespace masw

static __device__ __align__(256) uint8_t g_noalloc_scratch[masw::kNoAllocBytes];

// Device address of g_noalloc_scratch in the current context.  In host code the
// array's name is only a host-side stand-in; the kernel must be given this
// address.  It is looked up on every call (a table lookup in the runtime, no
// allocation) rather than cached, so it stays right when a context is torn
// down and re-created (cudaDeviceReset), which reloads the module and moves
// the array.
static int noalloc_scratch(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return masw_set_error(nullptr, MASW_ECUDA,
                              std::string("verify_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    }
    *out = p;
    return MASW_OK;
}

extern "C" int masw_verify_attn_noalloc(const void* q, const void* k_cache, const void* v_cache, const int* kv_len,
                                        int B, int Lq, int Hq, int Hkv, int D, int Tmax, int dtype, float scale,
                                        float* o, float* lse, int* status, masw_stream_t stream) {
    if (!q || !k_cache || !v_cache || !kv_len || !o)
        return masw_set_error(nullptr, MASW_EINVAL, "verify_noalloc: NULL pointer");
    if (dtype != MASW_BF16) return masw_set_error(nullptr, MASW_EINVAL, "verify_noalloc: only MASW_BF16 is supported");
    int rc = verify_check(B, Lq, Hq, Hkv, D, Tmax);
    if (rc) return masw_set_error(nullptr, rc, "verify_noalloc: unsupported sizes (D must be 128, Lq*Hq/Hkv <= 32)");
    if ((size_t)B * Hkv > (size_t)kNoAllocMaxPairs)
        return masw_set_error(nullptr, MASW_EINVAL,
                              "verify_noalloc: B * Hkv = " + std::to_string((size_t)B * Hkv) +
                                  " exceeds the static scratch limit of " + std::to_string(kNoAllocMaxPairs) +
                                  "; use masw_verify_attn with a workspace");
    if (((uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache) & 15)
        return masw_set_error(nullptr, MASW_EINVAL, "verify_noalloc: q and caches must be 16-byte aligned");
    if (((uintptr_t)o | (uintptr_t)lse | (uintptr_t)kv_len | (uintptr_t)status) & 3)
        return masw_set_error(nullptr, MASW_EINVAL, "verify_noalloc: o, lse, kv_len and status must be 4-byte aligned");
    int sms = 0;
    if (num_sms_current(&sms)) {
        cudaGetLastError();
        return masw_set_error(nullptr, MASW_ECUDA, "verify_noalloc: cannot query the current device");
    }
    void* scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch))) return rc;
    const int G = Hq / Hkv, NQ = G * Lq;
    const int n_split = noalloc_split_plan(B * Hkv, NQ, kVD, Tmax, verify_tc_occupancy() * sms, kVMaxSplit,
                                           kNoAllocPartBytes);
    cudaStream_t st = (cudaStream_t)stream;
    // the library's static array cannot be re-zeroed by the caller after a
    // failed call, so this variant clears the tickets and the status word on
    // the stream at the start of every call
    cudaError_t e = cudaMemsetAsync((uint8_t*)scratch + kNoAllocPartBytes, 0,
                                    (size_t)kNoAllocMaxPairs * sizeof(unsigned) + 16, st);
    if (e != cudaSuccess)
        return masw_set_error(nullptr, MASW_ECUDA, std::string("verify_noalloc: ") + cudaGetErrorString(e));
    const float sl2 = (scale > 0.f ? scale : 1.0f / sqrtf((float)D)) * 1.4426950408889634f;
    rc = launch_verify_tc(q, k_cache, v_cache, kv_len, B, Lq, Hq, Hkv, Tmax, sl2, o, lse, scratch, kNoAllocPartBytes,
                          n_split, st, "verify_noalloc");
    if (rc || !status) return rc;
    // the status word follows the B * Hkv tickets (launch_verify_tc's layout)
    const void* word = (const uint8_t*)scratch + kNoAllocPartBytes + (size_t)B * Hkv * sizeof(unsigned);
    e = cudaMemcpyAsync(status, word, sizeof(int), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess)
        return masw_set_error(nullptr, MASW_ECUDA, std::string("verify_noalloc: status copy: ") + cudaGetErrorString(e));
    return MASW_OK;
}
