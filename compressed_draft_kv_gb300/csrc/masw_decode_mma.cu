// Tensor-core split-KV decode attention for bf16 pools: draft attention over
// the MASW working memory ([EN] §3.1 Eq. 4 with Eq. 2 of §2.3), the slot-write
// query under the structured mask ([EN] §3.2 Algorithm 1), and full-KV
// decode over the contrast cache.
//
// With grouped-query attention the G = Hq/Hkv query heads of a kv head read
// the same K/V rows, so each 16-key tile is a small dense contraction
// [16 keys x D] x [D x G].  It runs on mma.sync m16n8k16 (bf16 in, fp32
// accumulate) with KEYS as the M dimension and the G <= 8 query heads as the N
// tile: S^T = K Q^T from ldmatrix fragments, online softmax per query column in
// the log2 domain, P^T moved from the accumulator layout into a B operand with
// movmatrix, and O^T += V^T P^T with ldmatrix.trans fragments of the same V
// stage.  About 150 warp instructions per 16 keys, against ~700 for the same
// work on CUDA cores with shuffle reductions, so the kernel keeps up with HBM
// at few warps per SM.
//
// Grid (n_split, Hkv, rows), 128 threads, one wave: n_split fills the resident
// CTA slots of the GPU.  K/V rows of the CTA's share of the logical key list
// are copied with 16-byte cp.async into XOR-swizzled shared-memory stages
// (NST in flight); rows come from up to five contiguous segments (sink, the
// window in one or two runs, the slot chain, a self-attended slot) and are
// never gathered in HBM.  Split partials are merged by split_epilogue.
#include "masw_internal.cuh"

#include <atomic>
#include <climits>

#include <cooperative_groups.h>
#include <cstring>

namespace cg = cooperative_groups;

namespace masw {

// NST stages of K/V in shared memory: 2 (64 KB, three CTAs fit on an SM, so the
// next launch's CTAs start copying while this one merges) or 3 (96 KB, more
// bytes in flight for CTAs that each stream a long run of keys)
template <int D, int NST_>
struct MmaCfg {
    static constexpr int KPS = 64;               // keys per stage (16 per warp)
    static constexpr int NST = NST_;
    static constexpr int CH = D / 8;             // 16-byte chunks per row
    static constexpr int ROWB = D * 2;           // bytes per bf16 row
    static constexpr int STAGE = 2 * KPS * ROWB; // K then V
    static constexpr int SMEM = NST * STAGE;
    static constexpr int KS = D / 16;            // k-steps of Q.K, m-tiles of P.V
    static_assert((2 * 4 * 8 + 4 * 8 * (D + 8) + 2 * 8 + 8 * D + epilogue_scratch_floats(8, kMaxSplit)) * 4 <= SMEM,
                  "merge does not fit in the stage buffers");
};

// 2^x by the MUFU instruction (an input of -inf gives 0)
__device__ __forceinline__ float fast_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Distributed shared memory hand-off of the cluster merge: a CTA writes into a
// peer's shared memory with st.async, whose bytes count down the peer's mbarrier
// (complete_tx), so each receiver waits only for the bytes it needs -- no
// cluster-wide barrier after the main loop.
__device__ __forceinline__ uint32_t mapa_rank(uint32_t saddr, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_async_v4(uint32_t raddr, float4 v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     raddr),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rbar)
                 : "memory");
}
__device__ __forceinline__ void st_async_v2(uint32_t raddr, float a, float b, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(raddr),
                 "f"(a), "f"(b), "r"(rbar)
                 : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
// bounded wait on phase 0 of a receive mbarrier, acquiring the peers' writes
__device__ __forceinline__ bool recv_wait(uint64_t* bar, int* err) {
    for (uint32_t i = 0; i < kWaitPolls; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], 0;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(smem_u32(bar))
            : "memory");
        if (ok) return true;
        if (i > 64) __nanosleep(64);
    }
    atomicExch(err, MASW_ETIMEOUT);
    return false;
}

// largest thread-block cluster of the split merge (above 8 needs the
// non-portable cluster-size attribute).  Sizes 14 and 16 were measured slower
// than 12 even where they shorten every CTA's key run, so the plan stops at 12.
constexpr int kMaxClusterSize = 12;

template <int ROWB>
__device__ __forceinline__ uint32_t swz_off(int row, int ch) {
    return (uint32_t)(row * ROWB + ((ch ^ (row & 7)) << 4));
}

// Fused step: store the new token's K/V row of head h, held in shared memory as
// row `row` of a stage (swizzled 16-byte chunks), in its sink or ring row (the
// ring write evicts token t+1-W-R, which no CTA of this launch reads) and in the
// full-KV cache.
template <int ROWB>
__device__ void step_store_row_smem(const DecodeParams& p, int lb, int h, int t, const uint8_t* stage_k,
                                    const uint8_t* stage_v, int row) {
    const int i = t + 1;
    const int prow = i <= p.S ? i - 1 : p.S + ring_row(i, p.S, p.Wc);
    const size_t dst = (((size_t)lb * p.Hkv + h) * p.C + prow) * ROWB;
    const bool to_full = p.full_k != nullptr && i <= p.Tmax;
    const size_t fdst = (((size_t)lb * p.Hkv + h) * p.Tmax + (i - 1)) * (size_t)ROWB;
    for (int c = threadIdx.x; c < ROWB / 16; c += blockDim.x) {
        const uint4 kv = *reinterpret_cast<const uint4*>(stage_k + swz_off<ROWB>(row, c));
        const uint4 vv = *reinterpret_cast<const uint4*>(stage_v + swz_off<ROWB>(row, c));
        *reinterpret_cast<uint4*>((uint8_t*)p.pool_k + dst + c * 16) = kv;
        *reinterpret_cast<uint4*>((uint8_t*)p.pool_v + dst + c * 16) = vv;
        if (to_full) {
            *reinterpret_cast<uint4*>((uint8_t*)p.full_k + fdst + c * 16) = kv;
            *reinterpret_cast<uint4*>((uint8_t*)p.full_v + fdst + c * 16) = vv;
        }
    }
}

// The minimum-blocks bound states the occupancy the plan uses (three CTAs per
// SM with two stages, two with three): it lets ptxas spend registers up to that
// occupancy (about 134 instead of 96), which measured 4-9% faster on GB300.
template <int D, int NST_>
__global__ void __launch_bounds__(128, NST_ == 2 ? 3 : 2) decode_mma_kernel(const __grid_constant__ DecodeParams p) {
    using C = MmaCfg<D, NST_>;
    constexpr int KPS = C::KPS, NST = C::NST, CH = C::CH, ROWB = C::ROWB, KS = C::KS;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Seg segs[5];
    __shared__ int s_start[6];
    __shared__ const uint8_t* s_vk[5];
    __shared__ const uint8_t* s_vv[5];
    __shared__ int s_nseg, s_m_before, s_t, s_respec;
    // cluster merge receive buffers (written by peer CTAs with st.async; never
    // aliased with the stages): (max, sum) per (rank, row), the o slices, and the
    // mbarrier their bytes count down
    __shared__ __align__(16) float2 r_ml[kMaxClusterSize * 8];
    __shared__ __align__(16) float r_o[8 * D + 4 * kMaxClusterSize];
    __shared__ uint64_t r_bar;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, h = blockIdx.y, z = blockIdx.z;
    const int b = (p.mode == kDevModeSlot) ? (int)p.seq_ids[z] : z;
    const int lb = p.layer * p.B + b;
    const int G = p.Hq / p.Hkv;
    const int si = p.q_slot ? (int)p.slot_of[z] : -1;   // fused slot query of this row, if any
    const int NR = si >= 0 ? 2 * G : G;                  // query columns of this pair
    // The pair's query rows into L2 now: they are read right after the
    // dependency wait, and an L2 prefetch is safe before it (it only warms L2,
    // which the previous kernel's writes update).
    if (tid == 32) {
        prefetch_l2((const uint8_t*)p.q + ((size_t)z * p.Hq + (size_t)h * G) * ROWB, (uint32_t)(G * ROWB));
        if (si >= 0) prefetch_l2((const uint8_t*)p.q_slot + ((size_t)si * p.Hq + (size_t)h * G) * ROWB, (uint32_t)(G * ROWB));
    }
    // cluster merge: rank k finalises elements [k*per, (k+1)*per) of the pair's
    // NR x D output (per a multiple of 4, so 16-byte pushes never straddle two
    // ranks) and receives, from each of the n_split ranks, that slice and the
    // (max, sum) of the NR rows.  The receive mbarrier is initialised here and
    // made visible to the peers by a cluster arrive whose wait comes just before
    // the first push.
    const int per = ((NR * D + p.n_split - 1) / p.n_split + 3) & ~3;
    if (p.cluster) {
        if (tid == 0) {
            const int slice = imax(0, imin(per, NR * D - split * per));
            mbar_init(&r_bar, 1);
            mbar_expect_tx(&r_bar, (uint32_t)(p.n_split * (slice * 4 + NR * 8)));
            fence_mbar_init();
        }
        cluster_arrive_relaxed();
    }
    // Segment table, built speculatively from the host mirror's counters (no
    // global read before the first copies) and verified against the device
    // counters, which are read after the dependency wait but compared only
    // after the main loop; in the rare case they differ (the previous kernel
    // changed this head's counters, or a graph replays from another state) the
    // table is rebuilt and the loop runs again.
    const size_t ci = (size_t)lb * p.Hkv + h;
    auto build = [&](int t, int mcnt) {
        s_m_before = mcnt;
        s_t = t;
        const int n = build_segments<ROWB>(p, lb, h, z, t, mcnt, segs);
        int acc = 0;
        for (int s = 0; s < n; ++s) {
            s_start[s] = acc;
            s_vk[s] = segs[s].k - (size_t)acc * ROWB;   // row j of the list is s_vk[s] + j*ROWB
            s_vv[s] = segs[s].v - (size_t)acc * ROWB;
            acc += segs[s].len;
        }
        if (n == 0) {
            s_vk[0] = (const uint8_t*)p.pool_k;
            s_vv[0] = (const uint8_t*)p.pool_v;
        }
        s_start[n] = acc;
        s_nseg = n;
    };
    if (tid == 0) build(p.t_spec[z], p.m_spec[z]);
    __syncthreads();

    int nseg = s_nseg;
    int total = s_start[nseg];
    const bool fresh = p.step && ((p.active[z >> 5] >> (z & 31)) & 1u);
    int chunk = (((total + p.n_split - 1) / p.n_split) + 15) & ~15;
    int r0 = imin(total, split * chunk);
    int r1 = imin(total, r0 + chunk);
    int nstage = (r1 - r0 + KPS - 1) / KPS;
    const uint32_t sbase = smem_u32(smem);

    // stage c <- logical rows [r0 + c*KPS, +KPS); rows past r1 are zero-filled.
    // Lanes take consecutive 16-byte chunks of a row (CH lanes per row), so each
    // warp-wide cp.async covers whole rows; a thread's rows are RPP apart and
    // walk the segment list monotonically (vbase[s] = segment base - start*ROWB).
    constexpr int RPP = 128 / CH;             // rows per pass of the CTA
    const int my_row = tid / CH, my_ch = tid % CH;
    auto load_stage = [&](int c) {
        const uint32_t sk = sbase + (uint32_t)(c % NST) * C::STAGE;
        const uint32_t sv = sk + KPS * ROWB;
        const int j0 = r0 + c * KPS + my_row;
        int s = 0;
        while (s + 1 < nseg && j0 >= s_start[s + 1]) ++s;
        int next = s + 1 < nseg ? s_start[s + 1] : 0x7fffffff;
#pragma unroll
        for (int i = 0; i < KPS / RPP; ++i) {
            const int row = my_row + i * RPP;
            const int j = j0 + i * RPP;
            const uint8_t* ks = s_vk[0];
            const uint8_t* vs = s_vv[0];
            int bytes = 0;
            if (j < r1) {
                while (j >= next) {
                    ++s;
                    next = s + 1 < nseg ? s_start[s + 1] : 0x7fffffff;
                }
                ks = s_vk[s] + (size_t)j * ROWB + my_ch * 16;
                vs = s_vv[s] + (size_t)j * ROWB + my_ch * 16;
                bytes = 16;
            }
            cp_async16(sk + swz_off<ROWB>(row, my_ch), ks, bytes);
            cp_async16(sv + swz_off<ROWB>(row, my_ch), vs, bytes);
        }
    };
    // The first stages are copied before the dependency wait when the previous
    // launch wrote no pool row of this layer (p.early) and they hold pool rows
    // only (the new token's row and a self-attended slot come from the caller's
    // buffers, which the previous kernel may still be writing).
    const int n_input = ((p.step && ((p.active[z >> 5] >> (z & 31)) & 1u)) ? 1 : 0) +
                        ((p.mode == kDevModeSlot && p.self_attend) ? 1 : 0);
    const bool early = p.early && imin(r1, r0 + (NST - 1) * KPS) <= total - n_input;
    // With two stages, when the stage after them holds pool rows only too, it
    // fills the other buffer before the wait as well (its own copy group; the
    // first iteration then issues and commits nothing), so the stream does not
    // stall on it after the dependency wait.  (Measured on GB300: 10.3 -> 9.8 us
    // per 36 MB launch; with three stages, whose CTAs stream long runs, it cost
    // 50.0 -> 51.2 us per 272 MB launch, so it is off there.)
    bool pre = NST == 2 && early && nstage >= NST && r0 + NST * KPS <= total - n_input;
    if (early) {
#pragma unroll 1
        for (int c = 0; c < (pre ? NST : NST - 1); ++c) {
            if (c < nstage) load_stage(c);
            cp_async_commit();
        }
    }
    pdl_wait();
    pdl_trigger();

    // Q^T as B fragments: column n < G is query head h*G + n of row z; columns
    // G..2G-1 are the fused slot query's heads; the rest are zero
    uint32_t qb[KS][2];
    {
        const int n = lane >> 2;
        const bool real = n < NR;
        const __nv_bfloat16* qrow =
            n < G ? (const __nv_bfloat16*)p.q + ((size_t)z * p.Hq + (size_t)h * G + n) * D
                  : (real ? (const __nv_bfloat16*)p.q_slot + ((size_t)si * p.Hq + (size_t)h * G + (n - G)) * D
                          : (const __nv_bfloat16*)p.q);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int d = ks * 16 + (lane & 3) * 2;
            qb[ks][0] = real ? *reinterpret_cast<const uint32_t*>(qrow + d) : 0u;
            qb[ks][1] = real ? *reinterpret_cast<const uint32_t*>(qrow + d + 8) : 0u;
        }
    }
    int dev_t = 0, dev_m = 0;                        // thread 0 only: compared after the loop
    if (tid == 0) {
        dev_t = *(volatile const int*)(p.d_t + ci);
        dev_m = *(volatile const int*)(p.d_m + ci);
    }
    if (!early) {
#pragma unroll
        for (int c = 0; c < NST - 1; ++c) {
            if (c < nstage) load_stage(c);
            cp_async_commit();
        }
    }

    // every peer arrived at its start, so this wait is free here and keeps the
    // cluster barrier off the merge's critical path
    if (p.cluster) cluster_wait();                   // every peer's receive mbarrier is initialised

    const float sl2 = p.scale_log2;
    float m_run[2], l_run[2];
    float acc[KS][4];
    for (int attempt = 0;; ++attempt) {
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

        // copy group g holds stage g (with pre, the first iteration commits none)
        for (int c = 0; c < nstage; ++c) {
            if (pre && c == 0)
                cp_async_wait<NST - 1>();
            else
                cp_async_wait<NST - 2>();
            __syncthreads();
            if (!(pre && c == 0)) {
                const int cn = c + NST - 1;   // refill the stage consumed in the previous iteration
                if (cn < nstage) load_stage(cn);
                cp_async_commit();
            }
            const uint32_t sk = sbase + (uint32_t)(c % NST) * C::STAGE;
            const uint32_t sv = sk + KPS * ROWB;
            const int kw = warp * 16;
            const int key_tile = r0 + c * KPS + kw;
            if (key_tile < r1) {
                // two accumulators (even and odd k-steps) halve the dependent MMA chain
                float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(sk + swz_off<ROWB>(kw + (lane & 7) + ((lane >> 3) & 1) * 8, ks * 2 + (lane >> 4)), a0, a1,
                            a2, a3);
                    mma16816((ks & 1) ? s2 : s, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) s[e] += s2[e];
                float x[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) x[e] = s[e] * sl2;
                if (key_tile + 16 > r1) {                   // the split's last, partial tile (warp-uniform)
                    const int key_a = key_tile + (lane >> 2), key_b = key_a + 8;
                    if (key_a >= r1) x[0] = x[1] = -INFINITY;
                    if (key_b >= r1) x[2] = x[3] = -INFINITY;
                }
                float pr[4];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float mx = fmaxf(x[e], x[e + 2]);
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const float m_new = fmaxf(m_run[e], mx);   // finite: key_tile < r1
                    const float alpha = fast_ex2(m_run[e] - m_new);
                    pr[e] = fast_ex2(x[e] - m_new);
                    pr[e + 2] = fast_ex2(x[e + 2] - m_new);
                    l_run[e] = l_run[e] * alpha + pr[e] + pr[e + 2];
                    m_run[e] = m_new;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        acc[mt][e] *= alpha;
                        acc[mt][e + 2] *= alpha;
                    }
                }
                const uint32_t pb0 = movmatrix_t(pack_bf16(pr[0], pr[1]));
                const uint32_t pb1 = movmatrix_t(pack_bf16(pr[2], pr[3]));
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(sv + swz_off<ROWB>(kw + (lane & 7) + (lane >> 4) * 8, mt * 2 + ((lane >> 3) & 1)), a0, a1,
                              a2, a3);
                    mma16816(acc[mt], a0, a1, a2, a3, pb0, pb1);
                }
            }
        }
        cp_async_wait<0>();
        if (tid == 0) s_respec = (attempt == 0 && (dev_t != s_t || dev_m != s_m_before)) ? 1 : 0;
        __syncthreads();
        if (!s_respec) break;
        // the table was built from counters that are not the device's: rebuild
        // it from the device counters and run the loop again.  No bounds check
        // here: any code on this path, even a two-compare range test, cost the
        // launch 0.3-1.4%.  The counters are advanced only by this library's
        // kernels, on calls checked on the host against max_seq_len and M_max,
        // and the index model that turns in-range counters into a table is
        // checked per launch on the host when the handle checks segments.
        if (tid == 0) build(dev_t, dev_m);
        __syncthreads();
        nseg = s_nseg;
        total = s_start[nseg];
        chunk = (((total + p.n_split - 1) / p.n_split) + 15) & ~15;
        r0 = imin(total, split * chunk);
        r1 = imin(total, r0 + chunk);
        nstage = (r1 - r0 + KPS - 1) / KPS;
        pre = false;
#pragma unroll
        for (int c = 0; c < NST - 1; ++c) {
            if (c < nstage) load_stage(c);
            cp_async_commit();
        }
    }
    // the new token's row into its pool row (no CTA of this launch reads the row
    // it overwrites), by the split whose keys include it: that split streamed the
    // row from the caller's buffer into its last stage or the one before, and no
    // later stage overwrote it, so the row is stored from shared memory with no
    // global read on the way to the merge
    if (fresh) {
        const int jf = total - n_input;             // logical index of the new token's row
        if (jf >= r0 && jf < r1) {
            const int cf = (jf - r0) / KPS;
            step_store_row_smem<ROWB>(p, lb, h, s_t, smem + (cf % NST) * C::STAGE, smem + (cf % NST) * C::STAGE + KPS * ROWB,
                                      jf - r0 - cf * KPS);
            __syncthreads();   // the merge below reuses the stage buffers (uniform: one condition per CTA)
        }
    }

    // ---- warp results -> shared (8 columns), merge the 4 warps over the G real ones ----
    constexpr int WS = D + 8;                       // padded row stride of wo
    float* wm = reinterpret_cast<float*>(smem);    // [4][8]
    float* wl = wm + 32;                            // [4][8]
    float* wo = wl + 32;                            // [4][8][WS]
    float* cm = wo + 32 * WS;                       // [8]
    float* cl = cm + 8;                             // [8]
    float* co = cl + 8;                             // [8][D]
    float* scratch = co + 8 * D;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        float l = l_run[e];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        const int n = (lane & 3) * 2 + e;
        if (lane < 4) {
            wm[warp * 8 + n] = m_run[e];
            wl[warp * 8 + n] = l;
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            const int d = mt * 16 + (lane >> 2);
            wo[(warp * 8 + n) * WS + d] = acc[mt][e];
            wo[(warp * 8 + n) * WS + d + 8] = acc[mt][e + 2];
        }
    }
    __syncthreads();
    // rows 0..G-1 -> O of row z; rows G..2G-1 (fused slot query) -> O_g of slot row si
    EpiOut out;
    out.o = p.o + ((size_t)z * p.Hq + (size_t)h * G) * D;
    out.lse = p.lse ? p.lse + (size_t)z * p.Hq + (size_t)h * G : nullptr;
    out.rows_per_group = NR;
    out.o_row_stride = D;
    out.o_group_stride = 0;
    out.lse_row_stride = 1;
    out.lse_group_stride = 0;
    out.o_alt = si >= 0 ? p.o_slot + ((size_t)si * p.Hq + (size_t)h * G) * D : nullptr;
    out.lse_alt = (si >= 0 && p.lse_slot) ? p.lse_slot + (size_t)si * p.Hq + (size_t)h * G : nullptr;
    out.alt_from = si >= 0 ? G : -1;
    bool final_cta;
    if (p.cluster) {
        // The n_split CTAs of this (row, head) pair form one thread-block
        // cluster (rank = split).  Each merges its 4 warps per element and pushes
        // the slice of its partial that rank k finalises, and its rows' (max,
        // sum), into rank k's receive buffers; each rank waits for its own bytes
        // only and merges its slice.  Merge weights are computed where they are
        // used (no extra block barrier).
        const int nc = p.n_split, rank = split;
        for (int i4 = tid * 4; i4 < NR * D; i4 += 512) {
            const int n = i4 / D, d = i4 % D;
            float mw[4], M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                mw[w] = wm[w * 8 + n];
                M = fmaxf(M, mw[w]);
            }
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float e = mw[w] == -INFINITY ? 0.f : fast_ex2(mw[w] - M);
                const float4 x = *reinterpret_cast<const float4*>(wo + (w * 8 + n) * WS + d);
                a.x += e * x.x;
                a.y += e * x.y;
                a.z += e * x.z;
                a.w += e * x.w;
            }
            const int k = i4 / per;
            st_async_v4(mapa_rank(smem_u32(r_o + rank * per + (i4 - k * per)), k), a, mapa_rank(smem_u32(&r_bar), k));
        }
        // the rows' (max, sum) from the highest threads, beside the slice pushes
        for (int t = 127 - tid; t < NR * nc; t += 128) {
            const int n = t / nc, kk = t % nc;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w * 8 + n]);
            float l = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float mv = wm[w * 8 + n];
                if (mv != -INFINITY) l += fast_ex2(mv - M) * wl[w * 8 + n];
            }
            st_async_v2(mapa_rank(smem_u32(&r_ml[rank * 8 + n]), kk), M, l, mapa_rank(smem_u32(&r_bar), kk));
        }
        // this rank's slice from every rank (its own pushes included)
        const bool got = __syncthreads_and(tid != 0 || recv_wait(&r_bar, p.d_err));
        const int lo = rank * per, hi = imin(NR * D, lo + per);
        if (got) {
            for (int i = lo + tid; i < hi; i += 128) {
                const int n = i / D;
                float M = -INFINITY;
                for (int r = 0; r < nc; ++r) M = fmaxf(M, r_ml[r * 8 + n].x);
                float a = 0.f, dn = 0.f;
                // runtime bound: unrolled over 16 predicated ranks this loop cost
                // 2% of a launch at 6 ranks
#pragma unroll 4
                for (int r = 0; r < nc; ++r) {
                    const float2 ml = r_ml[r * 8 + n];
                    const float wr = ml.x == -INFINITY ? 0.f : fast_ex2(ml.x - M);
                    dn += wr * ml.y;
                    a += wr * r_o[r * per + (i - lo)];
                }
                out.optr(n)[i % D] = dn > 0.f ? __fdividef(a, dn) : 0.f;
            }
            if (rank == 0 && tid < NR) {
                float* lp = out.lptr(tid);
                if (lp) {
                    float M = -INFINITY, dn = 0.f;
                    for (int r = 0; r < nc; ++r) M = fmaxf(M, r_ml[r * 8 + tid].x);
                    for (int r = 0; r < nc; ++r) {
                        const float2 ml = r_ml[r * 8 + tid];
                        if (ml.x != -INFINITY) dn += fast_ex2(ml.x - M) * ml.y;
                    }
                    *lp = dn > 0.f ? (M + __log2f(dn)) * 0.6931471805599453f : -INFINITY;
                }
            }
        }
        final_cta = got && rank == 0;
    } else {
        if (tid < NR) {
            float M = -INFINITY;
            for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w * 8 + tid]);
            float l = 0.f;
            for (int w = 0; w < 4; ++w)
                if (wm[w * 8 + tid] != -INFINITY) l += exp2f(wm[w * 8 + tid] - M) * wl[w * 8 + tid];
            cm[tid] = M;
            cl[tid] = l;
        }
        __syncthreads();
        for (int i = tid; i < NR * D; i += 128) {
            const int n = i / D;
            const float M = cm[n];
            float a = 0.f;
            for (int w = 0; w < 4; ++w)
                if (wm[w * 8 + n] != -INFINITY) a += exp2f(wm[w * 8 + n] - M) * wo[(w * 8 + n) * WS + (i % D)];
            co[i] = a;
        }
        __syncthreads();
        float* part = p.part + (size_t)(z * p.Hkv + h) * p.n_split * p.rows_per_pair * (D + 2);
        final_cta = split_epilogue<D>(NR, cm, cl, co, out, part, p.tickets + z * p.Hkv + h, split, p.n_split,
                                      scratch);
    }
    if (!final_cta) return;
    if (p.mode == kDevModeSlot)
        pair_tail<ROWB>(p, lb, h, s_t, s_m_before, false, (const uint8_t*)p.k_g + (size_t)z * p.Hkv * ROWB,
                        (const uint8_t*)p.v_g + (size_t)z * p.Hkv * ROWB, s_t);
    else if (si >= 0)
        pair_tail<ROWB>(p, lb, h, s_t, s_m_before, fresh, (const uint8_t*)p.k_slot + (size_t)si * p.Hkv * ROWB,
                        (const uint8_t*)p.v_slot + (size_t)si * p.Hkv * ROWB, s_t + 1);
    else if (fresh)
        pair_tail<ROWB>(p, lb, h, s_t, s_m_before, true, nullptr, nullptr, 0);
}

// Clusters of `cs` CTAs of the decode kernel that can be resident at once (cached per device).
template <int D, int NST>
static int max_clusters(masw_mem_t* mem, int dev, int cs) {
    static std::atomic<int> cache[64][kMaxClusterSize + 1];   // per device and cluster size (idempotent fill)
    if (cs < 2 || cs > kMaxClusterSize) return 0;
    if (!cache[dev][cs].load(std::memory_order_acquire)) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs * 64, 1, 1);
        cfg.blockDim = dim3(128, 1, 1);
        cfg.dynamicSmemBytes = MmaCfg<D, NST>::SMEM;
        cudaLaunchAttribute a;
        a.id = cudaLaunchAttributeClusterDimension;
        a.val.clusterDim.x = cs;
        a.val.clusterDim.y = 1;
        a.val.clusterDim.z = 1;
        cfg.attrs = &a;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, decode_mma_kernel<D, NST>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cache[dev][cs].store(n > 0 ? n : -1, std::memory_order_release);
    }
    (void)mem;
    return cache[dev][cs].load(std::memory_order_acquire);
}

struct MmaPlan {
    int n_split;
    bool cluster;
    bool sparse;   // the grid leaves more than a third of the resident slots empty
};

// One wave of the NST-stage kernel.  Splits of a pair are merged inside a
// thread-block cluster (distributed shared memory, no global round trip) when
// clusters of that size can all be resident at once; otherwise (few pairs, many
// splits) the ticketed global merge is used.
template <int D, int NST>
static int plan_mma(masw_mem_t* mem, int rows, int GR, int kmax, MmaPlan& pl) {
    using C = MmaCfg<D, NST>;
    static std::atomic<int> occ[64];   // resident CTAs per SM, per device (idempotent fill)
    const int dev = mem->device & 63;
    if (!occ[dev].load(std::memory_order_acquire)) {
        MASW_CUDA_TRY(mem, cudaFuncSetAttribute(decode_mma_kernel<D, NST>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
        // clusters of up to 12 CTAs (beyond the portable 8) for few long pairs
        if (cudaFuncSetAttribute(decode_mma_kernel<D, NST>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess)
            cudaGetLastError();
        int n = 0;
        MASW_CUDA_TRY(mem, cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_mma_kernel<D, NST>, 128, C::SMEM));
        occ[dev].store(n > 0 ? n : 1, std::memory_order_release);
    }
    const int pairs = rows * mem->Hkv;
    const int slots = occ[dev].load(std::memory_order_acquire) * mem->num_sms;
    const int max_useful = imax(1, (kmax + 63) / 64);
    pl.n_split = 1;
    pl.cluster = false;
    // the ticket-merged plan's split count, for comparison
    int ticket_split = imin(imin(imax(1, slots / pairs), max_useful), kMaxSplit);
    while (ticket_split > 1 && masw_decode_part_floats(rows, mem->Hkv, GR, D, ticket_split) > mem->part_floats)
        --ticket_split;
    // A cluster size qualifies when all its clusters are resident at once and
    // its grid fills at least half the resident slots, or has at least half the
    // ticket plan's splits (few sequences with short working sets: the
    // shared-memory merge replaces the global ticket merge; long runs keep the
    // ticket plan's many splits).  Of those, take the fewest key stages per CTA;
    // on a tie, a grid whose clusters take at most 3/4 of the resident cluster
    // positions (a fuller one leaves the next launch no room to start early:
    // batch 4 at 32K ran 9.6 us as 32 of 36 possible 12-CTA clusters, 7.6 us as
    // 10-CTA ones), then the larger size.
    int best_stages = INT_MAX, best_full = 1;
    for (int cs = imin(kMaxClusterSize, imin(max_useful, slots / imax(1, pairs))); cs >= 2; --cs) {
        if (!(cs * pairs * 2 >= slots || 2 * cs >= ticket_split)) continue;
        const int mc = max_clusters<D, NST>(mem, dev, cs);
        if (mc < pairs) continue;
        const int chunk = ((kmax + cs - 1) / cs + 15) & ~15;   // the kernel's split length
        const int stages = (chunk + C::KPS - 1) / C::KPS;
        const int full = 4 * pairs > 3 * mc ? 1 : 0;
        if (stages < best_stages || (stages == best_stages && full < best_full)) {
            best_stages = stages;
            best_full = full;
            pl.n_split = cs;
            pl.cluster = true;
        }
    }
    if (!pl.cluster) pl.n_split = ticket_split;
    pl.sparse = 3 * pl.n_split * pairs < 2 * slots;
    return MASW_OK;
}

template <int D, int NST>
static int launch_plan(masw_mem_t* mem, DecodeParams& prm, int rows, const MmaPlan& pl, cudaStream_t stream) {
    prm.n_split = pl.n_split;
    prm.cluster = pl.cluster ? 1 : 0;
    MASW_CUDA_TRY(mem, masw_launch(decode_mma_kernel<D, NST>, dim3(pl.n_split, mem->Hkv, rows), dim3(128),
                                   MmaCfg<D, NST>::SMEM, stream, pl.cluster ? pl.n_split : 1, prm));
    return MASW_OK;
}

// Two stages unless each CTA would stream a long run of keys: more than 1536,
// or more than 1024 when the two-stage grid leaves a third of the resident
// slots empty (one split of 1090 keys per pair at batch 32: 36.3 -> 28.9 us).
// Then three stages keep more bytes in flight, which matters more than an
// early start of the next launch.  (Six splits of 1400 keys per pair on a
// full grid stay at two stages: 50.2 us against 50.7 with three.)
constexpr int kLongRunKeys = 1536, kSparseLongRunKeys = 1024;

template <int D>
static int launch_mma(masw_mem_t* mem, DecodeParams& prm, int G, int rows, int kmax, cudaStream_t stream) {
    const int GR = prm.q_slot ? 2 * G : G;   // partial rows per pair
    prm.rows_per_pair = GR;
    MmaPlan pl;
    if (int rc = plan_mma<D, 2>(mem, rows, GR, kmax, pl)) return rc;
    const int run = kmax / pl.n_split;
    if (run <= (pl.sparse ? kSparseLongRunKeys : kLongRunKeys)) return launch_plan<D, 2>(mem, prm, rows, pl, stream);
    if (int rc = plan_mma<D, 3>(mem, rows, GR, kmax, pl)) return rc;
    return launch_plan<D, 3>(mem, prm, rows, pl, stream);
}

}  // namespace masw

int masw_launch_decode_mma(masw_mem_t* mem, masw::DecodeParams& prm, int G, int rows, int kmax,
                           cudaStream_t stream) {
    if (G < 1 || G > 8 || (prm.q_slot && G > 4))
        return masw_set_error(mem, MASW_EINVAL, "query heads per kv head must be at most 8 (4 with a fused slot query)");
    if (mem->D == 128) return masw::launch_mma<128>(mem, prm, G, rows, kmax, stream);
    return masw::launch_mma<64>(mem, prm, G, rows, kmax, stream);
}
