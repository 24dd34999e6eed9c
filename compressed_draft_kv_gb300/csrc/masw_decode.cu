// Split-KV decode attention on CUDA cores, used for fp32 pools (bf16 pools
// use the tensor-core kernel of masw_decode_mma.cu): the MASW draft working memory
// (sink block, ring-indexed local window, slot chain), the slot-write query
// under the structured mask, and the full-KV contrast cache.
//
// Computes Eq. 2 of [EN] §2.3 for one query token per sequence over the sets
// of [EN] §3.1 Eq. 4 (draft), [EN] §3.2 Algorithm 1 (slot write) or
// the whole prefix (full KV).
//
// Grid: (n_split, Hkv, rows).  One CTA streams one contiguous share of the
// logical key list of one (row, kv head) pair through shared memory with TMA
// bulk copies (cp.async.bulk + mbarrier, NST stages in flight) and serves all
// G = Hq/Hkv query heads of the GQA group from each staged K/V row.  Within a
// warp, LPR lanes share one row (16 bytes each, 128-bit loads from shared
// memory); partial dot products are finished with a transpose-reduce over the
// LPR lanes (about one shuffle per row per head), online softmax runs in the
// log2 domain, and P*V is accumulated in fp32 registers.  Splits are merged by
// the last CTA of each pair (split_epilogue).
#include "masw_internal.cuh"

#include <atomic>

#include <cstring>

namespace masw {

template <typename T, int D>
struct DecodeCfg {
    static constexpr int VEC = Elem<T>::kPerVec;        // elements per 16-byte vector
    static constexpr int LPR = D / VEC;                  // lanes per row
    static constexpr int RPI = 32 / LPR;                 // rows per warp instruction
    static constexpr int U = 8;                          // rows per lane per tile
    static constexpr int LOG2U = 3;
    static constexpr int WT = RPI * U;                   // rows per warp tile
    static constexpr int NWARPS = 4;
    static constexpr int THREADS = NWARPS * 32;
    static constexpr int RPS = NWARPS * WT;              // rows per stage
    static constexpr int ROWB = D * (int)sizeof(T);      // bytes per row
    static constexpr int STAGE_BYTES = 2 * RPS * ROWB;   // K then V
    static constexpr int NST = 3;                        // stages in flight
    static constexpr int SMEM_BYTES = NST * STAGE_BYTES;
    static_assert(LPR >= U && LPR <= 32 && (32 % LPR) == 0, "unsupported row geometry");
    // the CTA merge reuses the stage buffers
    static_assert((2 * NWARPS * MASW_MAX_GROUP + NWARPS * MASW_MAX_GROUP * D + 2 * MASW_MAX_GROUP +
                   MASW_MAX_GROUP * D + epilogue_scratch_floats(MASW_MAX_GROUP, kMaxSplit)) * 4 <= SMEM_BYTES,
                  "merge does not fit in the stage buffers");
};

// Finish U partial dot products held by the LPR lanes of a row group.  After
// the halving stages lane `sub` holds the full sum of row reduced_row(sub);
// lanes differing only in the low log2(LPR/U) bits hold duplicates.
template <int U, int LOG2U, int LPR>
__device__ __forceinline__ float transpose_reduce(float (&v)[U], int lane) {
#pragma unroll
    for (int k = 0; k < LOG2U; ++k) {
        const int off = LPR >> (k + 1);
        const int half = U >> (k + 1);
        const bool hi = (lane & off) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
            const float send = hi ? v[j] : v[j + half];
            const float keep = hi ? v[j + half] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (int off = (LPR >> LOG2U) >> 1; off >= 1; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    return v[0];
}
template <int U, int LOG2U, int LPR>
__device__ __forceinline__ int reduced_row(int sub) {
    int r = 0;
#pragma unroll
    for (int k = 0; k < LOG2U; ++k)
        if (sub & (LPR >> (k + 1))) r += U >> (k + 1);
    return r;
}
template <int U, int LOG2U, int LPR>
__host__ __device__ constexpr int row_owner(int u) {
    int s = 0;
    for (int k = 0; k < LOG2U; ++k)
        if (u & (U >> (k + 1))) s += LPR >> (k + 1);
    return s;
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

template <typename T, int D, int G>
__global__ void __launch_bounds__(DecodeCfg<T, D>::THREADS)
decode_kernel(const __grid_constant__ DecodeParams p) {
    using Cfg = DecodeCfg<T, D>;
    constexpr int VEC = Cfg::VEC, LPR = Cfg::LPR, U = Cfg::U, LOG2U = Cfg::LOG2U, WT = Cfg::WT;
    constexpr int RPS = Cfg::RPS, ROWB = Cfg::ROWB, NST = Cfg::NST, NWARPS = Cfg::NWARPS;

    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[NST];
    __shared__ Seg segs[5];
    __shared__ int s_nseg, s_m_before, s_t;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, h = blockIdx.y, z = blockIdx.z;
    const int b = (p.mode == kModeSlot) ? (int)p.seq_ids[z] : z;
    const int lb = p.layer * p.B + b;
    pdl_wait();
    pdl_trigger();

    if (tid == 0) {
        const int t = p.d_t[(size_t)lb * p.Hkv + h];
        const int mcnt = p.d_m[(size_t)lb * p.Hkv + h];
        s_m_before = mcnt;
        s_t = t;
        const int n = build_segments_checked<ROWB>(p, lb, h, z, t, mcnt, segs);
        s_nseg = n;
        for (int s = 0; s < NST; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    int total = 0;
    for (int s = 0; s < s_nseg; ++s) total += segs[s].len;
    const int chunk = (((total + p.n_split - 1) / p.n_split) + 15) & ~15;
    const int r0 = imin(total, split * chunk);
    const int r1 = imin(total, r0 + chunk);
    const int nrows = r1 - r0;
    const int nstage = (nrows + RPS - 1) / RPS;

    // producer: copy logical rows [r0 + c*RPS, ...) of the segment list into stage c % NST
    auto issue = [&](int c) {
        uint8_t* dk = smem + (size_t)(c % NST) * Cfg::STAGE_BYTES;
        uint8_t* dv = dk + RPS * ROWB;
        const int lo = r0 + c * RPS, hi = imin(r1, lo + RPS);
        mbar_expect_tx(&bars[c % NST], (uint32_t)(hi - lo) * ROWB * 2u);
        int seg_lo = 0;
        for (int s = 0; s < s_nseg; ++s) {
            const int seg_hi = seg_lo + segs[s].len;
            const int a = imax(lo, seg_lo), e = imin(hi, seg_hi);
            if (a < e) {
                const uint32_t bytes = (uint32_t)(e - a) * ROWB;
                bulk_g2s(dk + (size_t)(a - lo) * ROWB, segs[s].k + (size_t)(a - seg_lo) * ROWB, bytes,
                         &bars[c % NST]);
                bulk_g2s(dv + (size_t)(a - lo) * ROWB, segs[s].v + (size_t)(a - seg_lo) * ROWB, bytes,
                         &bars[c % NST]);
            }
            seg_lo = seg_hi;
        }
    };
    if (tid == 0)
        for (int c = 0; c < imin(NST, nstage); ++c) issue(c);

    // query fragment of this lane: G heads x VEC elements, scaled into log2 units
    const int g = lane / LPR, sub = lane % LPR;
    float qf[G][VEC];
    {
        const T* qrow = (const T*)p.q + ((size_t)z * p.Hq + (size_t)h * G) * D + sub * VEC;
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            const uint4 raw = *reinterpret_cast<const uint4*>(qrow + (size_t)gi * D);
            Elem<T>::unpack(raw, qf[gi]);
#pragma unroll
            for (int e = 0; e < VEC; ++e) qf[gi][e] *= p.scale_log2;
        }
    }

    float m_run[G], l_run[G], acc[G][VEC];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
        m_run[gi] = -INFINITY;
        l_run[gi] = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[gi][e] = 0.f;
    }
    const bool primary = (sub & ((LPR >> LOG2U) - 1)) == 0;
    const int my_row = g * U + reduced_row<U, LOG2U, LPR>(sub);

    bool ok = true;
    int c = 0;
    for (; c < nstage; ++c) {
        const int s = c % NST;
        const bool waited = __all_sync(0xffffffffu, mbar_wait(&bars[s], (uint32_t)(c / NST) & 1u, p.d_err));
        const int valid_stage = imin(RPS, nrows - c * RPS);
        const int valid = valid_stage - warp * WT;       // rows of this warp's tile
        if (waited && valid > 0) {
            const uint8_t* kt = smem + (size_t)s * Cfg::STAGE_BYTES + (size_t)(warp * WT + g * U) * ROWB + sub * 16;
            const uint8_t* vt = kt + RPS * ROWB;
            float sc[G][U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float kf[VEC];
                const uint4 raw = (g * U + u < valid) ? lds128(kt + u * ROWB) : make_uint4(0, 0, 0, 0);
                Elem<T>::unpack(raw, kf);
#pragma unroll
                for (int gi = 0; gi < G; ++gi) {
                    float d0 = 0.f;
#pragma unroll
                    for (int e = 0; e < VEC; ++e) d0 = fmaf(qf[gi][e], kf[e], d0);
                    sc[gi][u] = d0;
                }
            }
            float pr[G];
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
                float sv = transpose_reduce<U, LOG2U, LPR>(sc[gi], lane);
                if (my_row >= valid) sv = -INFINITY;
                float tmax = sv;
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
                const float m_new = fmaxf(m_run[gi], tmax);   // finite: the tile has a valid row
                const float alpha = exp2f(m_run[gi] - m_new);
                const float pv = exp2f(sv - m_new);
                l_run[gi] = l_run[gi] * alpha + (primary ? pv : 0.f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[gi][e] *= alpha;
                m_run[gi] = m_new;
                pr[gi] = pv;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool rv = g * U + u < valid;
                float vf[VEC];
                const uint4 raw = rv ? lds128(vt + u * ROWB) : make_uint4(0, 0, 0, 0);
                Elem<T>::unpack(raw, vf);
                const int src = g * LPR + row_owner<U, LOG2U, LPR>(u);
#pragma unroll
                for (int gi = 0; gi < G; ++gi) {
                    const float pu = __shfl_sync(0xffffffffu, pr[gi], src);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) acc[gi][e] = fmaf(pu, vf[e], acc[gi][e]);
                }
            }
        }
        ok = __syncthreads_and(waited) != 0;
        if (!ok) break;
        if (tid == 0 && c + NST < nstage) issue(c + NST);
    }
    if (!ok) {
        // a bounded wait ran out: wait (bounded) for the copies still in flight, then leave
        if (tid == 0)
            for (int c2 = c; c2 < imin(nstage, c + NST); ++c2)
                mbar_wait(&bars[c2 % NST], (uint32_t)(c2 / NST) & 1u, nullptr);
        __syncthreads();
        return;
    }

    // ---- reduce the warp: l over lanes, acc over the RPI row groups ----
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) l_run[gi] += __shfl_xor_sync(0xffffffffu, l_run[gi], off);
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[gi][e] += __shfl_xor_sync(0xffffffffu, acc[gi][e], off);
    }
    // the stage buffers are free now (every copy was consumed): reuse them for the CTA merge
    float* wm = reinterpret_cast<float*>(smem);           // [NWARPS][G]
    float* wl = wm + NWARPS * G;                           // [NWARPS][G]
    float* wo = wl + NWARPS * G;                           // [NWARPS][G][D]
    float* cm = wo + NWARPS * G * D;                       // [G]
    float* cl = cm + G;                                    // [G]
    float* co = cl + G;                                    // [G][D]
    float* scratch = co + G * D;                           // merge scratch
    if (lane < LPR) {
#pragma unroll
        for (int gi = 0; gi < G; ++gi)
#pragma unroll
            for (int e = 0; e < VEC; ++e) wo[(warp * G + gi) * D + sub * VEC + e] = acc[gi][e];
    }
    if (lane == 0)
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            wm[warp * G + gi] = m_run[gi];
            wl[warp * G + gi] = l_run[gi];
        }
    __syncthreads();
    if (tid < G) {
        float M = -INFINITY;
        for (int w = 0; w < NWARPS; ++w) M = fmaxf(M, wm[w * G + tid]);
        float l = 0.f;
        for (int w = 0; w < NWARPS; ++w)
            if (wm[w * G + tid] != -INFINITY) l += exp2f(wm[w * G + tid] - M) * wl[w * G + tid];
        cm[tid] = M;
        cl[tid] = l;
    }
    __syncthreads();
    for (int i = tid; i < G * D; i += blockDim.x) {
        const int gi = i / D;
        const float M = cm[gi];
        float a = 0.f;
        for (int w = 0; w < NWARPS; ++w)
            if (wm[w * G + gi] != -INFINITY) a += exp2f(wm[w * G + gi] - M) * wo[(w * G + gi) * D + (i % D)];
        co[i] = a;
    }
    __syncthreads();

    EpiOut out;
    out.o = p.o + ((size_t)z * p.Hq + (size_t)h * G) * D;
    out.lse = p.lse ? p.lse + (size_t)z * p.Hq + (size_t)h * G : nullptr;
    out.rows_per_group = G;
    out.o_row_stride = D;
    out.o_group_stride = 0;
    out.lse_row_stride = 1;
    out.lse_group_stride = 0;
    out.o_alt = nullptr;
    out.lse_alt = nullptr;
    out.alt_from = -1;
    float* part = p.part + (size_t)(z * p.Hkv + h) * p.n_split * G * (D + 2);
    const bool final_cta = split_epilogue<D>(G, cm, cl, co, out, part, p.tickets + z * p.Hkv + h, split,
                                             p.n_split, scratch);

    if (p.mode == kModeSlot && final_cta)
        pair_tail<ROWB>(p, lb, h, s_t, s_m_before, false, (const uint8_t*)p.k_g + (size_t)z * p.Hkv * ROWB,
                        (const uint8_t*)p.v_g + (size_t)z * p.Hkv * ROWB, s_t);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <typename T, int D, int G>
static int launch_t(masw_mem_t* mem, const DecodeParams& prm, int rows, cudaStream_t stream) {
    using Cfg = DecodeCfg<T, D>;
    static std::atomic<bool> configured[64];   // per device, set once (idempotent)
    const int dev = mem->device & 63;
    if (!configured[dev].load(std::memory_order_acquire)) {
        MASW_CUDA_TRY(mem, cudaFuncSetAttribute(decode_kernel<T, D, G>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES));
        configured[dev].store(true, std::memory_order_release);
    }
    MASW_CUDA_TRY(mem, masw_launch(decode_kernel<T, D, G>, dim3(prm.n_split, mem->Hkv, rows), dim3(Cfg::THREADS),
                                   Cfg::SMEM_BYTES, stream, 1, prm));
    return MASW_OK;
}

template <typename T, int D>
static int launch_g(masw_mem_t* mem, const DecodeParams& prm, int G, int rows, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_t<T, D, 1>(mem, prm, rows, stream);
        case 2: return launch_t<T, D, 2>(mem, prm, rows, stream);
        case 3: return launch_t<T, D, 3>(mem, prm, rows, stream);
        case 4: return launch_t<T, D, 4>(mem, prm, rows, stream);
        case 6: return launch_t<T, D, 6>(mem, prm, rows, stream);
        case 8: return launch_t<T, D, 8>(mem, prm, rows, stream);
        default: return masw_set_error(mem, MASW_EINVAL, "query heads per kv head must be 1, 2, 3, 4, 6 or 8");
    }
}

}  // namespace masw

using namespace masw;

size_t masw_decode_part_floats(int rows, int Hkv, int G, int D, int n_split) {
    return (size_t)rows * Hkv * n_split * G * (D + 2);
}

// Keys walked by one (row, head) pair, from the host mirror (only used to pick
// the split count; the kernel re-derives everything from device counters).
static int host_keys(const masw_mem_t* mem, int mode, int l, int b) {
    const int t = mem->h_t[(size_t)l * mem->B + b];
    const int m = mem->h_m[(size_t)l * mem->B + b];
    if (mode == kModeFull) return t;
    return imin(mem->S, t) + n_local(t, mem->S, mem->W) + m + (mode == kModeSlot && mem->self_attend ? 1 : 0);
}

int masw_launch_decode(masw_mem_t* mem, int mode, int layer, const void* q, int n_q_heads, float* o,
                       float* lse, const int* seq_ids, int n_rows, const void* k_g, const void* v_g,
                       cudaStream_t stream, const unsigned* step_active, const SlotFuse* fuse) {
    const int G = n_q_heads / mem->Hkv;
    DecodeParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.q = q;
    prm.o = o;
    prm.lse = lse;
    prm.pool_k = mem->pool_k;
    prm.pool_v = mem->pool_v;
    prm.full_k = mem->full_k;
    prm.full_v = mem->full_v;
    prm.k_g = k_g;
    prm.v_g = v_g;
    prm.d_t = mem->d_t;
    prm.d_m = mem->d_m;
    prm.d_pos = mem->d_pos;
    prm.d_err = mem->d_err;
    prm.part = mem->part;
    prm.tickets = mem->tickets;
    prm.scale_log2 = mem->scale * 1.4426950408889634f;
    prm.mode = mode;
    prm.layer = layer;
    prm.B = mem->B;
    prm.Hkv = mem->Hkv;
    prm.Hq = n_q_heads;
    prm.S = mem->S;
    prm.W = mem->W;
    prm.Wc = mem->Wc;
    prm.C = mem->C;
    prm.Tmax = mem->max_seq_len;
    prm.M_max = mem->M_max;
    prm.self_attend = mem->self_attend;
    prm.early = masw_may_copy_early(mem, stream, layer) ? 1 : 0;
    if (step_active) {
        prm.step = 1;
        for (int i = 0; i < MASW_MAX_BATCH / 32; ++i) prm.active[i] = step_active[i];
    }
    prm.rows_per_pair = G;
    for (int i = 0; i < MASW_MAX_BATCH; ++i) prm.slot_of[i] = -1;
    if (fuse) {
        prm.q_slot = fuse->q_g;
        prm.k_slot = fuse->k_g;
        prm.v_slot = fuse->v_g;
        prm.o_slot = fuse->o_g;
        prm.lse_slot = fuse->lse_g;
        for (int i = 0; i < fuse->n; ++i) prm.slot_of[fuse->seq_ids[i]] = (short)i;
    }
    int kmax = 0;
    for (int i = 0; i < n_rows; ++i) {
        const int b = seq_ids ? seq_ids[i] : i;
        prm.seq_ids[i] = (short)b;
        prm.t_spec[i] = mem->h_t[(size_t)layer * mem->B + b];
        prm.m_spec[i] = mem->h_m[(size_t)layer * mem->B + b];
        kmax = imax(kmax, host_keys(mem, mode, layer, b) + (step_active ? 1 : 0));
    }
    // split count: about three CTAs per SM in total, at least 64 keys per split,
    // and no more partials than the scratch holds
    const int pairs = n_rows * mem->Hkv;
    const int target = 3 * mem->num_sms;
    int n_split = imax(1, (target + pairs - 1) / pairs);
    n_split = imin(n_split, imax(1, (kmax + 63) / 64));
    n_split = imin(n_split, kMaxSplit);
    while (n_split > 1 && masw_decode_part_floats(n_rows, mem->Hkv, G, mem->D, n_split) > mem->part_floats)
        --n_split;
    prm.n_split = n_split;
    if (mem->check_segments && mem->dtype == MASW_BF16) {
        // the tables the tensor-core kernel builds from the host mirror, before it runs
        Seg segs[5];
        for (int z = 0; z < n_rows; ++z)
            for (int h = 0; h < mem->Hkv; ++h) {
                const int lbz = layer * mem->B + prm.seq_ids[z];
                const int n = mem->D == 128
                                  ? build_segments<256>(prm, lbz, h, z, prm.t_spec[z], prm.m_spec[z], segs)
                                  : build_segments<128>(prm, lbz, h, z, prm.t_spec[z], prm.m_spec[z], segs);
                const bool ok = mem->D == 128 ? segments_in_block<256>(prm, lbz, h, z, segs, n)
                                              : segments_in_block<128>(prm, lbz, h, z, segs, n);
                if (!ok)
                    return masw_set_error(mem, MASW_EGUARD, "decode: segment table of row " + std::to_string(z) +
                                                                ", head " + std::to_string(h) + " leaves its block");
            }
    }
    int rc;
    if (mem->dtype == MASW_BF16)
        rc = masw_launch_decode_mma(mem, prm, G, n_rows, kmax, stream);
    else if (mem->D == 128)
        rc = launch_g<float, 128>(mem, prm, G, n_rows, stream);
    else
        rc = launch_g<float, 64>(mem, prm, G, n_rows, stream);
    // a fused step stores the new token's row, a slot write stores the slot's rows
    masw_note_launch(mem, stream, (prm.step || mode == kModeSlot || fuse) ? layer : -1);
    return rc;
}
