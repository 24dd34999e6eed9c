// Draft prefill under the structured write mask ([EN] §3.3 Algorithm 2 step 2
// with the mask of §3.2 Algorithm 1 step 2): one layer of attention over a whole
// prefix of T raw tokens with the M = m(T) memory-slot tokens interleaved, then
// the resulting memory M_0 is stored in the pool.
//
// Query rows: raw token i (1-based) reads the sink, raw tokens of its window
// [max(S+1, i-W+1), i], and the slots materialised before it (tau_m < i); slot
// token g_m reads the sink, the window at tau_m and slots 1..m-1.  Key rows come
// from the caller's raw and slot K/V arrays ([T, Hkv, D], [M, Hkv, D]); the
// visible set of a 64-row query tile is a handful of contiguous key ranges
// (sink, window band, slot prefix), walked in 64-key blocks with the exact
// per-element mask.
//
// Tensor cores (mma.sync m16n8k16 bf16 -> fp32), FlashAttention-style: 4 warps,
// 16 query rows each, Q as the A operand, K rows as B fragments (ldmatrix),
// online softmax per row, P reused from the accumulator layout as the A operand
// of P.V, V as B fragments (ldmatrix.trans), K/V blocks staged with cp.async in
// XOR-swizzled shared memory (2 stages).  Grid (query tiles, Hq).
#include "masw_internal.cuh"

#include <algorithm>
#include <cstring>

namespace masw {

struct PrefillParams {
    const __nv_bfloat16* q_raw;   // [T][Hq][D]
    const __nv_bfloat16* k_raw;   // [T][Hkv][D]
    const __nv_bfloat16* v_raw;
    const __nv_bfloat16* q_slot;  // [M][Hq][D]
    const __nv_bfloat16* k_slot;  // [M][Hkv][D]
    const __nv_bfloat16* v_slot;
    float* o_raw;                 // [T][Hq][D]
    float* lse_raw;               // [T][Hq] or null
    float* o_slot;                // [M][Hq][D]
    float* lse_slot;              // [M][Hq] or null
    int T, M, S, W, r, Hq, Hkv, self_attend;
    int raw_tiles;                // tiles of raw query rows (the rest are slot tiles)
    int slot_rows;                // slot query rows per slot tile (SB)
    float scale_log2;
};

constexpr int kPD = 128;            // head_dim
constexpr int kPRowB = kPD * 2;
constexpr int kPBM = 64;            // query rows per CTA
constexpr int kPBN = 64;            // keys per block
constexpr int kPStage = 2 * kPBN * kPRowB;
constexpr int kPNst = 2;
constexpr int kPSmem = kPBM * kPRowB + kPNst * kPStage;   // Q tile + K/V stages

__device__ __forceinline__ uint32_t pswz(int row, int ch) { return (uint32_t)(row * kPRowB + ((ch ^ (row & 7)) << 4)); }

// key range: rows [a, b) of either the raw (slot = 0) or the slot (slot = 1) arrays
struct KRange {
    int a, b, slot;
};

__global__ void __launch_bounds__(128) prefill_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hq = blockIdx.y, G = p.Hq / p.Hkv, kvh = hq / G;
    const bool slot_tile = (int)blockIdx.x >= p.raw_tiles;
    // raw tiles hold 64 consecutive positions; slot tiles hold slot_rows slots, so
    // that their windows (r apart) span at most about 2W raw keys
    const int q0 = slot_tile ? ((int)blockIdx.x - p.raw_tiles) * p.slot_rows : (int)blockIdx.x * kPBM;
    const int nq = slot_tile ? p.M : p.T;
    const int q1 = imin(nq, q0 + (slot_tile ? p.slot_rows : kPBM));
    const __nv_bfloat16* qsrc = slot_tile ? p.q_slot : p.q_raw;

    // visible key ranges of the tile (0-based rows)
    KRange rg[3];
    int nr = 0;
    const int S = p.S, W = p.W, r = p.r;
    if (!slot_tile) {
        const int i0 = q0 + 1, i1 = q1;            // 1-based raw positions of the tile
        if (S > 0) rg[nr++] = KRange{0, imin(S, i1), 0};
        const int wlo = imax(S + 1, i0 - W + 1);
        if (i1 >= wlo) rg[nr++] = KRange{wlo - 1, i1, 0};
        const int ns = slot_count(i1 - 1, S, W, r);
        if (ns > 0) rg[nr++] = KRange{0, ns, 1};
    } else {
        const int m0 = q0 + 1, m1 = q1;            // 1-based slot indices of the tile
        const int tau0 = S + W + m0 * r, tau1 = S + W + m1 * r;
        if (S > 0) rg[nr++] = KRange{0, S, 0};
        rg[nr++] = KRange{imax(S, tau0 - W), tau1, 0};
        const int ns = p.self_attend ? m1 : m1 - 1;
        if (ns > 0) rg[nr++] = KRange{0, ns, 1};
    }
    int nblk = 0, bstart[4];
    for (int k = 0; k < nr; ++k) {
        bstart[k] = nblk;
        nblk += (rg[k].b - rg[k].a + kPBN - 1) / kPBN;
    }
    bstart[nr] = nblk;

    const uint32_t sq = smem_u32(smem);
    const uint32_t sbase = sq + kPBM * kPRowB;
    // Q tile (rows past q1 zero-filled)
    for (int idx = tid; idx < kPBM * 16; idx += 128) {
        const int row = idx >> 4, ch = idx & 15;
        const int qr = q0 + row;
        const bool in = qr < q1;
        cp_async16(sq + pswz(row, ch), qsrc + ((size_t)(in ? qr : q0) * p.Hq + hq) * kPD + ch * 8, in ? 16 : 0);
    }
    auto load_block = [&](int blk, int stage) {
        int k = 0;
        while (k + 1 < nr && blk >= bstart[k + 1]) ++k;
        const int key0 = rg[k].a + (blk - bstart[k]) * kPBN;
        const int kend = rg[k].b;
        const __nv_bfloat16* ks = rg[k].slot ? p.k_slot : p.k_raw;
        const __nv_bfloat16* vs = rg[k].slot ? p.v_slot : p.v_raw;
        const uint32_t sk = sbase + (uint32_t)stage * kPStage;
        const uint32_t sv = sk + kPBN * kPRowB;
        for (int idx = tid; idx < kPBN * 16; idx += 128) {
            const int row = idx >> 4, ch = idx & 15;
            const int key = key0 + row;
            const bool in = key < kend;
            const size_t off = ((size_t)(in ? key : key0) * p.Hkv + kvh) * kPD + ch * 8;
            cp_async16(sk + pswz(row, ch), ks + off, in ? 16 : 0);
            cp_async16(sv + pswz(row, ch), vs + off, in ? 16 : 0);
        }
    };
    if (nblk > 0) load_block(0, 0);
    cp_async_commit();

    // per-lane query rows (0-based within the tile): lane/4 and lane/4 + 8 of this warp's 16
    const int qa = q0 + warp * 16 + (lane >> 2), qb = qa + 8;
    uint32_t qf[8][4];
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float acc[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

    for (int blk = 0; blk < nblk; ++blk) {
        if (blk + 1 < nblk) load_block(blk + 1, (blk + 1) & 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (blk == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                ldsm_x4(sq + pswz(warp * 16 + (lane & 15), ks * 2 + (lane >> 4)), qf[ks][0], qf[ks][1], qf[ks][2],
                        qf[ks][3]);
        }
        int k = 0;
        while (k + 1 < nr && blk >= bstart[k + 1]) ++k;
        const int key0 = rg[k].a + (blk - bstart[k]) * kPBN;
        const int kend = rg[k].b;
        const bool kslot = rg[k].slot != 0;
        const uint32_t sk = sbase + (uint32_t)(blk & 1) * kPStage;
        const uint32_t sv = sk + kPBN * kPRowB;

        // S = Q K^T for this warp's 16 rows x 64 keys (8 n-tiles of 8 keys)
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {   // two n-tiles per ldmatrix.x4
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sk + pswz(np * 16 + (lane & 7) + ((lane >> 4) << 3), ks * 2 + ((lane >> 3) & 1)), b0, b1, b2,
                        b3);
                mma16816(s[2 * np], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
                mma16816(s[2 * np + 1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
            }
        }
        // structured mask, scale, online softmax per row
        float rmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = key0 + nt * 8 + (lane & 3) * 2 + (e & 1);
                const int qrow = (e < 2) ? qa : qb;
                bool vis = key < kend && qrow < q1;
                if (vis) {
                    if (!slot_tile) {
                        const int i = qrow + 1;                      // raw query position
                        if (!kslot) {
                            const int j = key + 1;                   // raw key position
                            vis = (j <= S) ? (j <= i) : (j >= imax(S + 1, i - W + 1) && j <= i);
                        } else {
                            vis = key < slot_count(i - 1, S, W, r);  // slot key+1 has tau <= i-1
                        }
                    } else {
                        const int m = qrow + 1;                      // slot query index
                        const int tau = S + W + m * r;
                        if (!kslot) {
                            const int j = key + 1;
                            vis = (j <= S) || (j >= tau - W + 1 && j <= tau);
                        } else {
                            vis = p.self_attend ? key < m : key < m - 1;
                        }
                    }
                }
                s[nt][e] = vis ? s[nt][e] * p.scale_log2 : -INFINITY;
                rmax[e >> 1] = fmaxf(rmax[e >> 1], s[nt][e]);
            }
        float alpha[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            float mx = rmax[h2];
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_run[h2], mx);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            alpha[h2] = exp2f(m_run[h2] - m_use);
            m_run[h2] = m_new;
            rmax[h2] = m_use;
        }
        float rsum[2] = {0.f, 0.f};
        uint32_t pa[4][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const float p0 = exp2f(s[nt][0] - rmax[0]), p1 = exp2f(s[nt][1] - rmax[0]);
            const float p2 = exp2f(s[nt][2] - rmax[1]), p3 = exp2f(s[nt][3] - rmax[1]);
            rsum[0] += p0 + p1;
            rsum[1] += p2 + p3;
            // accumulator tile nt -> half of the A fragment of k-step nt/2
            pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p0, p1);
            pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) l_run[h2] = l_run[h2] * alpha[h2] + rsum[h2];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            acc[nt][0] *= alpha[0];
            acc[nt][1] *= alpha[0];
            acc[nt][2] *= alpha[1];
            acc[nt][3] *= alpha[1];
        }
        // O += P V: k-steps of 16 keys, 16 n-tiles of 8 head dims
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int dp = 0; dp < 8; ++dp) {   // two d n-tiles per ldmatrix.x4.trans
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(sv + pswz(kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), dp * 2 + (lane >> 4)), b0, b1,
                          b2, b3);
                mma16816(acc[2 * dp], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
                mma16816(acc[2 * dp + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
            }
        }
        __syncthreads();   // the stage is refilled by the next iteration's prefetch
    }
    cp_async_wait<0>();

    // finish: row sums over the 4 lanes of a row, normalise, store
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        l_run[h2] += __shfl_xor_sync(0xffffffffu, l_run[h2], 1);
        l_run[h2] += __shfl_xor_sync(0xffffffffu, l_run[h2], 2);
    }
    float* obase = slot_tile ? p.o_slot : p.o_raw;
    float* lbase = slot_tile ? p.lse_slot : p.lse_raw;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        const int qrow = h2 ? qb : qa;
        if (qrow >= q1) continue;
        const float l = l_run[h2];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float* orow = obase + ((size_t)qrow * p.Hq + hq) * kPD;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int d = nt * 8 + (lane & 3) * 2;
            *reinterpret_cast<float2*>(orow + d) = make_float2(acc[nt][2 * h2] * inv, acc[nt][2 * h2 + 1] * inv);
        }
        if (lbase && (lane & 3) == 0)
            lbase[(size_t)qrow * p.Hq + hq] = l > 0.f ? (m_run[h2] + __log2f(l)) * 0.6931471805599453f : -INFINITY;
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

extern "C" int masw_prefill(masw_mem_t* mem, int layer, int seq, int T, const void* q_raw, const void* k_raw,
                            const void* v_raw, const void* q_slot, const void* k_slot, const void* v_slot,
                            int n_q_heads, float* o_raw, float* lse_raw, float* o_slot, float* lse_slot,
                            masw_stream_t stream) {
    if (!mem) return masw_set_error(nullptr, MASW_EINVAL, "prefill: NULL handle");
    if (layer < 0 || layer >= mem->L || seq < 0 || seq >= mem->B)
        return masw_set_error(mem, MASW_EINVAL, "prefill: layer or seq out of range");
    if (mem->dtype != MASW_BF16 || mem->D != kPD)
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
    PrefillParams p;
    std::memset(&p, 0, sizeof(p));
    p.q_raw = (const __nv_bfloat16*)q_raw;
    p.k_raw = (const __nv_bfloat16*)k_raw;
    p.v_raw = (const __nv_bfloat16*)v_raw;
    p.q_slot = (const __nv_bfloat16*)q_slot;
    p.k_slot = (const __nv_bfloat16*)k_slot;
    p.v_slot = (const __nv_bfloat16*)v_slot;
    p.o_raw = o_raw;
    p.lse_raw = lse_raw;
    p.o_slot = o_slot;
    p.lse_slot = lse_slot;
    p.T = T;
    p.M = M;
    p.S = mem->S;
    p.W = mem->W;
    p.r = mem->r;
    p.Hq = n_q_heads;
    p.Hkv = mem->Hkv;
    p.self_attend = mem->self_attend;
    p.raw_tiles = (T + kPBM - 1) / kPBM;
    p.slot_rows = imin(kPBM, imax(1, mem->W / mem->r + 1));
    p.scale_log2 = mem->scale * 1.4426950408889634f;
    const int tiles = p.raw_tiles + (M + p.slot_rows - 1) / p.slot_rows;
    cudaStream_t st = (cudaStream_t)stream;
    static bool configured[64] = {};
    if (!configured[mem->device & 63]) {
        MASW_CUDA_TRY(mem, cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem));
        configured[mem->device & 63] = true;
    }
    MASW_CUDA_TRY(mem, masw_launch(prefill_kernel, dim3(tiles, n_q_heads), dim3(128), kPSmem, st, 1, p));
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
