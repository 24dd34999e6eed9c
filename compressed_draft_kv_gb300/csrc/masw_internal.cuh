// Internal declarations of libmasw: the index model, the handle, PTX helpers
// (TMA bulk copies, mbarriers with bounded waits) and the split-KV merge
// shared by the decode and verify kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <string>
#include <utility>
#include <vector>

#include "../../include/masw.h"

// ---------------------------------------------------------------------------
// Index model of one (layer, sequence), 1-based token ids as on the pages
// ([EN] §3.1 Eq. 4 and the bullets under it; §3.2 Algorithm 1).
// ---------------------------------------------------------------------------
namespace masw {

__host__ __device__ inline int imax(int a, int b) { return a > b ? a : b; }
__host__ __device__ inline int imin(int a, int b) { return a < b ? a : b; }

// lowest token of M_local,t: max(S+1, t-W+1)
__host__ __device__ inline int window_lo(int t, int S, int W) { return imax(S + 1, t - W + 1); }
// |M_local,t| = clamp(t - S, 0, W)
__host__ __device__ inline int n_local(int t, int S, int W) { return imax(0, imin(W, t - S)); }
// slots once step t is done: one per r tokens that left the window
__host__ __device__ inline int slot_count(int t, int S, int W, int r) {
    return t - S - W >= r ? (t - S - W) / r : 0;
}
__host__ __device__ inline bool is_boundary(int t, int S, int W, int r) {
    return t >= S + W + r && (t - S - W) % r == 0;
}
// ring row of non-sink token i in a ring of Wc rows
__host__ __device__ inline int ring_row(int i, int S, int Wc) { return (i - S - 1) % Wc; }
// Row `pos` (0-based) of the interleaved order of a prefix of T raw tokens and
// its M slots -- slot token g_m right after raw token tau_m = S + W + m r, the
// order in which the pages' prefill writes the memory --: the raw token i
// (1-based, > 0) or -m for slot m.  Past the first S + W raw tokens the order
// repeats r raw tokens and one slot, M times, then raw tokens only.
__host__ __device__ inline int interleaved_row(int pos, int S, int W, int r, int M) {
    const int q = pos - (S + W);
    if (q < r) return pos + 1;
    const int k = q / (r + 1);
    if (k >= M) return pos + 1 - M;
    const int o = q - k * (r + 1);
    return o < r ? S + W + k * r + o + 1 : -(k + 1);
}

}  // namespace masw

// ---------------------------------------------------------------------------
// The handle.
// ---------------------------------------------------------------------------
struct masw_mem {
    int S = 0, W = 0, r = 0, Hkv = 0, D = 0, L = 0, B = 0, dtype = MASW_BF16;
    int max_seq_len = 0, R = 0, Wc = 0, M_max = 0, C = 0;  // C = rows per (l,b,h) block
    int full_kv = 0, self_attend = 0;
    float scale = 0.f;
    size_t esize = 2;
    void* pool_k = nullptr;
    void* pool_v = nullptr;
    void* full_k = nullptr;
    void* full_v = nullptr;
    int* d_t = nullptr;      // [L*B*Hkv] raw tokens appended (one copy per kv head)
    int* d_m = nullptr;      // [L*B*Hkv] slots in the chain (one copy per kv head)
    int* d_pos = nullptr;    // [L*B*M_max] 0-based slot position ids
    int* d_err = nullptr;    // [4] error word (bounded wait ran out)
    float* part = nullptr;   // split partials
    size_t part_floats = 0;  // capacity of `part`
    unsigned* tickets = nullptr;      // [B*Hkv] per-(row, head) split tickets
    std::vector<int> h_t, h_m;
    int device = 0, num_sms = 0;
    // The handle's last launch: its stream and the layer whose pool rows it
    // wrote (-1: none; -2: unknown, e.g. after set-up).  A decode launch on the
    // same stream for another layer may copy its first K/V stages before its
    // programmatic-launch dependency wait: the only kernel it can overlap with is
    // the previous one on that stream, which wrote none of those rows.
    void* last_stream = nullptr;
    int last_write_layer = -2;
    std::string err;
    // Every device buffer above is the middle of one allocation with a guard
    // band of masw::kGuardBytes on each side, filled with masw::kGuardByte at
    // create time; masw_check_guards reads the bands back.
    struct Alloc {
        void* raw;          // cudaMalloc'd base: [guard][buffer][guard]
        size_t bytes;       // buffer bytes
        const char* name;
    };
    std::vector<Alloc> allocs;
    size_t alloc_total = 0;   // bytes allocated (guards included)
    size_t alloc_limit = 0;   // 0: none; else create refuses to allocate beyond it
    // MASW_CHECK_SEGMENTS=1 at create: every decode launch checks, on the host,
    // the segment tables its CTAs will build from the host mirror
    bool check_segments = false;
};

namespace masw {

constexpr int kMaxSplit = 256;

// guard bands around every handle-owned device buffer (out-of-bounds write
// evidence): 4 KiB of 0xC3 before and after; 4 KiB keeps the buffers'
// 256-byte alignment
constexpr size_t kGuardBytes = 4096;
constexpr unsigned char kGuardByte = 0xC3;

// bounded-wait budget: ~2^22 polls with backoff is seconds, far above any
// legitimate TMA latency; running out records MASW_ETIMEOUT and returns.
constexpr uint32_t kWaitPolls = 1u << 22;

// ---------------------------------------------------------------------------
// PTX helpers (bulk copies and mbarriers, sm_90 and later; valid on sm_103a).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// hint: bring `bytes` (a multiple of 16, 16-byte aligned) at `src` into L2
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// contiguous global -> shared bulk copy (TMA engine), completes on `bar`
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait on a phase of `bar`.  Returns false (and records the failure in
// *err) if the phase did not complete within the poll budget.
__device__ __forceinline__ bool mbar_wait_polls(uint64_t* bar, uint32_t parity, int* err, uint32_t polls) {
    for (uint32_t i = 0; i < polls; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i > 64) __nanosleep(128);
    }
    if (err) atomicExch(err, MASW_ETIMEOUT);
    return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
    return mbar_wait_polls(bar, parity, err, kWaitPolls);
}

// Programmatic dependent launch.  Every library kernel is launched with the
// programmatic-serialization attribute, so it may start while the previous
// kernel on the stream is finishing; pdl_wait() blocks until that kernel has
// completed and its memory is visible, and must come before any access to data
// an earlier kernel may write.  pdl_trigger() lets the next kernel launch early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kPerVec = 4;  // elements per 16-byte vector
    __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
        f[0] = bf16lo(v.x); f[1] = bf16hi(v.x); f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
        f[4] = bf16lo(v.z); f[5] = bf16hi(v.z); f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
    }
};

// ---------------------------------------------------------------------------
// Tensor-core and async-copy helpers (mma.sync m16n8k16, ldmatrix, movmatrix,
// cp.async): used where the GQA group turns K/V rows into a small dense
// contraction.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}


// ---------------------------------------------------------------------------
// Split-KV epilogue.  A CTA that has reduced its key range to (m, l, o) per
// query row -- m the running max of log2-scaled scores, l = sum 2^(s-m),
// o = sum 2^(s-m) v (unnormalised) -- either writes the final output (one
// split) or stores a partial and, if it is the last split of its (row, head)
// pair to arrive, merges all partials with the log-sum-exp identity
//   O = sum_s 2^(m_s-M) o_s / sum_s 2^(m_s-M) l_s,
//   LSE = (M + log2 sum_s 2^(m_s-M) l_s) ln 2.
// The ticket is taken with an atomic after a device-scope fence (no spinning)
// and reset by the last CTA, so the next launch finds it at zero.
// ---------------------------------------------------------------------------
struct EpiOut {
    float* o;            // output base for this pair
    float* lse;          // LSE base for this pair (nullable)
    // query row n of the pair lives at (n / rows_per_group) * *_group_stride
    // + (n % rows_per_group) * *_row_stride floats from the base
    int rows_per_group;
    int o_row_stride, o_group_stride;
    int lse_row_stride, lse_group_stride;
    // rows n >= alt_from go to o_alt / lse_alt instead (a second query set of
    // the same pair, e.g. a slot query fused into a draft step); alt_from < 0: none
    float* o_alt;
    float* lse_alt;
    int alt_from;
    __device__ __forceinline__ float* optr(int n) const {
        if (alt_from >= 0 && n >= alt_from) return o_alt + (size_t)(n - alt_from) * o_row_stride;
        return o + (size_t)(n / rows_per_group) * o_group_stride + (size_t)(n % rows_per_group) * o_row_stride;
    }
    __device__ __forceinline__ float* lptr(int n) const {
        if (alt_from >= 0 && n >= alt_from) return lse_alt ? lse_alt + (size_t)(n - alt_from) * lse_row_stride : nullptr;
        return lse ? lse + (size_t)(n / rows_per_group) * lse_group_stride + (size_t)(n % rows_per_group) * lse_row_stride
                   : nullptr;
    }
};

// Shared-memory floats split_epilogue needs in `sm_scratch`.
__host__ __device__ constexpr int epilogue_scratch_floats(int nrows, int n_split) {
    return nrows * n_split + 2 * nrows;
}

__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Returns true in every thread of the CTA that wrote the final output of its pair.
// Partials are stored by all threads; after a CTA barrier thread 0 takes the
// ticket with an acq_rel atomic (release of this CTA's stores, acquire of the
// earlier splits' stores for the last one).  The last CTA merges all splits in
// one pass per output element with an online log-sum-exp merge, loading the
// (m, l, o) of up to 8 splits at a time so the L2 round trips overlap.
template <int D>
__device__ bool split_epilogue(int nrows, const float* sm_m, const float* sm_l, const float* sm_o,
                               const EpiOut& out, float* part, unsigned* ticket, int split, int n_split,
                               float* sm_scratch) {
    const int tid = threadIdx.x, nt = blockDim.x;
    constexpr float kLn2 = 0.6931471805599453f;
    (void)sm_scratch;
    if (n_split == 1) {
        for (int i = tid; i < nrows * D; i += nt) {
            const int row = i / D, d = i % D;
            const float l = sm_l[row];
            out.optr(row)[d] = l > 0.f ? sm_o[row * D + d] / l : 0.f;
        }
        for (int row = tid; row < nrows; row += nt) {
            float* lp = out.lptr(row);
            const float l = sm_l[row];
            if (lp) *lp = l > 0.f ? (sm_m[row] + __log2f(l)) * kLn2 : -INFINITY;
        }
        return true;
    }
    // store this split's partial: part[split][row][D + 2] = (o[D], m, l)
    float* mine = part + (size_t)split * nrows * (D + 2);
    for (int i = tid; i < nrows * D; i += nt) {
        const int row = i / D, d = i % D;
        __stcg(mine + row * (D + 2) + d, sm_o[row * D + d]);
    }
    for (int row = tid; row < nrows; row += nt) {
        __stcg(mine + row * (D + 2) + D, sm_m[row]);
        __stcg(mine + row * (D + 2) + D + 1, sm_l[row]);
    }
    __syncthreads();
    __shared__ unsigned s_last;
    if (tid == 0) s_last = atom_add_acq_rel_gpu(ticket, 1u) == (unsigned)(n_split - 1);
    __syncthreads();
    if (!s_last) return false;
    const size_t stride = (size_t)nrows * (D + 2);
    for (int i = tid; i < nrows * D; i += nt) {
        const int row = i / D, d = i % D;
        const float* base = part + row * (D + 2);
        float M = -INFINITY, den = 0.f, acc = 0.f;
        for (int s0 = 0; s0 < n_split; s0 += 8) {
            float ms[8], ls[8], os[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const bool in = s0 + k < n_split;
                const float* ps = base + (size_t)(in ? s0 + k : 0) * stride;
                ms[k] = in ? __ldcg(ps + D) : -INFINITY;
                ls[k] = in ? __ldcg(ps + D + 1) : 0.f;
                os[k] = in ? __ldcg(ps + d) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (ms[k] == -INFINITY) continue;
                if (ms[k] > M) {
                    const float sc = exp2f(M - ms[k]);   // M = -inf gives 0
                    acc *= sc;
                    den *= sc;
                    M = ms[k];
                }
                const float w = exp2f(ms[k] - M);
                acc += w * os[k];
                den += w * ls[k];
            }
        }
        out.optr(row)[d] = den > 0.f ? acc / den : 0.f;
        if (d == 0) {
            float* lp = out.lptr(row);
            if (lp) *lp = den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
        }
    }
    if (tid == 0) *ticket = 0u;
    return true;
}

// ---------------------------------------------------------------------------
// Decode launch parameters and the segment walker shared by the decode kernels.
// ---------------------------------------------------------------------------
enum DecodeModeDev { kDevModeDraft = 0, kDevModeFull = 1, kDevModeSlot = 2 };

struct DecodeParams {
    const void* q;        // [rows][Hq][D]
    float* o;             // [rows][Hq][D]
    float* lse;           // [rows][Hq] or null
    const void* pool_k;   // [L][B][Hkv][C][D]
    const void* pool_v;
    const void* full_k;   // [L][B][Hkv][Tmax][D]
    const void* full_v;
    const void* k_g;      // slot mode: slot K/V [rows][Hkv][D]; step: new token K/V [B][Hkv][D]
    const void* v_g;
    int* d_t;
    int* d_m;
    int* d_pos;
    int* d_err;
    float* part;
    unsigned* tickets;
    float scale_log2;     // softmax scale * log2(e)
    int mode, layer, B, Hkv, Hq, S, W, Wc, C, Tmax, M_max, n_split, self_attend;
    int step;             // 1: append the new token (k_g/v_g) of every active row first (fused step)
    int cluster;          // 1: the n_split CTAs of a pair form a cluster and merge in shared memory
    int early;            // 1: the previous launch wrote no pool row of this layer; pool rows may be
                          // copied before the dependency wait (counters are re-checked after it)
    // fused boundary step: slot query / K / V / outputs for the listed rows
    // (slot_of[z] = index into them, -1 for rows not at a boundary)
    const void* q_slot;
    const void* k_slot;
    const void* v_slot;
    float* o_slot;
    float* lse_slot;
    int rows_per_pair;    // partial rows per pair in the split scratch (G, or 2G with slot queries)
    short slot_of[MASW_MAX_BATCH];
    unsigned active[MASW_MAX_BATCH / 32];
    short seq_ids[MASW_MAX_BATCH];
    // the host mirror's counters of each row at launch time: the source of the
    // speculative segment table (checked against the device counters in-kernel)
    int t_spec[MASW_MAX_BATCH];
    int m_spec[MASW_MAX_BATCH];
};

struct Seg {
    const uint8_t* k;
    const uint8_t* v;
    int len;
};

// Contiguous runs of K/V rows one (row z, kv head h) pair reads, in order:
// the sink, the window (one run, or two when it wraps around the ring), the
// slot chain, and -- for a slot write with self-attention -- the caller's own
// K_g/V_g row.  Draft mode: [EN] §3.1 Eq. 4; slot mode: [EN] §3.2 Algorithm 1
// (slots 1..m-1 only); full mode: every raw token.
template <int ROWB>
__host__ __device__ __forceinline__ int build_segments(const DecodeParams& p, int lb, int h, int z, int t, int mcnt,
                                              Seg* segs) {
    // fused step: the query sees token t+1, whose K/V row comes straight from
    // the caller's buffer; the pool holds tokens 1..t
    const bool fresh = p.step && ((p.active[z >> 5] >> (z & 31)) & 1u);
    const size_t new_off = ((size_t)z * p.Hkv + h) * ROWB;
    int n = 0;
    if (p.mode == kDevModeFull) {
        const size_t base = ((size_t)lb * p.Hkv + h) * (size_t)p.Tmax * ROWB;
        if (t > 0) segs[n++] = Seg{(const uint8_t*)p.full_k + base, (const uint8_t*)p.full_v + base, t};
        if (fresh) segs[n++] = Seg{(const uint8_t*)p.k_g + new_off, (const uint8_t*)p.v_g + new_off, 1};
        return n;
    }
    const int tq = fresh ? t + 1 : t;               // step the query sits at
    const size_t base = ((size_t)lb * p.Hkv + h) * (size_t)p.C * ROWB;
    const uint8_t* kb = (const uint8_t*)p.pool_k + base;
    const uint8_t* vb = (const uint8_t*)p.pool_v + base;
    const int ns = imin(p.S, t);                    // sink rows already in the pool
    if (ns > 0) segs[n++] = Seg{kb, vb, ns};
    if (tq > p.S) {
        const int lo = window_lo(tq, p.S, p.W);
        const int nl = t - lo + 1;                  // window tokens already in the ring: lo..t
        if (nl > 0) {
            const int start = ring_row(lo, p.S, p.Wc);
            const int first = imin(nl, p.Wc - start);
            segs[n++] = Seg{kb + (size_t)(p.S + start) * ROWB, vb + (size_t)(p.S + start) * ROWB, first};
            if (nl > first) segs[n++] = Seg{kb + (size_t)p.S * ROWB, vb + (size_t)p.S * ROWB, nl - first};
        }
    }
    if (mcnt > 0) segs[n++] = Seg{kb + (size_t)(p.S + p.Wc) * ROWB, vb + (size_t)(p.S + p.Wc) * ROWB, mcnt};
    if (fresh) segs[n++] = Seg{(const uint8_t*)p.k_g + new_off, (const uint8_t*)p.v_g + new_off, 1};
    if (p.mode == kDevModeSlot && p.self_attend) {
        const size_t off = ((size_t)z * p.Hkv + h) * ROWB;
        segs[n++] = Seg{(const uint8_t*)p.k_g + off, (const uint8_t*)p.v_g + off, 1};
    }
    return n;
}

// Out-of-bounds check of the index model's result: every run of pool rows must
// lie inside its own (layer, sequence, kv head) block and in its region -- the
// sink in rows [0, S), window runs in the ring rows [S, S + Wc), the slot chain
// in [S + Wc, S + Wc + M_max); full-KV runs inside the block's max_seq_len rows
// -- a caller row must be the one the API places for (row z, head h), and no two
// runs may overlap.  Pointer comparisons only (it also runs on the host, over
// the speculative tables, when a handle checks its launches).
template <int ROWB>
__host__ __device__ inline bool segments_in_block(const DecodeParams& p, int lb, int h, int z, const Seg* segs, int n) {
    const bool full = p.mode == kDevModeFull;
    const uint8_t* kb = (const uint8_t*)(full ? p.full_k : p.pool_k);
    const ptrdiff_t dv = (const uint8_t*)(full ? p.full_v : p.pool_v) - kb;
    const size_t rows = full ? (size_t)p.Tmax : (size_t)p.C;
    const uint8_t* b0 = kb + ((size_t)lb * p.Hkv + h) * rows * ROWB;
    const uint8_t* b1 = full ? b0 + rows * ROWB : b0 + (size_t)p.S * ROWB;
    const uint8_t* b2 = b1 + (size_t)(full ? 0 : p.Wc) * ROWB;
    const uint8_t* b3 = b2 + (size_t)(full ? 0 : p.M_max) * ROWB;
    const uint8_t* own_k = p.k_g ? (const uint8_t*)p.k_g + ((size_t)z * p.Hkv + h) * ROWB : nullptr;
    const uint8_t* own_v = p.v_g ? (const uint8_t*)p.v_g + ((size_t)z * p.Hkv + h) * ROWB : nullptr;
    bool ok = n <= 5;
    for (int s = 0; s < n; ++s) {
        const Seg& g = segs[s];
        const uint8_t* e = g.k + (size_t)g.len * ROWB;
        if (g.k == own_k) {
            ok = ok && g.len == 1 && g.v == own_v;
            continue;
        }
        const uint8_t* lo = g.k < b1 ? b0 : (g.k < b2 ? b1 : b2);
        const uint8_t* hi = g.k < b1 ? b1 : (g.k < b2 ? b2 : b3);
        ok = ok && g.len >= 1 && g.k >= lo && e <= hi && g.v - g.k == dv;
        for (int q = 0; q < s; ++q)
            if (segs[q].k != own_k) ok = ok && (e <= segs[q].k || segs[q].k + (size_t)segs[q].len * ROWB <= g.k);
    }
    return ok;
}

// build_segments plus that check on the device, for the tables built from the
// device counters; a table that fails is recorded in d_err[3] (masw_sync
// reports it as MASW_EGUARD) and replaced by an empty one, so no copy leaves
// its block.
template <int ROWB>
__device__ int build_segments_checked(const DecodeParams& p, int lb, int h, int z, int t, int mcnt, Seg* segs) {
    const int n = build_segments<ROWB>(p, lb, h, z, t, mcnt, segs);
    if (segments_in_block<ROWB>(p, lb, h, z, segs, n)) return n;
    atomicExch(p.d_err + 3, 1);
    return 0;
}

// After the attention of pair (row z, head h) is final -- its last split, or
// rank 0 of its cluster -- every CTA of the pair has read this head's copy of
// the counters, so the pair updates them on its own, with no cross-head
// coordination: a slot write appends head h's K_g/V_g row as chain entry
// m_before and records the slot's position id; a fused step bumps the token
// counter.  (Counters are kept per (layer, sequence, kv head); all heads of a
// sequence hold equal values between launches.)
template <int ROWB>
__device__ void pair_tail(const DecodeParams& p, int lb, int h, int t, int m_before, bool fresh,
                          const uint8_t* slot_k, const uint8_t* slot_v, int pos_id) {
    const int tid = threadIdx.x;
    const size_t ci = (size_t)lb * p.Hkv + h;
    if (slot_k) {
        const size_t dst = (ci * p.C + (size_t)(p.S + p.Wc + m_before)) * ROWB;
        for (int c = tid; c < ROWB / 16; c += blockDim.x) {
            *reinterpret_cast<uint4*>((uint8_t*)p.pool_k + dst + c * 16) =
                *reinterpret_cast<const uint4*>(slot_k + (size_t)h * ROWB + c * 16);
            *reinterpret_cast<uint4*>((uint8_t*)p.pool_v + dst + c * 16) =
                *reinterpret_cast<const uint4*>(slot_v + (size_t)h * ROWB + c * 16);
        }
    }
    if (tid == 0) {
        if (slot_k) {
            if (h == 0) p.d_pos[(size_t)lb * p.M_max + m_before] = pos_id;
            p.d_m[ci] = m_before + 1;
        }
        if (fresh) {
            if (p.full_k != nullptr && t + 1 > p.Tmax) atomicExch(p.d_err + 1, MASW_ECAPACITY);
            p.d_t[ci] = t + 1;
        }
    }
}

}  // namespace masw

// ---------------------------------------------------------------------------
// Host helpers shared by the translation units.
// ---------------------------------------------------------------------------
int masw_set_error(masw_mem_t* mem, int code, const std::string& msg);
// record a launch of the handle (see masw_mem::last_stream)
inline void masw_note_launch(masw_mem_t* mem, void* stream, int wrote_layer) {
    mem->last_stream = stream;
    mem->last_write_layer = wrote_layer;
}
inline bool masw_may_copy_early(const masw_mem_t* mem, void* stream, int layer) {
    return mem->last_write_layer != -2 && mem->last_stream == stream && mem->last_write_layer != layer;
}
#define MASW_CUDA_TRY(mem, call)                                                        \
    do {                                                                                \
        cudaError_t e_ = (call);                                                        \
        if (e_ != cudaSuccess)                                                          \
            return masw_set_error((mem), MASW_ECUDA, std::string(#call) + ": " +       \
                                                         cudaGetErrorString(e_));      \
    } while (0)

// Launch `kern` with the programmatic-serialization attribute (and an optional
// cluster of cluster_x CTAs along x).
template <typename... KArgs, typename... Args>
cudaError_t masw_launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                        int cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (cluster_x > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster_x;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// decode-kernel launcher (masw_decode.cu)
enum DecodeMode { kModeDraft = 0, kModeFull = 1, kModeSlot = 2 };
struct SlotFuse {            // slot queries fused into a draft step
    const int* seq_ids;
    int n;
    const void* q_g;
    const void* k_g;
    const void* v_g;
    float* o_g;
    float* lse_g;
};
int masw_launch_decode(masw_mem_t* mem, int mode, int layer, const void* q, int n_q_heads, float* o,
                       float* lse, const int* seq_ids, int n_rows, const void* k_g, const void* v_g,
                       cudaStream_t stream, const unsigned* step_active = nullptr, const SlotFuse* fuse = nullptr);
// floats of split scratch one decode launch with these sizes may use
size_t masw_decode_part_floats(int rows, int Hkv, int G, int D, int n_split);
// tensor-core decode for bf16 pools (masw_decode_mma.cu)
int masw_launch_decode_mma(masw_mem_t* mem, masw::DecodeParams& prm, int G, int rows, int kmax, cudaStream_t stream);
