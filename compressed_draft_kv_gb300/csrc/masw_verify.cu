// Target verify attention over an uncompressed cache ([EN] §3.3 Algorithm 2
// step 5): Lq query positions per sequence, causal inside the block, GQA.
//
// This is the one dense contraction on the path (Lq*G query rows share every
// K/V row, 24 flop per byte at Lq = 6, G = 4), so it runs on tensor cores:
// mma.sync m16n8k16 bf16 -> fp32 with KEYS as the M dimension and the Lq*G
// query rows as N (8 per tile), so 24 query rows fill three N tiles without
// padding.  Each warp owns one N tile of one 16-key group (4 NT warps per CTA),
// which keeps its accumulators at about 80 registers.  S^T = K Q^T is accumulated per 16-key tile from ldmatrix fragments
// of a padded-row shared-memory stage (cp.async, 3 stages), softmax runs
// online per query column in the log2 domain, P^T is turned from the
// accumulator layout into a B operand with movmatrix, and O^T += V^T P^T uses
// ldmatrix.trans on the same V stage.  Splits over the key axis are merged by
// split_epilogue.
#include "masw_internal.cuh"

#include <atomic>

#include <cstring>

namespace masw {

struct VerifyParams {
    const __nv_bfloat16* q;   // [B][Lq][Hq][D]
    const __nv_bfloat16* k;   // [B][Hkv][Tmax][D]
    const __nv_bfloat16* v;
    const int* kv_len;        // [B]
    float* o;                 // [B][Lq][Hq][D]
    float* lse;               // [B][Lq][Hq] or null
    float* part;              // [B*Hkv][n_split][NQ][D+2]
    unsigned* tickets;        // [B*Hkv]
    int B, Lq, Hq, Hkv, G, NQ, Tmax, n_split;
    float scale_log2;
};

constexpr int kVD = 128;             // head_dim
constexpr int kVKeys = 64;           // keys per stage (16 per warp)
constexpr int kVRowB = kVD * 2;      // bytes per K/V row
constexpr int kVRowP = kVRowB + 16;  // padded row stride in shared memory: the 8 row addresses of an
                                     // ldmatrix phase fall in distinct banks, and every k-step's offset
                                     // is a compile-time immediate (no per-access swizzle arithmetic)
constexpr int kVStage = 2 * kVKeys * kVRowP;
constexpr int kVNst = 3;
constexpr int kVSmem = kVNst * kVStage;
constexpr int kVMaxSplit = 64;       // bounds the merge scratch kept in shared memory
constexpr int kVMaxNQ = 32;
static_assert((2 * 4 * kVMaxNQ + 4 * kVMaxNQ * (kVD + 8) + 2 * kVMaxNQ + kVMaxNQ * kVD +
               epilogue_scratch_floats(kVMaxNQ, kVMaxSplit)) * 4 <= kVSmem,
              "verify merge does not fit in the stage buffers");

// 2^x by the MUFU instruction (an input of -inf gives 0)
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pad_off(int row, int chunk) {  // byte offset of a 16-B chunk
    return (uint32_t)(row * kVRowP + (chunk << 4));
}
// three stages for every tile count (two CTAs per SM at three tiles; six stages
// on one CTA per SM measured slower)
template <int NT>
__host__ __device__ constexpr int verify_stages() { return kVNst; }
template <int NT>
__host__ __device__ constexpr int verify_smem() { return verify_stages<NT>() * kVStage; }

// NT tiles of 8 query columns; warp w handles keys 16 (w % 4) .. +15 of each
// stage for column tile w / 4, so a warp keeps one tile's accumulators (about
// 96 registers) and a CTA has 4 NT warps: more warps in flight than one warp
// holding every tile.
template <int NT>
__global__ void __launch_bounds__(128 * NT) verify_kernel(const __grid_constant__ VerifyParams p) {
    constexpr int NSTV = verify_stages<NT>();
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
    const int kg = warp & 3, ct = warp >> 2;   // key group, column tile
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int G = p.G, NQ = p.NQ;
    pdl_wait();
    pdl_trigger();

    const int n_keys = p.kv_len[b];
    const int chunk = (((n_keys + p.n_split - 1) / p.n_split) + kVKeys - 1) / kVKeys * kVKeys;
    const int k0 = imin(n_keys, split * chunk);
    const int k1 = imin(n_keys, k0 + chunk);
    const int nstage = (k1 - k0 + kVKeys - 1) / kVKeys;

    const __nv_bfloat16* kbase = p.k + ((size_t)b * p.Hkv + h) * (size_t)p.Tmax * kVD;
    const __nv_bfloat16* vbase = p.v + ((size_t)b * p.Hkv + h) * (size_t)p.Tmax * kVD;
    const uint32_t sbase = smem_u32(smem);

    // one stage = 64 keys of K and V in padded rows; rows past k1 are
    // zero-filled (src-size 0 reads nothing)
    auto load_stage = [&](int c) {
        const uint32_t sk = sbase + (uint32_t)(c % NSTV) * kVStage;
        const uint32_t sv = sk + kVKeys * kVRowP;
        const int key0 = k0 + c * kVKeys;
        for (int idx = tid; idx < kVKeys * 16; idx += nthr) {
            const int row = idx >> 4, ch = idx & 15;
            const int key = key0 + row;
            const bool in = key < k1;
            const size_t goff = (size_t)(in ? key : k0) * kVD + ch * 8;
            cp_async16(sk + pad_off(row, ch), kbase + goff, in ? 16 : 0);
            cp_async16(sv + pad_off(row, ch), vbase + goff, in ? 16 : 0);
        }
    };
#pragma unroll
    for (int c = 0; c < NSTV - 1; ++c) {
        if (c < nstage) load_stage(c);
        cp_async_commit();
    }

    // Q^T as B fragments of this warp's column tile: column n = query row
    // (j = n / G, gi = n % G)
    uint32_t qb[8][2];
    {
        const int n = ct * 8 + (lane >> 2);
        const bool real = n < NQ;
        const int j = real ? n / G : 0, gi = real ? n % G : 0;
        const __nv_bfloat16* qrow = p.q + (((size_t)b * p.Lq + j) * p.Hq + (size_t)h * G + gi) * kVD;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int d = ks * 16 + (lane & 3) * 2;
            qb[ks][0] = real ? *reinterpret_cast<const uint32_t*>(qrow + d) : 0u;
            qb[ks][1] = real ? *reinterpret_cast<const uint32_t*>(qrow + d + 8) : 0u;
        }
    }
    // causal limit of this lane's two columns: key < lim
    int lim[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int n = ct * 8 + (lane & 3) * 2 + e;
        lim[e] = n < NQ ? imin(k1, n_keys - p.Lq + 1 + n / G) : k1;
    }

    // this lane's ldmatrix row addresses within a stage (k-step / m-tile add 32 bytes)
    const uint32_t k_off = pad_off(kg * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, lane >> 4);
    const uint32_t v_off = pad_off(kg * 16 + (lane & 7) + (lane >> 4) * 8, (lane >> 3) & 1);
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float acc[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

    for (int c = 0; c < nstage; ++c) {
        cp_async_wait<NSTV - 2>();
        __syncthreads();
        {   // refill the stage consumed in the previous iteration
            const int cn = c + NSTV - 1;
            if (cn < nstage) load_stage(cn);
            cp_async_commit();
        }
        const uint32_t sk = sbase + (uint32_t)(c % NSTV) * kVStage;
        const uint32_t sv = sk + kVKeys * kVRowP;
        const int kw = kg * 16;
        const int key_tile = k0 + c * kVKeys + kw;
        if (key_tile < k1) {
            // two accumulators (even and odd k-steps) halve the dependent MMA chain
            float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(sk + k_off + ks * 32, a0, a1, a2, a3);
                mma16816((ks & 1) ? s2 : s, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) s[e] += s2[e];
            float x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] = s[e] * p.scale_log2;
            // the causal mask only bites in the tile that crosses the block's
            // diagonal (warp-uniform test: every key of the tile below every
            // column's limit)
            if (!__all_sync(0xffffffffu, key_tile + 16 <= imin(lim[0], lim[1]))) {
                const int key_a = key_tile + (lane >> 2), key_b = key_a + 8;
                if (key_a >= lim[0]) x[0] = -INFINITY;
                if (key_a >= lim[1]) x[1] = -INFINITY;
                if (key_b >= lim[0]) x[2] = -INFINITY;
                if (key_b >= lim[1]) x[3] = -INFINITY;
            }
            float pr[4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float mx = fmaxf(x[e], x[e + 2]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float m_new = fmaxf(m_run[e], mx);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;   // column fully masked so far
                const float alpha = ex2_ftz(m_run[e] - m_use);
                pr[e] = ex2_ftz(x[e] - m_use);
                pr[e + 2] = ex2_ftz(x[e + 2] - m_use);
                l_run[e] = l_run[e] * alpha + pr[e] + pr[e + 2];
                m_run[e] = m_new;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    acc[mt][e] *= alpha;
                    acc[mt][e + 2] *= alpha;
                }
            }
            const uint32_t pb0 = movmatrix_t(pack_bf16(pr[0], pr[1]));
            const uint32_t pb1 = movmatrix_t(pack_bf16(pr[2], pr[3]));
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(sv + v_off + mt * 32, a0, a1, a2, a3);
                mma16816(acc[mt], a0, a1, a2, a3, pb0, pb1);
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- warp results -> shared, then merge the 4 key groups ----
    constexpr int NQM = NT * 8;
    constexpr int WS = kVD + 8;                     // padded row stride: conflict-free stores
    float* wm = reinterpret_cast<float*>(smem);    // [4][NQM]
    float* wl = wm + 4 * NQM;                       // [4][NQM]
    float* wo = wl + 4 * NQM;                       // [4][NQM][WS]
    float* cm = wo + 4 * NQM * WS;                  // [NQM]
    float* cl = cm + NQM;
    float* co = cl + NQM;                           // [NQM][D]
    float* scratch = co + NQM * kVD;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        float l = l_run[e];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        const int n = ct * 8 + (lane & 3) * 2 + e;
        if (lane < 4) {
            wm[kg * NQM + n] = m_run[e];
            wl[kg * NQM + n] = l;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int d = mt * 16 + (lane >> 2);
            wo[(kg * NQM + n) * WS + d] = acc[mt][e];
            wo[(kg * NQM + n) * WS + d + 8] = acc[mt][e + 2];
        }
    }
    __syncthreads();
    if (tid < NQ) {
        float M = -INFINITY;
        for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w * NQM + tid]);
        float l = 0.f;
        for (int w = 0; w < 4; ++w)
            if (wm[w * NQM + tid] != -INFINITY) l += exp2f(wm[w * NQM + tid] - M) * wl[w * NQM + tid];
        cm[tid] = M;
        cl[tid] = l;
    }
    __syncthreads();
    for (int i = tid; i < NQ * kVD; i += nthr) {
        const int n = i / kVD;
        const float M = cm[n];
        float a = 0.f;
        for (int w = 0; w < 4; ++w)
            if (wm[w * NQM + n] != -INFINITY) a += exp2f(wm[w * NQM + n] - M) * wo[(w * NQM + n) * WS + (i % kVD)];
        co[i] = a;
    }
    __syncthreads();

    EpiOut out;
    out.o = p.o + ((size_t)b * p.Lq * p.Hq + (size_t)h * G) * kVD;
    out.lse = p.lse ? p.lse + (size_t)b * p.Lq * p.Hq + (size_t)h * G : nullptr;
    out.rows_per_group = G;
    out.o_row_stride = kVD;
    out.o_group_stride = p.Hq * kVD;
    out.lse_row_stride = 1;
    out.lse_group_stride = p.Hq;
    out.o_alt = nullptr;
    out.lse_alt = nullptr;
    out.alt_from = -1;
    float* part = p.part + (size_t)(b * p.Hkv + h) * p.n_split * NQ * (kVD + 2);
    split_epilogue<kVD>(NQ, cm, cl, co, out, part, p.tickets + b * p.Hkv + h, split, p.n_split, scratch);
}

template <int NT>
static cudaError_t verify_configure(int* n) {
    cudaError_t e = cudaFuncSetAttribute(verify_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         verify_smem<NT>());
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, verify_kernel<NT>, 128 * NT, verify_smem<NT>());
    return e;
}

// Resident verify CTAs per SM for NT query tiles (cached per device).
static int verify_occupancy(int NT) {
    static std::atomic<int> cache[64][5];   // per device and tile count (idempotent fill)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || NT < 1 || NT > 4) return 1;
    if (!cache[dev][NT].load(std::memory_order_acquire)) {
        int n = 0;
        cudaError_t e = cudaSuccess;
        switch (NT) {
            case 1: e = verify_configure<1>(&n); break;
            case 2: e = verify_configure<2>(&n); break;
            case 3: e = verify_configure<3>(&n); break;
            default: e = verify_configure<4>(&n); break;
        }
        if (e != cudaSuccess) cudaGetLastError();
        cache[dev][NT].store(n > 0 ? n : 1, std::memory_order_release);
    }
    return cache[dev][NT].load(std::memory_order_acquire);
}

// Split count shared by the launcher and the workspace query: one wave of the
// resident CTA slots, at least 256 keys per split.
static int verify_splits(int B, int Hkv, int Tmax, int num_sms, int NT) {
    const int pairs = B * Hkv;
    const int slots = verify_occupancy(NT) * num_sms;
    int n = imax(1, slots / pairs);
    n = imin(n, imax(1, (Tmax + 255) / 256));
    return imin(n, kVMaxSplit);
}

static int num_sms_current(int* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MASW_ECUDA;
    if (cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MASW_ECUDA;
    return MASW_OK;
}

static size_t verify_part_bytes(int B, int Hkv, int NQ, int n_split) {
    const size_t partb = (size_t)B * Hkv * n_split * NQ * (kVD + 2) * sizeof(float);
    return ((partb + 255) / 256) * 256;
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
    const int n_split = verify_splits(B, Hkv, Tmax, sms, (NQ + 7) / 8);
    *bytes = verify_part_bytes(B, Hkv, NQ, n_split) + (size_t)B * Hkv * sizeof(unsigned);
    return MASW_OK;
}

template <int NT>
static cudaError_t launch_verify(const VerifyParams& prm, cudaStream_t stream) {
    static std::atomic<bool> configured[64];   // per device, set once (idempotent)
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configured[dev & 63].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(verify_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             verify_smem<NT>());
        if (e != cudaSuccess) return e;
        configured[dev & 63].store(true, std::memory_order_release);
    }
    return masw_launch(verify_kernel<NT>, dim3(prm.n_split, prm.Hkv, prm.B), dim3(128 * NT), verify_smem<NT>(),
                       stream, 1, prm);
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
    const int n_split = verify_splits(B, Hkv, Tmax, sms, (NQ + 7) / 8);
    const size_t partb = verify_part_bytes(B, Hkv, NQ, n_split);
    if (workspace_bytes < partb + (size_t)B * Hkv * sizeof(unsigned))
        return masw_set_error(nullptr, MASW_EINVAL, "verify: workspace too small");
    VerifyParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.q = (const __nv_bfloat16*)q;
    prm.k = (const __nv_bfloat16*)k_cache;
    prm.v = (const __nv_bfloat16*)v_cache;
    prm.kv_len = kv_len;
    prm.o = o;
    prm.lse = lse;
    prm.part = (float*)workspace;
    prm.tickets = (unsigned*)((uint8_t*)workspace + partb);
    prm.B = B;
    prm.Lq = Lq;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.G = G;
    prm.NQ = NQ;
    prm.Tmax = Tmax;
    prm.n_split = n_split;
    prm.scale_log2 = (scale > 0.f ? scale : 1.0f / sqrtf((float)D)) * 1.4426950408889634f;
    cudaStream_t st = (cudaStream_t)stream;
    // the tickets are zero on entry (zero-filled workspace, reset by the last
    // CTA of each pair in every call): no memset node between calls, so
    // consecutive verify launches keep their programmatic overlap
    cudaError_t e = cudaSuccess;
    const int NT = (NQ + 7) / 8;
    switch (NT) {
        case 1: e = launch_verify<1>(prm, st); break;
        case 2: e = launch_verify<2>(prm, st); break;
        case 3: e = launch_verify<3>(prm, st); break;
        default: e = launch_verify<4>(prm, st); break;
    }
    if (e != cudaSuccess) return masw_set_error(nullptr, MASW_ECUDA, std::string("verify: ") + cudaGetErrorString(e));
    return MASW_OK;
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
// Limits: B * Hkv <= kNoAllocMaxPairs; when the partials of the usual split
// count would not fit in kNoAllocPartBytes the call uses fewer splits (one
// split needs no partials at all), so it is never refused for length alone.
// All calls share the array and each leaves its partials in it; the tickets
// are cleared on the stream at the start of every call.  Two calls that
// overlap on the GPU (different streams, or different host threads) race on
// the array and give wrong results: serialise them.
// ---------------------------------------------------------------------------
#include <mutex>

namespace masw {
constexpr size_t kNoAllocPartBytes = (size_t)4 << 20;
constexpr int kNoAllocMaxPairs = 4096;
constexpr size_t kNoAllocBytes = kNoAllocPartBytes + (size_t)kNoAllocMaxPairs * sizeof(unsigned);
}  // namespace masw

static __device__ __align__(256) uint8_t g_noalloc_scratch[masw::kNoAllocBytes];

// Device address of g_noalloc_scratch per device.  In host code the array's
// name is only a host-side stand-in; the kernel must be given this address.
static void* g_noalloc_ptr[64];
static std::mutex g_noalloc_mu;

static int noalloc_scratch(int dev, void** out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return masw_set_error(nullptr, MASW_ECUDA, std::string("verify_noalloc: cudaGetSymbolAddress: ") +
                                                           cudaGetErrorString(e));
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return MASW_OK;
}

extern "C" int masw_verify_attn_noalloc(const void* q, const void* k_cache, const void* v_cache, const int* kv_len,
                                        int B, int Lq, int Hq, int Hkv, int D, int Tmax, int dtype, float scale,
                                        float* o, float* lse, masw_stream_t stream) {
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
    if (((uintptr_t)o | (uintptr_t)lse | (uintptr_t)kv_len) & 3)
        return masw_set_error(nullptr, MASW_EINVAL, "verify_noalloc: o, lse and kv_len must be 4-byte aligned");
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || num_sms_current(&sms)) {
        cudaGetLastError();
        return masw_set_error(nullptr, MASW_ECUDA, "verify_noalloc: cannot query the current device");
    }
    void* scratch = nullptr;
    if ((rc = noalloc_scratch(dev, &scratch))) return rc;
    const int G = Hq / Hkv, NQ = G * Lq;
    int n_split = verify_splits(B, Hkv, Tmax, sms, (NQ + 7) / 8);
    while (n_split > 1 && verify_part_bytes(B, Hkv, NQ, n_split) > kNoAllocPartBytes) --n_split;
    VerifyParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.q = (const __nv_bfloat16*)q;
    prm.k = (const __nv_bfloat16*)k_cache;
    prm.v = (const __nv_bfloat16*)v_cache;
    prm.kv_len = kv_len;
    prm.o = o;
    prm.lse = lse;
    prm.part = (float*)scratch;
    prm.tickets = (unsigned*)((uint8_t*)scratch + kNoAllocPartBytes);
    prm.B = B;
    prm.Lq = Lq;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.G = G;
    prm.NQ = NQ;
    prm.Tmax = Tmax;
    prm.n_split = n_split;
    prm.scale_log2 = (scale > 0.f ? scale : 1.0f / sqrtf((float)D)) * 1.4426950408889634f;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(prm.tickets, 0, (size_t)B * Hkv * sizeof(unsigned), st);
    if (e != cudaSuccess)
        return masw_set_error(nullptr, MASW_ECUDA, std::string("verify_noalloc: ") + cudaGetErrorString(e));
    switch ((NQ + 7) / 8) {
        case 1: e = launch_verify<1>(prm, st); break;
        case 2: e = launch_verify<2>(prm, st); break;
        case 3: e = launch_verify<3>(prm, st); break;
        default: e = launch_verify<4>(prm, st); break;
    }
    if (e != cudaSuccess)
        return masw_set_error(nullptr, MASW_ECUDA, std::string("verify_noalloc: ") + cudaGetErrorString(e));
    return MASW_OK;
}
