// Greedy speculative acceptance on the target's verify logits ([EN] §2.2 Eq. 1
// and §3.3 Algorithm 2; the pages' experiments decode greedily, T = 0).
//
// For sequence b the target's token at block position j (0..L) is the argmax of
// logits[b][j][0..V) (ties to the smallest id; NaN entries are skipped, since
// every comparison with NaN is false; a row with nothing but NaN has no token
// and reports -1, which no draft equals).  Draft token j is accepted while
// it equals the target's token at j; the first mismatch (or position L when all
// L drafts match) contributes the target's own token, so L_acc + 1 tokens are
// emitted and they are exactly tokens[b][0 .. L_acc].
//
// Grid (chunks, L+1, B): each CTA reduces one vocabulary chunk of one row with
// 16-byte loads to a (max, id) pair; the last CTA of a sequence (ticket) merges
// the chunks of its L+1 rows, computes L_acc and resets its ticket, so the
// workspace is zero-filled again when the call completes.  HBM-bound: the
// logits are read once.
#include "masw_internal.cuh"

#include <cstring>

namespace masw {

struct AcceptParams {
    const void* logits;   // [B][L+1][V]
    const int* draft;     // [B][L]
    int* tokens;          // [B][L+1]
    int* n_emit;          // [B]
    float* part_v;        // [B][L+1][chunks]
    int* part_i;          // [B][L+1][chunks]
    unsigned* tickets;    // [B]
    int B, L, V, chunks, chunk;
    int bf16;
    int vec;              // 1: rows are 16-byte aligned
};

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(256) accept_kernel(const __grid_constant__ AcceptParams p) {
    pdl_wait();
    pdl_trigger();
    const int c = blockIdx.x, j = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    // the sequence's first 64 draft tokens, read now so that the last CTA
    // compares them from shared memory instead of waiting on global reads
    __shared__ int s_draft[64];
    if (tid < imin(p.L, 64)) s_draft[tid] = __ldg(p.draft + (size_t)b * p.L + tid);
    const int row = b * (p.L + 1) + j;
    const int v0 = c * p.chunk, v1 = imin(p.V, v0 + p.chunk);
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    if (p.bf16) {
        const __nv_bfloat16* x = (const __nv_bfloat16*)p.logits + (size_t)row * p.V;
        int v = v0;
        if (p.vec) {
            const int vv0 = (v0 + 7) & ~7, vv1 = v1 & ~7;
            for (int i = v0 + tid; i < imin(vv0, v1); i += 256) {
                const float f = __bfloat162float(x[i]);
                if (better(f, i, bv, bi)) { bv = f; bi = i; }
            }
            // eight independent 16-byte loads in flight per thread per round (a
            // chunk is read in one round trip; four took two: 8.1 -> 6.9 us)
            for (int i0 = vv0 + tid * 8; i0 < vv1; i0 += 8 * 256 * 8) {
                uint4 w[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * 256 * 8;
                    w[u] = i < vv1 ? __ldcs(reinterpret_cast<const uint4*>(x + i)) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * 256 * 8;
                    if (i >= vv1) break;
                    float f[8];
                    Elem<__nv_bfloat16>::unpack(w[u], f);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if (better(f[k], i + k, bv, bi)) { bv = f[k]; bi = i + k; }
                }
            }
            v = imax(vv0, vv1);
        }
        for (int i = v + tid; i < v1; i += 256) {
            const float f = __bfloat162float(x[i]);
            if (better(f, i, bv, bi)) { bv = f; bi = i; }
        }
    } else {
        const float* x = (const float*)p.logits + (size_t)row * p.V;
        int v = v0;
        if (p.vec) {
            const int vv0 = (v0 + 3) & ~3, vv1 = v1 & ~3;
            for (int i = v0 + tid; i < imin(vv0, v1); i += 256)
                if (better(x[i], i, bv, bi)) { bv = x[i]; bi = i; }
            for (int i = vv0 + tid * 4; i < vv1; i += 256 * 4) {
                const float4 w = *reinterpret_cast<const float4*>(x + i);
                const float f[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (better(f[k], i + k, bv, bi)) { bv = f[k]; bi = i + k; }
            }
            v = imax(vv0, vv1);
        }
        for (int i = v + tid; i < v1; i += 256)
            if (better(x[i], i, bv, bi)) { bv = x[i]; bi = i; }
    }
    // block reduce (max, smallest id)
    for (int off = 16; off; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    __shared__ float sv[8];
    __shared__ int si[8];
    if ((tid & 31) == 0) { sv[tid >> 5] = bv; si[tid >> 5] = bi; }
    __syncthreads();
    __shared__ unsigned s_last;
    if (tid == 0) {
        for (int w = 1; w < 8; ++w)
            if (better(sv[w], si[w], sv[0], si[0])) { sv[0] = sv[w]; si[0] = si[w]; }
        const size_t k = (size_t)row * p.chunks + c;
        __stcg(p.part_v + k, sv[0]);
        __stcg(p.part_i + k, si[0]);
        s_last = atom_add_acq_rel_gpu(p.tickets + b, 1u) == (unsigned)(p.chunks * (p.L + 1) - 1);
    }
    __syncthreads();
    if (!s_last) return;
    // last CTA of sequence b: warp w merges the chunks of rows w, w+8, ... (lanes
    // stride over chunks), then thread 0 finds the first rejected draft
    __shared__ int s_tok[64];
    const int lane = tid & 31, warp = tid >> 5;
    for (int jj = warp; jj <= p.L; jj += 8) {
        const size_t base = (size_t)(b * (p.L + 1) + jj) * p.chunks;
        float mv = -INFINITY;
        int mi = 0x7fffffff;
        for (int cc = lane; cc < p.chunks; cc += 32) {
            const float v2 = __ldcg(p.part_v + base + cc);
            const int i2 = __ldcg(p.part_i + base + cc);
            if (better(v2, i2, mv, mi)) { mv = v2; mi = i2; }
        }
        for (int off = 16; off; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, mv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, mi, off);
            if (better(ov, oi, mv, mi)) { mv = ov; mi = oi; }
        }
        if (lane == 0) {
            // no id survives only when every entry of the row is NaN: no greedy token
            const int tok = mi == 0x7fffffff ? -1 : mi;
            p.tokens[b * (p.L + 1) + jj] = tok;
            if (jj < 64) s_tok[jj] = tok;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int l_acc = p.L;
        for (int jj = 0; jj < p.L; ++jj) {
            const int tj = jj < 64 ? s_tok[jj] : __ldcg(p.tokens + b * (p.L + 1) + jj);
            const int dj = jj < 64 ? s_draft[jj] : __ldg(p.draft + (size_t)b * p.L + jj);
            if (dj != tj) { l_acc = jj; break; }
        }
        p.n_emit[b] = l_acc + 1;
        p.tickets[b] = 0u;
    }
}

static int accept_chunks(int B, int L, int V, int sms) {
    const int rows = B * (L + 1);
    int ch = imax(1, (4 * sms + rows - 1) / rows);
    return imin(ch, imax(1, (V + 2047) / 2048));
}

static size_t accept_ws_bytes(int B, int L, int chunks) {
    const size_t n = (size_t)B * (L + 1) * chunks;
    return ((n * 8 + 255) / 256) * 256 + (size_t)B * sizeof(unsigned);
}

}  // namespace masw

using namespace masw;

static int accept_sms(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return MASW_ECUDA;
    }
    return MASW_OK;
}

extern "C" int masw_greedy_workspace_bytes(int B, int L, int V, size_t* bytes) {
    if (!bytes || B < 1 || L < 0 || V < 1 || B > 65535 || L > 65534)
        return masw_set_error(nullptr, MASW_EINVAL, "greedy: bad sizes");
    int sms = 0;
    if (accept_sms(&sms)) return masw_set_error(nullptr, MASW_ECUDA, "greedy: cannot query the device");
    *bytes = accept_ws_bytes(B, L, accept_chunks(B, L, V, sms));
    return MASW_OK;
}

extern "C" int masw_greedy_accept(const void* logits, const int* draft, int B, int L, int V, int dtype, int* tokens,
                                  int* n_emit, void* workspace, size_t workspace_bytes, masw_stream_t stream) {
    if (!logits || (!draft && L > 0) || !tokens || !n_emit || !workspace)
        return masw_set_error(nullptr, MASW_EINVAL, "greedy: NULL pointer");
    if (B < 1 || L < 0 || V < 1 || B > 65535 || L > 65534) return masw_set_error(nullptr, MASW_EINVAL, "greedy: bad sizes");
    if (dtype != MASW_BF16 && dtype != MASW_F32) return masw_set_error(nullptr, MASW_EINVAL, "greedy: bad dtype");
    if (((uintptr_t)workspace & 15) || ((uintptr_t)tokens & 3) || ((uintptr_t)n_emit & 3) || ((uintptr_t)draft & 3))
        return masw_set_error(nullptr, MASW_EINVAL, "greedy: misaligned pointer");
    int sms = 0;
    if (accept_sms(&sms)) return masw_set_error(nullptr, MASW_ECUDA, "greedy: cannot query the device");
    const int chunks = accept_chunks(B, L, V, sms);
    if (workspace_bytes < accept_ws_bytes(B, L, chunks)) return masw_set_error(nullptr, MASW_EINVAL, "greedy: workspace too small");
    AcceptParams p;
    std::memset(&p, 0, sizeof(p));
    p.logits = logits;
    p.draft = draft;
    p.tokens = tokens;
    p.n_emit = n_emit;
    const size_t n = (size_t)B * (L + 1) * chunks;
    p.part_v = (float*)workspace;
    p.part_i = (int*)((uint8_t*)workspace + n * 4);
    p.tickets = (unsigned*)((uint8_t*)workspace + ((n * 8 + 255) / 256) * 256);
    p.B = B;
    p.L = L;
    p.V = V;
    p.chunks = chunks;
    p.chunk = (V + chunks - 1) / chunks;
    p.bf16 = dtype == MASW_BF16;
    const size_t es = p.bf16 ? 2 : 4;
    p.vec = (((uintptr_t)logits & 15) == 0 && ((size_t)V * es) % 16 == 0) ? 1 : 0;
    cudaStream_t st = (cudaStream_t)stream;
    // the tickets are zero on entry (zero-filled workspace, reset by the last
    // CTA of every call): no memset node between calls
    const cudaError_t e = masw_launch(accept_kernel, dim3(chunks, L + 1, B), dim3(256), 0, st, 1, p);
    if (e != cudaSuccess) return masw_set_error(nullptr, MASW_ECUDA, std::string("greedy: ") + cudaGetErrorString(e));
    return MASW_OK;
}

extern "C" double masw_eq1_speedup(double l_acc, int l_draft, double t_draft, double t_target) {
    if (l_draft < 0 || !(t_target > 0.0) || t_draft < 0.0 || l_acc < 0.0) return -1.0;
    return (l_acc + 1.0) / (l_draft * (t_draft / t_target) + 1.0);
}
