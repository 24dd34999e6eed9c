// libmasw host side: the segmented memory pool (sink block, ring block, slot
// chain per (layer, sequence, kv head)), its device-resident counters, the
// append / rollback / load kernels, argument validation and the C entry points.
//
// Layout in HBM (head-major, so each (layer, sequence, head) block is one
// contiguous run that the decode kernel copies with a few bulk transfers):
//   pool_k, pool_v : [L][B][Hkv][C][D],  C = S + (W + R) + M_max rows:
//                    rows [0, S) sink, [S, S+W+R) ring, [S+W+R, C) slots
//   full_k, full_v : [L][B][Hkv][max_seq_len][D]  (optional contrast cache)
//   d_t, d_m       : [L][B] raw-token and slot counters (device copy; the
//                    host keeps a mirror for validation and launch sizing)
//   d_pos          : [L][B][M_max] 0-based slot position ids
#include "masw_internal.cuh"

#include <cstdlib>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <exception>
#include <new>

using namespace masw;

static thread_local std::string g_err;

int masw_set_error(masw_mem_t* mem, int code, const std::string& msg) {
    if (mem)
        mem->err = msg;
    else
        g_err = msg;
    return code;
}

namespace {

struct AppendParams {
    const uint8_t* k;
    const uint8_t* v;
    uint8_t* pool_k;
    uint8_t* pool_v;
    uint8_t* full_k;
    uint8_t* full_v;
    int* d_t;
    int* d_err;
    int layer, B, Hkv, rowb, S, Wc, C, Tmax;
    unsigned active[MASW_MAX_BATCH / 32];
};

// One CTA per sequence: token i = t+1 goes to its sink or ring row (the ring
// write overwrites, i.e. evicts, the token W+R positions older) and to row i-1
// of the full cache; then the counter advances.
__global__ void append_kernel(const __grid_constant__ AppendParams p) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    if (!((p.active[b >> 5] >> (b & 31)) & 1u)) return;
    const int lb = p.layer * p.B + b;
    const int t = p.d_t[(size_t)lb * p.Hkv];
    const int i = t + 1;
    const int row = (i <= p.S) ? i - 1 : p.S + ring_row(i, p.S, p.Wc);
    const int vpr = p.rowb / 16;
    const bool to_full = p.full_k != nullptr && i <= p.Tmax;
    for (int idx = threadIdx.x; idx < p.Hkv * vpr; idx += blockDim.x) {
        const int hh = idx / vpr, cc = idx % vpr;
        const size_t src = ((size_t)b * p.Hkv + hh) * p.rowb + cc * 16;
        const size_t dst = (((size_t)lb * p.Hkv + hh) * p.C + row) * p.rowb + cc * 16;
        const uint4 kv = *reinterpret_cast<const uint4*>(p.k + src);
        const uint4 vv = *reinterpret_cast<const uint4*>(p.v + src);
        *reinterpret_cast<uint4*>(p.pool_k + dst) = kv;
        *reinterpret_cast<uint4*>(p.pool_v + dst) = vv;
        if (to_full) {
            const size_t fd = (((size_t)lb * p.Hkv + hh) * p.Tmax + (i - 1)) * p.rowb + cc * 16;
            *reinterpret_cast<uint4*>(p.full_k + fd) = kv;
            *reinterpret_cast<uint4*>(p.full_v + fd) = vv;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && p.full_k != nullptr && i > p.Tmax) atomicExch(p.d_err + 1, MASW_ECAPACITY);
    for (int hh = threadIdx.x; hh < p.Hkv; hh += blockDim.x) p.d_t[(size_t)lb * p.Hkv + hh] = i;
}

struct RollbackParams {
    int* d_t;
    int* d_m;
    int L, B, Hkv, S, W, r, n;
    short seq[MASW_MAX_BATCH];
    int t_new[MASW_MAX_BATCH];
};

// Counters of the listed sequences go back to t_new in every layer; slots with
// tau_m > t_new are dropped (the chain keeps m(t_new) slots at most).
__global__ void rollback_kernel(const __grid_constant__ RollbackParams p) {
    pdl_wait();
    pdl_trigger();
    const int b = p.seq[blockIdx.x];
    const int tn = p.t_new[blockIdx.x];
    for (int i = threadIdx.x; i < p.L * p.Hkv; i += blockDim.x) {
        const size_t ci = ((size_t)(i / p.Hkv) * p.B + b) * p.Hkv + (i % p.Hkv);
        p.d_t[ci] = tn;
        p.d_m[ci] = imin(p.d_m[ci], slot_count(tn, p.S, p.W, p.r));
    }
}

// Copy rows [0, n) of src [n][Hkv][rowb] into dst head blocks:
// dst + h * head_stride + (row0 + j) * rowb.
// Failure-detection self-test: thread 0 waits, with the given poll budget, on
// an mbarrier that nothing ever arrives on.  The bounded wait runs out and
// records MASW_ETIMEOUT exactly as a stalled copy would in the attention
// kernels; no copy is in flight and nothing else is held, so the context stays
// usable.
__global__ void wait_timeout_probe(int* d_err, unsigned polls) {
    __shared__ uint64_t bar;
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_wait_polls(&bar, 0, d_err, polls);
    }
}

__global__ void scatter_rows_kernel(const uint8_t* src, int n, int Hkv, int rowb, uint8_t* dst,
                                    size_t head_stride, int row0) {
    const int vpr = rowb / 16;
    const size_t total = (size_t)n * Hkv * vpr;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int cc = (int)(idx % vpr);
        const size_t rest = idx / vpr;
        const int hh = (int)(rest % Hkv);
        const size_t j = rest / Hkv;
        *reinterpret_cast<uint4*>(dst + hh * head_stride + (row0 + j) * rowb + cc * 16) =
            *reinterpret_cast<const uint4*>(src + (j * Hkv + hh) * rowb + cc * 16);
    }
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

int check_layer(masw_mem_t* mem, int layer) {
    if (layer < 0 || layer >= mem->L) return masw_set_error(mem, MASW_EINVAL, "layer out of range");
    return MASW_OK;
}

int check_heads(masw_mem_t* mem, int n_q_heads) {
    if (n_q_heads < mem->Hkv || n_q_heads % mem->Hkv)
        return masw_set_error(mem, MASW_EINVAL, "n_q_heads must be a positive multiple of n_kv_heads");
    const int G = n_q_heads / mem->Hkv;
    if (G != 1 && G != 2 && G != 3 && G != 4 && G != 6 && G != 8)
        return masw_set_error(mem, MASW_EINVAL, "query heads per kv head must be 1, 2, 3, 4, 6 or 8");
    return MASW_OK;
}

void free_all(masw_mem_t* m) {
    for (const masw_mem::Alloc& a : m->allocs) cudaFree(a.raw);
    m->allocs.clear();
    m->alloc_total = 0;
}

// A handle-owned device buffer of `bytes` with a guard band on each side
// (filled with kGuardByte); false when the allocation fails or would take the
// handle past its allocation limit.
bool guarded_alloc(masw_mem_t* m, void** out, size_t bytes, const char* name) {
    const size_t raw_bytes = bytes + 2 * kGuardBytes;
    if (m->alloc_limit && m->alloc_total + raw_bytes > m->alloc_limit) return false;
    void* raw = nullptr;
    if (cudaMalloc(&raw, raw_bytes) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    m->allocs.push_back({raw, bytes, name});
    m->alloc_total += raw_bytes;
    if (cudaMemset(raw, kGuardByte, kGuardBytes) != cudaSuccess ||
        cudaMemset((uint8_t*)raw + kGuardBytes + bytes, kGuardByte, kGuardBytes) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    *out = (uint8_t*)raw + kGuardBytes;
    return true;
}

// the allocation limit of a new handle: MASW_DEVICE_MEMORY_LIMIT (bytes), 0 = none
size_t alloc_limit_from_env() {
    const char* e = std::getenv("MASW_DEVICE_MEMORY_LIMIT");
    if (!e || !*e) return 0;
    char* end = nullptr;
    const unsigned long long v = std::strtoull(e, &end, 10);
    return (end && *end == '\0') ? (size_t)v : 0;
}

bool is_device_ptr(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// Copy n rows [n][Hkv][D] (host or device) to the head blocks of `dst`.
int put_rows(masw_mem_t* mem, const void* src, int n, uint8_t* dst, size_t head_stride, int row0) {
    if (n <= 0) return MASW_OK;
    const size_t rowb = (size_t)mem->D * mem->esize;
    const size_t bytes = (size_t)n * mem->Hkv * rowb;
    const uint8_t* dsrc = (const uint8_t*)src;
    void* staging = nullptr;
    if (!is_device_ptr(src)) {
        if (cudaMalloc(&staging, bytes) != cudaSuccess) {
            cudaGetLastError();
            return masw_set_error(mem, MASW_ENOMEM, "load: staging allocation failed");
        }
        cudaError_t e = cudaMemcpy(staging, src, bytes, cudaMemcpyDefault);
        if (e != cudaSuccess) {
            cudaFree(staging);
            return masw_set_error(mem, MASW_ECUDA, std::string("load: ") + cudaGetErrorString(e));
        }
        dsrc = (const uint8_t*)staging;
    }
    const size_t vecs = bytes / 16;
    const int blocks = (int)std::min<size_t>((vecs + 255) / 256, 4096);
    scatter_rows_kernel<<<blocks, 256>>>(dsrc, n, mem->Hkv, (int)rowb, dst, head_stride, row0);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (staging) cudaFree(staging);
    if (e != cudaSuccess) return masw_set_error(mem, MASW_ECUDA, std::string("load: ") + cudaGetErrorString(e));
    return MASW_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// C entry points
// ---------------------------------------------------------------------------
extern "C" {

const char* masw_version(void) { return "0.1.0"; }

const char* masw_last_error(const masw_mem_t* mem) { return mem ? mem->err.c_str() : g_err.c_str(); }

int masw_index(int which, int t, int S, int W, int r, int R) {
    if (t < 0 || S < 0 || W < 1 || r < 1 || R < 0) return -1;
    switch (which) {
        case 0: return window_lo(t, S, W);
        case 1: return n_local(t, S, W);
        case 2: return slot_count(t, S, W, r);
        case 3: return is_boundary(t, S, W, r) ? 1 : 0;
        case 4: return (t >= 1 && t > S) ? ring_row(t, S, W + R) : -1;
        case 5: return imin(S, t) + n_local(t, S, W) + slot_count(t, S, W, r);
        default: return -1;
    }
}

int masw_mem_create(int S, int W, int r, int n_kv_heads, int head_dim, int layers, const masw_opts_t* opts,
                    masw_mem_t** out) {
    if (!out) return masw_set_error(nullptr, MASW_EINVAL, "create: out is NULL");
    *out = nullptr;
    masw_opts_t o;
    std::memset(&o, 0, sizeof(o));
    if (opts) o = *opts;
    if (o.batch == 0) o.batch = 1;
    if (o.max_seq_len == 0) o.max_seq_len = 32768;
    if (!opts) o.dtype = MASW_BF16;
    if (S < 0 || W < 1 || r < 1 || n_kv_heads < 1 || layers < 1)
        return masw_set_error(nullptr, MASW_EINVAL, "create: need S >= 0, W >= 1, r >= 1, heads >= 1, layers >= 1");
    if (head_dim != 64 && head_dim != 128) return masw_set_error(nullptr, MASW_EINVAL, "create: head_dim must be 64 or 128");
    if (o.batch < 1 || o.batch > MASW_MAX_BATCH)
        return masw_set_error(nullptr, MASW_EINVAL, "create: batch must be in [1, MASW_MAX_BATCH]");
    if (o.dtype != MASW_BF16 && o.dtype != MASW_F32) return masw_set_error(nullptr, MASW_EINVAL, "create: bad dtype");
    if (o.max_seq_len < 1 || o.rollback_reserve < 0 || !(o.softmax_scale >= 0.f) || std::isinf(o.softmax_scale))
        return masw_set_error(nullptr, MASW_EINVAL, "create: bad max_seq_len, rollback_reserve or softmax_scale");
    if (n_kv_heads > 65535 || layers > 4096)
        return masw_set_error(nullptr, MASW_EINVAL, "create: too many heads or layers");

    masw_mem_t* m = new (std::nothrow) masw_mem_t();
    if (!m) return masw_set_error(nullptr, MASW_ENOMEM, "create: host allocation failed");
    m->S = S;
    m->W = W;
    m->r = r;
    m->Hkv = n_kv_heads;
    m->D = head_dim;
    m->L = layers;
    m->B = o.batch;
    m->dtype = o.dtype;
    m->esize = o.dtype == MASW_BF16 ? 2 : 4;
    m->max_seq_len = o.max_seq_len;
    m->R = o.rollback_reserve;
    m->Wc = W + m->R;
    m->M_max = slot_count(o.max_seq_len, S, W, r);
    m->C = S + m->Wc + m->M_max;
    m->full_kv = o.full_kv ? 1 : 0;
    m->self_attend = o.slot_self_attend ? 1 : 0;
    m->scale = o.softmax_scale > 0.f ? o.softmax_scale : 1.0f / std::sqrt((float)head_dim);
    m->h_t.assign((size_t)layers * m->B, 0);
    m->h_m.assign((size_t)layers * m->B, 0);

    auto fail = [&](int code, const std::string& msg) {
        cudaGetLastError();
        free_all(m);
        delete m;
        return masw_set_error(nullptr, code, msg);
    };
    m->alloc_limit = alloc_limit_from_env();
    {
        const char* e = std::getenv("MASW_CHECK_SEGMENTS");
        m->check_segments = e && e[0] == '1';
    }
    {
        // the pools alone (before any CUDA call): a limit below them is refused here
        const size_t pool_raw = (size_t)layers * m->B * n_kv_heads * m->C * head_dim * m->esize + 2 * kGuardBytes;
        if (m->alloc_limit && 2 * pool_raw > m->alloc_limit)
            return fail(MASW_ENOMEM, "create: the pool needs " + std::to_string(2 * pool_raw) +
                                         " bytes, above the allocation limit (MASW_DEVICE_MEMORY_LIMIT) of " +
                                         std::to_string(m->alloc_limit));
    }
    if (cudaGetDevice(&m->device) != cudaSuccess) return fail(MASW_ECUDA, "create: no CUDA device");
    if (cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device) != cudaSuccess)
        return fail(MASW_ECUDA, "create: cannot query the device");

    const size_t rowb = (size_t)head_dim * m->esize;
    const size_t blocks = (size_t)layers * m->B * n_kv_heads;
    const size_t pool_bytes = blocks * m->C * rowb;
    if (!guarded_alloc(m, &m->pool_k, pool_bytes, "pool_k") || !guarded_alloc(m, &m->pool_v, pool_bytes, "pool_v"))
        return fail(MASW_ENOMEM, "create: pool allocation failed");
    if (cudaMemset(m->pool_k, 0, pool_bytes) != cudaSuccess || cudaMemset(m->pool_v, 0, pool_bytes) != cudaSuccess)
        return fail(MASW_ECUDA, "create: pool clear failed");
    if (m->full_kv) {
        const size_t fb = blocks * (size_t)m->max_seq_len * rowb;
        if (!guarded_alloc(m, &m->full_k, fb, "full_k") || !guarded_alloc(m, &m->full_v, fb, "full_v"))
            return fail(MASW_ENOMEM, "create: full-KV cache allocation failed");
    }
    const size_t lb = (size_t)layers * m->B;
    const size_t lbh = lb * n_kv_heads;
    if (!guarded_alloc(m, (void**)&m->d_t, lbh * sizeof(int), "d_t") ||
        !guarded_alloc(m, (void**)&m->d_m, lbh * sizeof(int), "d_m") ||
        !guarded_alloc(m, (void**)&m->d_pos, std::max<size_t>(1, lb * m->M_max) * sizeof(int), "d_pos") ||
        !guarded_alloc(m, (void**)&m->d_err, 4 * sizeof(int), "d_err"))
        return fail(MASW_ENOMEM, "create: counter allocation failed");
    // split scratch: enough partials for ~3 CTAs per SM at G <= 8
    const size_t pairs = (size_t)m->B * n_kv_heads;
    const size_t splits = std::min<size_t>(kMaxSplit, std::max<size_t>(8, (3 * (size_t)m->num_sms + pairs - 1) / pairs));
    m->part_floats = pairs * splits * MASW_MAX_GROUP * (head_dim + 2);
    if (!guarded_alloc(m, (void**)&m->part, m->part_floats * sizeof(float), "part") ||
        !guarded_alloc(m, (void**)&m->tickets, pairs * sizeof(unsigned), "tickets"))
        return fail(MASW_ENOMEM, "create: scratch allocation failed");
    if (cudaMemset(m->d_t, 0, lbh * sizeof(int)) != cudaSuccess || cudaMemset(m->d_m, 0, lbh * sizeof(int)) != cudaSuccess ||
        cudaMemset(m->d_pos, 0xff, std::max<size_t>(1, lb * m->M_max) * sizeof(int)) != cudaSuccess ||
        cudaMemset(m->d_err, 0, 4 * sizeof(int)) != cudaSuccess ||
        cudaMemset(m->tickets, 0, pairs * sizeof(unsigned)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
        return fail(MASW_ECUDA, "create: counter clear failed");
    *out = m;
    return MASW_OK;
}

int masw_check_guards(masw_mem_t* mem) {
    if (!mem) return masw_set_error(nullptr, MASW_EINVAL, "check_guards: NULL handle");
    MASW_CUDA_TRY(mem, cudaDeviceSynchronize());
    std::vector<unsigned char> band(kGuardBytes);
    for (const masw_mem::Alloc& a : mem->allocs) {
        for (int side = 0; side < 2; ++side) {
            const uint8_t* src = (const uint8_t*)a.raw + (side ? kGuardBytes + a.bytes : 0);
            MASW_CUDA_TRY(mem, cudaMemcpy(band.data(), src, kGuardBytes, cudaMemcpyDeviceToHost));
            for (size_t i = 0; i < kGuardBytes; ++i)
                if (band[i] != kGuardByte) {
                    const long long off = side ? (long long)(a.bytes + i) : (long long)i - (long long)kGuardBytes;
                    return masw_set_error(mem, MASW_EGUARD,
                                          std::string("check_guards: ") + a.name + " overwritten at byte offset " +
                                              std::to_string(off) + " (buffer of " + std::to_string(a.bytes) +
                                              " bytes)");
                }
        }
    }
    return MASW_OK;
}

int masw_mem_destroy(masw_mem_t* mem) {
    if (!mem) return MASW_OK;
    cudaDeviceSynchronize();
    free_all(mem);
    delete mem;
    return MASW_OK;
}

int masw_append_kv(masw_mem_t* mem, int layer, const void* k, const void* v, const uint8_t* active,
                   masw_stream_t stream) {
    if (!mem) return masw_set_error(nullptr, MASW_EINVAL, "append: NULL handle");
    try {
        if (int rc = check_layer(mem, layer)) return rc;
        if (!k || !v || !aligned16(k) || !aligned16(v))
            return masw_set_error(mem, MASW_EINVAL, "append: k and v must be non-NULL and 16-byte aligned");
        AppendParams p;
        std::memset(&p, 0, sizeof(p));
        for (int b = 0; b < mem->B; ++b) {
            if (active && !active[b]) continue;
            if (mem->h_t[(size_t)layer * mem->B + b] + 1 > mem->max_seq_len)
                return masw_set_error(mem, MASW_ECAPACITY, "append: sequence would exceed max_seq_len");
            p.active[b >> 5] |= 1u << (b & 31);
        }
        p.k = (const uint8_t*)k;
        p.v = (const uint8_t*)v;
        p.pool_k = (uint8_t*)mem->pool_k;
        p.pool_v = (uint8_t*)mem->pool_v;
        p.full_k = (uint8_t*)mem->full_k;
        p.full_v = (uint8_t*)mem->full_v;
        p.d_t = mem->d_t;
        p.d_err = mem->d_err;
        p.layer = layer;
        p.B = mem->B;
        p.Hkv = mem->Hkv;
        p.rowb = mem->D * (int)mem->esize;
        p.S = mem->S;
        p.Wc = mem->Wc;
        p.C = mem->C;
        p.Tmax = mem->max_seq_len;
        masw_note_launch(mem, (void*)stream, layer);
        MASW_CUDA_TRY(mem, masw_launch(append_kernel, dim3(mem->B), dim3(128), 0, (cudaStream_t)stream, 1, p));
        for (int b = 0; b < mem->B; ++b)
            if (!active || active[b]) mem->h_t[(size_t)layer * mem->B + b] += 1;
        return MASW_OK;
    } catch (const std::exception& e) {
        return masw_set_error(mem, MASW_EINVAL, e.what());
    } catch (...) {
        return masw_set_error(mem, MASW_EINVAL, "append: unexpected error");
    }
}

int masw_materialize_slot(masw_mem_t* mem, int layer, const int* seq_ids, int n, const void* q_g, const void* k_g,
                          const void* v_g, float* o_g, float* lse_g, int n_q_heads, masw_stream_t stream) {
    if (!mem) return masw_set_error(nullptr, MASW_EINVAL, "materialize: NULL handle");
    try {
        if (int rc = check_layer(mem, layer)) return rc;
        if (int rc = check_heads(mem, n_q_heads)) return rc;
        if (!seq_ids || n < 1 || n > mem->B) return masw_set_error(mem, MASW_EINVAL, "materialize: need 1 <= n <= batch");
        if (!q_g || !k_g || !v_g || !o_g || !aligned16(q_g) || !aligned16(k_g) || !aligned16(v_g) ||
            !aligned4(o_g) || !aligned4(lse_g))
            return masw_set_error(mem, MASW_EINVAL, "materialize: bad pointer (NULL or misaligned)");
        std::vector<char> seen(mem->B, 0);
        for (int i = 0; i < n; ++i) {
            const int b = seq_ids[i];
            if (b < 0 || b >= mem->B || seen[b]) return masw_set_error(mem, MASW_EINVAL, "materialize: bad or repeated seq id");
            seen[b] = 1;
            const int t = mem->h_t[(size_t)layer * mem->B + b];
            const int m = mem->h_m[(size_t)layer * mem->B + b];
            if (!is_boundary(t, mem->S, mem->W, mem->r) || m != slot_count(t, mem->S, mem->W, mem->r) - 1)
                return masw_set_error(mem, MASW_ESTATE, "materialize: sequence " + std::to_string(b) +
                                                            " is not at an unmaterialised compression boundary (t=" +
                                                            std::to_string(t) + ", m=" + std::to_string(m) + ")");
            if (m + 1 > mem->M_max) return masw_set_error(mem, MASW_ECAPACITY, "materialize: slot chain is full");
        }
        int rc = masw_launch_decode(mem, kModeSlot, layer, q_g, n_q_heads, o_g, lse_g, seq_ids, n, k_g, v_g,
                                    (cudaStream_t)stream);
        if (rc) return rc;
        for (int i = 0; i < n; ++i) mem->h_m[(size_t)layer * mem->B + seq_ids[i]] += 1;
        return MASW_OK;
    } catch (const std::exception& e) {
        return masw_set_error(mem, MASW_EINVAL, e.what());
    } catch (...) {
        return masw_set_error(mem, MASW_EINVAL, "materialize: unexpected error");
    }
}

int masw_rollback(masw_mem_t* mem, const int* seq_ids, const int* t_new, int n, masw_stream_t stream) {
    if (!mem) return masw_set_error(nullptr, MASW_EINVAL, "rollback: NULL handle");
    if (!seq_ids || !t_new || n < 1 || n > mem->B) return masw_set_error(mem, MASW_EINVAL, "rollback: need 1 <= n <= batch");
    RollbackParams p;
    std::memset(&p, 0, sizeof(p));
    std::vector<char> seen(mem->B, 0);
    for (int i = 0; i < n; ++i) {
        const int b = seq_ids[i];
        if (b < 0 || b >= mem->B || seen[b]) return masw_set_error(mem, MASW_EINVAL, "rollback: bad or repeated seq id");
        seen[b] = 1;
        for (int l = 0; l < mem->L; ++l) {
            const int t = mem->h_t[(size_t)l * mem->B + b];
            if (t_new[i] < 0 || t_new[i] > t || t - t_new[i] > mem->R)
                return masw_set_error(mem, MASW_ESTATE, "rollback: depth must be within [0, rollback_reserve]");
        }
        p.seq[i] = (short)b;
        p.t_new[i] = t_new[i];
    }
    p.d_t = mem->d_t;
    p.d_m = mem->d_m;
    p.L = mem->L;
    p.B = mem->B;
    p.Hkv = mem->Hkv;
    p.S = mem->S;
    p.W = mem->W;
    p.r = mem->r;
    p.n = n;
    masw_note_launch(mem, (void*)stream, -1);   // counters only (re-checked by every decode launch)
    MASW_CUDA_TRY(mem, masw_launch(rollback_kernel, dim3(n), dim3(32), 0, (cudaStream_t)stream, 1, p));
    for (int i = 0; i < n; ++i)
        for (int l = 0; l < mem->L; ++l) {
            const size_t lb = (size_t)l * mem->B + seq_ids[i];
            mem->h_t[lb] = t_new[i];
            mem->h_m[lb] = imin(mem->h_m[lb], slot_count(t_new[i], mem->S, mem->W, mem->r));
        }
    return MASW_OK;
}

static int attn_common(masw_mem_t* mem, int mode, int layer, const void* q, int n_q_heads, float* o, float* lse,
                       masw_stream_t stream) {
    if (!mem) return masw_set_error(nullptr, MASW_EINVAL, "attn: NULL handle");
    try {
        if (int rc = check_layer(mem, layer)) return rc;
        if (int rc = check_heads(mem, n_q_heads)) return rc;
        if (!q || !o || !aligned16(q) || !aligned4(o) || !aligned4(lse))
            return masw_set_error(mem, MASW_EINVAL, "attn: bad pointer (NULL or misaligned)");
        if (mode == kModeFull && !mem->full_kv)
            return masw_set_error(mem, MASW_ESTATE, "full_attn: pool was created without full_kv");
        return masw_launch_decode(mem, mode, layer, q, n_q_heads, o, lse, nullptr, mem->B, nullptr, nullptr,
                                  (cudaStream_t)stream);
    } catch (const std::exception& e) {
        return masw_set_error(mem, MASW_EINVAL, e.what());
    } catch (...) {
        return masw_set_error(mem, MASW_EINVAL, "attn: unexpected error");
    }
}

int masw_draft_attn(masw_mem_t* mem, int layer, const void* q, int n_q_heads, float* o, float* lse,
                    masw_stream_t stream) {
    return attn_common(mem, kModeDraft, layer, q, n_q_heads, o, lse, stream);
}

int masw_full_attn(masw_mem_t* mem, int layer, const void* q, int n_q_heads, float* o, float* lse,
                   masw_stream_t stream) {
    return attn_common(mem, kModeFull, layer, q, n_q_heads, o, lse, stream);
}

static int step_common(masw_mem_t* mem, int mode, int layer, const void* q, const void* k, const void* v,
                       const uint8_t* active, int n_q_heads, float* o, float* lse, masw_stream_t stream) {
    if (!mem) return masw_set_error(nullptr, MASW_EINVAL, "step: NULL handle");
    try {
        if (int rc = check_layer(mem, layer)) return rc;
        if (int rc = check_heads(mem, n_q_heads)) return rc;
        if (!q || !o || !k || !v || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned4(o) || !aligned4(lse))
            return masw_set_error(mem, MASW_EINVAL, "step: bad pointer (NULL or misaligned)");
        if (mode == kModeFull && !mem->full_kv)
            return masw_set_error(mem, MASW_ESTATE, "full_step: pool was created without full_kv");
        if (mem->dtype != MASW_BF16) {
            // fp32 pools: the same two steps as separate launches
            int rc = masw_append_kv(mem, layer, k, v, active, stream);
            if (rc) return rc;
            return attn_common(mem, mode, layer, q, n_q_heads, o, lse, stream);
        }
        unsigned bits[MASW_MAX_BATCH / 32] = {0};
        for (int b = 0; b < mem->B; ++b) {
            if (active && !active[b]) continue;
            if (mem->h_t[(size_t)layer * mem->B + b] + 1 > mem->max_seq_len)
                return masw_set_error(mem, MASW_ECAPACITY, "step: sequence would exceed max_seq_len");
            bits[b >> 5] |= 1u << (b & 31);
        }
        int rc = masw_launch_decode(mem, mode, layer, q, n_q_heads, o, lse, nullptr, mem->B, k, v,
                                    (cudaStream_t)stream, bits);
        if (rc) return rc;
        for (int b = 0; b < mem->B; ++b)
            if (!active || active[b]) mem->h_t[(size_t)layer * mem->B + b] += 1;
        return MASW_OK;
    } catch (const std::exception& e) {
        return masw_set_error(mem, MASW_EINVAL, e.what());
    } catch (...) {
        return masw_set_error(mem, MASW_EINVAL, "step: unexpected error");
    }
}

int masw_draft_step(masw_mem_t* mem, int layer, const void* q, const void* k, const void* v, const uint8_t* active,
                    int n_q_heads, float* o, float* lse, masw_stream_t stream) {
    return step_common(mem, kModeDraft, layer, q, k, v, active, n_q_heads, o, lse, stream);
}

int masw_full_step(masw_mem_t* mem, int layer, const void* q, const void* k, const void* v, const uint8_t* active,
                   int n_q_heads, float* o, float* lse, masw_stream_t stream) {
    return step_common(mem, kModeFull, layer, q, k, v, active, n_q_heads, o, lse, stream);
}

int masw_draft_step_slot(masw_mem_t* mem, int layer, const void* q, const void* k, const void* v,
                         const uint8_t* active, int n_q_heads, float* o, float* lse, const int* seq_ids, int n,
                         const void* q_g, const void* k_g, const void* v_g, float* o_g, float* lse_g,
                         masw_stream_t stream) {
    if (!mem) return masw_set_error(nullptr, MASW_EINVAL, "step_slot: NULL handle");
    try {
        if (int rc = check_layer(mem, layer)) return rc;
        if (int rc = check_heads(mem, n_q_heads)) return rc;
        if (!seq_ids || n < 1 || n > mem->B) return masw_set_error(mem, MASW_EINVAL, "step_slot: need 1 <= n <= batch");
        if (!q || !o || !k || !v || !q_g || !k_g || !v_g || !o_g || !aligned16(q) || !aligned16(k) ||
            !aligned16(v) || !aligned16(q_g) || !aligned16(k_g) || !aligned16(v_g) || !aligned4(o) ||
            !aligned4(lse) || !aligned4(o_g) || !aligned4(lse_g))
            return masw_set_error(mem, MASW_EINVAL, "step_slot: bad pointer (NULL or misaligned)");
        // every listed sequence appends this step and lands on an unmaterialised boundary
        std::vector<char> seen(mem->B, 0);
        for (int i = 0; i < n; ++i) {
            const int b = seq_ids[i];
            if (b < 0 || b >= mem->B || seen[b]) return masw_set_error(mem, MASW_EINVAL, "step_slot: bad or repeated seq id");
            seen[b] = 1;
            if (active && !active[b]) return masw_set_error(mem, MASW_ESTATE, "step_slot: listed sequence is not active");
            const int t1 = mem->h_t[(size_t)layer * mem->B + b] + 1;
            const int m = mem->h_m[(size_t)layer * mem->B + b];
            if (!is_boundary(t1, mem->S, mem->W, mem->r) || m != slot_count(t1, mem->S, mem->W, mem->r) - 1)
                return masw_set_error(mem, MASW_ESTATE, "step_slot: sequence " + std::to_string(b) +
                                                            " does not reach an unmaterialised boundary this step");
            if (m + 1 > mem->M_max) return masw_set_error(mem, MASW_ECAPACITY, "step_slot: slot chain is full");
        }
        const int G = n_q_heads / mem->Hkv;
        if (mem->dtype != MASW_BF16 || G > 4 || mem->self_attend) {
            // no shared query tile: the two calls as two launches
            int rc = masw_draft_step(mem, layer, q, k, v, active, n_q_heads, o, lse, stream);
            if (rc) return rc;
            return masw_materialize_slot(mem, layer, seq_ids, n, q_g, k_g, v_g, o_g, lse_g, n_q_heads, stream);
        }
        unsigned bits[MASW_MAX_BATCH / 32] = {0};
        for (int b = 0; b < mem->B; ++b) {
            if (active && !active[b]) continue;
            if (mem->h_t[(size_t)layer * mem->B + b] + 1 > mem->max_seq_len)
                return masw_set_error(mem, MASW_ECAPACITY, "step_slot: sequence would exceed max_seq_len");
            bits[b >> 5] |= 1u << (b & 31);
        }
        SlotFuse fuse{seq_ids, n, q_g, k_g, v_g, o_g, lse_g};
        int rc = masw_launch_decode(mem, kModeDraft, layer, q, n_q_heads, o, lse, nullptr, mem->B, k, v,
                                    (cudaStream_t)stream, bits, &fuse);
        if (rc) return rc;
        for (int b = 0; b < mem->B; ++b)
            if (!active || active[b]) mem->h_t[(size_t)layer * mem->B + b] += 1;
        for (int i = 0; i < n; ++i) mem->h_m[(size_t)layer * mem->B + seq_ids[i]] += 1;
        return MASW_OK;
    } catch (const std::exception& e) {
        return masw_set_error(mem, MASW_EINVAL, e.what());
    } catch (...) {
        return masw_set_error(mem, MASW_EINVAL, "step_slot: unexpected error");
    }
}

int masw_mem_load(masw_mem_t* mem, int layer, int seq, int t, const void* k_raw, const void* v_raw,
                  const void* k_slots, const void* v_slots, int n_slots) {
    if (!mem) return masw_set_error(nullptr, MASW_EINVAL, "load: NULL handle");
    try {
        if (int rc = check_layer(mem, layer)) return rc;
        if (seq < 0 || seq >= mem->B) return masw_set_error(mem, MASW_EINVAL, "load: seq out of range");
        if (t < 0 || t > mem->max_seq_len) return masw_set_error(mem, MASW_ECAPACITY, "load: t exceeds max_seq_len");
        if (t > 0 && (!k_raw || !v_raw)) return masw_set_error(mem, MASW_EINVAL, "load: NULL raw K/V");
        if (n_slots != slot_count(t, mem->S, mem->W, mem->r))
            return masw_set_error(mem, MASW_EINVAL, "load: n_slots must equal max(0, (t-S-W)/r)");
        if (n_slots > 0 && (!k_slots || !v_slots)) return masw_set_error(mem, MASW_EINVAL, "load: NULL slot K/V");
        if (n_slots > mem->M_max) return masw_set_error(mem, MASW_ECAPACITY, "load: slot chain is full");
        masw_note_launch(mem, nullptr, -2);   // set-up: no early copies right after a load
        MASW_CUDA_TRY(mem, cudaDeviceSynchronize());
        const size_t rowb = (size_t)mem->D * mem->esize;
        const size_t lb = (size_t)layer * mem->B + seq;
        const size_t hs = (size_t)mem->C * rowb;
        const size_t src_row = (size_t)mem->Hkv * rowb;
        uint8_t* pk = (uint8_t*)mem->pool_k + lb * mem->Hkv * hs;
        uint8_t* pv = (uint8_t*)mem->pool_v + lb * mem->Hkv * hs;
        const uint8_t* kr = (const uint8_t*)k_raw;
        const uint8_t* vr = (const uint8_t*)v_raw;
        // sink: tokens 1..min(S, t) -> rows 0..
        const int ns = imin(mem->S, t);
        int rc;
        if ((rc = put_rows(mem, kr, ns, pk, hs, 0)) || (rc = put_rows(mem, vr, ns, pv, hs, 0))) return rc;
        // ring: the last min(W+R, t-S) non-sink tokens, at rows (i-S-1) mod (W+R)
        if (t > mem->S) {
            int i = imax(mem->S + 1, t - mem->Wc + 1);
            while (i <= t) {
                const int row = ring_row(i, mem->S, mem->Wc);
                const int run = imin(t - i + 1, mem->Wc - row);
                const uint8_t* ks = kr + (size_t)(i - 1) * src_row;
                const uint8_t* vs = vr + (size_t)(i - 1) * src_row;
                if ((rc = put_rows(mem, ks, run, pk, hs, mem->S + row)) ||
                    (rc = put_rows(mem, vs, run, pv, hs, mem->S + row)))
                    return rc;
                i += run;
            }
        }
        // slots
        if ((rc = put_rows(mem, k_slots, n_slots, pk, hs, mem->S + mem->Wc)) ||
            (rc = put_rows(mem, v_slots, n_slots, pv, hs, mem->S + mem->Wc)))
            return rc;
        // full cache
        if (mem->full_kv) {
            const size_t fhs = (size_t)mem->max_seq_len * rowb;
            uint8_t* fk = (uint8_t*)mem->full_k + lb * mem->Hkv * fhs;
            uint8_t* fv = (uint8_t*)mem->full_v + lb * mem->Hkv * fhs;
            if ((rc = put_rows(mem, kr, t, fk, fhs, 0)) || (rc = put_rows(mem, vr, t, fv, fhs, 0))) return rc;
        }
        // counters and slot position ids
        std::vector<int> pos(std::max(1, mem->M_max), -1);
        for (int j = 0; j < n_slots; ++j) pos[j] = mem->S + mem->W + (j + 1) * mem->r;
        std::vector<int> tv(mem->Hkv, t), mv(mem->Hkv, n_slots);
        MASW_CUDA_TRY(mem, cudaMemcpy(mem->d_t + lb * mem->Hkv, tv.data(), mem->Hkv * sizeof(int), cudaMemcpyHostToDevice));
        MASW_CUDA_TRY(mem, cudaMemcpy(mem->d_m + lb * mem->Hkv, mv.data(), mem->Hkv * sizeof(int), cudaMemcpyHostToDevice));
        if (mem->M_max > 0)
            MASW_CUDA_TRY(mem, cudaMemcpy(mem->d_pos + lb * mem->M_max, pos.data(), mem->M_max * sizeof(int),
                                          cudaMemcpyHostToDevice));
        mem->h_t[lb] = t;
        mem->h_m[lb] = n_slots;
        return MASW_OK;
    } catch (const std::exception& e) {
        return masw_set_error(mem, MASW_EINVAL, e.what());
    } catch (...) {
        return masw_set_error(mem, MASW_EINVAL, "load: unexpected error");
    }
}

int masw_mem_export(masw_mem_t* mem, int layer, int seq, void* k_out, void* v_out, int* slot_pos) {
    if (!mem) return masw_set_error(nullptr, MASW_EINVAL, "export: NULL handle");
    if (int rc = check_layer(mem, layer)) return rc;
    if (seq < 0 || seq >= mem->B) return masw_set_error(mem, MASW_EINVAL, "export: seq out of range");
    const size_t lb = (size_t)layer * mem->B + seq;
    const size_t blk = (size_t)mem->Hkv * mem->C * mem->D * mem->esize;
    MASW_CUDA_TRY(mem, cudaDeviceSynchronize());
    if (k_out) MASW_CUDA_TRY(mem, cudaMemcpy(k_out, (uint8_t*)mem->pool_k + lb * blk, blk, cudaMemcpyDefault));
    if (v_out) MASW_CUDA_TRY(mem, cudaMemcpy(v_out, (uint8_t*)mem->pool_v + lb * blk, blk, cudaMemcpyDefault));
    if (slot_pos && mem->M_max > 0)
        MASW_CUDA_TRY(mem, cudaMemcpy(slot_pos, mem->d_pos + lb * mem->M_max, mem->M_max * sizeof(int),
                                      cudaMemcpyDeviceToHost));
    return MASW_OK;
}

int masw_query(masw_mem_t* mem, int layer, int seq, masw_state_t* out) {
    if (!mem || !out) return masw_set_error(mem, MASW_EINVAL, "query: NULL argument");
    if (int rc = check_layer(mem, layer)) return rc;
    if (seq < 0 || seq >= mem->B) return masw_set_error(mem, MASW_EINVAL, "query: seq out of range");
    const size_t lb = (size_t)layer * mem->B + seq;
    std::memset(out, 0, sizeof(*out));
    out->t = mem->h_t[lb];
    out->m = mem->h_m[lb];
    out->n_sink = imin(mem->S, out->t);
    out->n_local = n_local(out->t, mem->S, mem->W);
    out->ring_rows = mem->Wc;
    out->rows = mem->C;
    out->slot_capacity = mem->M_max;
    MASW_CUDA_TRY(mem, cudaDeviceSynchronize());
    std::vector<int> tv(mem->Hkv), mv(mem->Hkv);
    MASW_CUDA_TRY(mem, cudaMemcpy(tv.data(), mem->d_t + lb * mem->Hkv, mem->Hkv * sizeof(int), cudaMemcpyDeviceToHost));
    MASW_CUDA_TRY(mem, cudaMemcpy(mv.data(), mem->d_m + lb * mem->Hkv, mem->Hkv * sizeof(int), cudaMemcpyDeviceToHost));
    out->dev_t = tv[0];
    out->dev_m = mv[0];
    for (int h = 1; h < mem->Hkv; ++h)   // every kv head's copy must agree
        if (tv[h] != tv[0] || mv[h] != mv[0]) out->dev_t = out->dev_m = -1;
    return MASW_OK;
}

int masw_selftest_timeout(masw_mem_t* mem, int polls, masw_stream_t stream) {
    if (!mem) return masw_set_error(nullptr, MASW_EINVAL, "selftest: NULL handle");
    if (polls < 1 || polls > (1 << 20)) return masw_set_error(mem, MASW_EINVAL, "selftest: polls must be in [1, 2^20]");
    MASW_CUDA_TRY(mem, masw_launch(wait_timeout_probe, dim3(1), dim3(32), 0, (cudaStream_t)stream, 1, mem->d_err,
                                   (unsigned)polls));
    return MASW_OK;
}

int masw_sync(masw_mem_t* mem, masw_stream_t stream) {
    if (!mem) return masw_set_error(nullptr, MASW_EINVAL, "sync: NULL handle");
    MASW_CUDA_TRY(mem, cudaStreamSynchronize((cudaStream_t)stream));
    int err[4] = {0, 0, 0, 0};
    MASW_CUDA_TRY(mem, cudaMemcpy(err, mem->d_err, sizeof(err), cudaMemcpyDeviceToHost));
    if (err[0] || err[1] || err[2] || err[3]) {
        const int zero[4] = {0, 0, 0, 0};
        MASW_CUDA_TRY(mem, cudaMemcpy(mem->d_err, zero, sizeof(zero), cudaMemcpyHostToDevice));
        if (err[3])
            return masw_set_error(mem, MASW_EGUARD,
                                  "a decode kernel's segment table left its (layer, sequence, kv head) block");
        if (err[0]) return masw_set_error(mem, MASW_ETIMEOUT, "a device-side bounded wait ran out");
        if (err[2]) return masw_set_error(mem, MASW_ECUDA, "a kernel's shared memory was not 1024-byte aligned");
        return masw_set_error(mem, MASW_ECAPACITY, "a device-side append exceeded max_seq_len");
    }
    return MASW_OK;
}

}  // extern "C"
