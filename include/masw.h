/*
 * masw.h -- C ABI of libmasw: GB300 (sm_103a) draft-side compressed KV memory
 * and attention for Memory-Augmented Sliding-Window (MASW) drafting.
 *
 * Pages this interface follows (titles abbreviated):
 *   [EN] "Strong Drafts Need Compact Memories: A Technical Review of
 *        Memory-Augmented Sliding-Window (MASW) Drafting for Long-Context
 *        Speculative Decoding", sections 2.3 (Eq. 2), 3.1 (Eq. 4), 3.2
 *        (Algorithm 1) and 3.3 (Algorithm 2).
 *
 * Model of the state.  For every (layer l, sequence b) the library keeps the
 * draft working memory of Eq. 4, M_t = M_sink u M_local,t u M_slot,t:
 *   - M_sink : exact K/V of raw tokens 1..S, never evicted;
 *   - M_local,t : exact K/V of raw tokens max(S+1, t-W+1) .. t, held in a ring
 *     of W + R rows (R = rollback reserve, 0 by default); token i sits in ring
 *     row (i-S-1) mod (W+R), so appending token i overwrites (evicts) token
 *     i-W-R;
 *   - M_slot,t : an append-only chain of memory slots, one K/V row per kv head
 *     each, one slot per r raw tokens that have left the window.  Slot g_m is
 *     written at boundary tau_m = S + W + m*r.
 * Token ids on the pages are 1-based; the library stores row p = i-1 and
 * reports 0-based position ids.
 *
 * Conventions for every call:
 *   - Return value is a status: MASW_OK (0) or a negative MASW_E* code.  No C++
 *     exception and no abort() crosses this interface.  masw_last_error()
 *     gives a message for the last failing call on a handle.
 *   - Pointers named "device" must be CUDA device (or managed) memory owned by
 *     the caller; the library never frees them.  The memory pool, its counters
 *     and its scratch are owned by the handle: allocated in masw_mem_create,
 *     freed in masw_mem_destroy.
 *   - Compute calls are asynchronous on the given stream (a cudaStream_t,
 *     NULL = legacy default stream).  Argument and state errors are returned
 *     synchronously, before anything is enqueued.  Errors raised inside a
 *     kernel (a bounded wait that ran out) are recorded in a device flag and
 *     returned by the next masw_sync().
 *   - A handle is used from one host thread and one stream at a time; calls on
 *     one handle that overlap on the GPU race on the pool and its scratch.
 *   - Element types: MASW_BF16 (bfloat16) or MASW_F32 for Q/K/V inputs, chosen
 *     at create time.  Attention outputs O are float32; LSE outputs are the
 *     float32 natural-log normaliser log sum_j exp(scale * q.k_j).
 *   - Layouts are C-contiguous, innermost dimension last.  Q/K/V pointers must
 *     be 16-byte aligned, O/LSE pointers 4-byte aligned.
 */
#ifndef MASW_H
#define MASW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define MASW_OK          0
#define MASW_EINVAL     -1  /* bad argument (size, pointer, layer, dtype, head counts) */
#define MASW_ENOMEM     -2  /* device allocation failed */
#define MASW_ECAPACITY  -3  /* pool capacity exceeded (max_seq_len, slot chain) */
#define MASW_ESTATE     -4  /* call not valid in the current state (e.g. not at a boundary) */
#define MASW_ECUDA      -5  /* a CUDA runtime call failed */
#define MASW_ETIMEOUT   -6  /* a bounded device-side wait ran out (kernel returned early) */
#define MASW_EGUARD     -7  /* out of bounds: a guard band around a handle-owned buffer was
                               overwritten, or a decode kernel's segment table left its block */

/* ---- element types ------------------------------------------------------- */
#define MASW_F32   0
#define MASW_BF16  1

/* ---- limits --------------------------------------------------------------- */
#define MASW_MAX_BATCH  512   /* sequences per handle */
#define MASW_MAX_GROUP  8     /* query heads per kv head (G = Hq / Hkv): 1,2,3,4,6,8 */

typedef struct masw_mem masw_mem_t;
typedef void* masw_stream_t;   /* a cudaStream_t */

typedef struct {
    int   batch;            /* sequences held, 1..MASW_MAX_BATCH (0 -> 1) */
    int   dtype;            /* MASW_BF16 (default) or MASW_F32 */
    int   max_seq_len;      /* longest sequence, in raw tokens; sizes the slot chain
                               (m(max_seq_len) slots) and the full-KV cache.
                               0 -> 32768 */
    float softmax_scale;    /* 0 -> 1/sqrt(head_dim) (Eq. 2) */
    int   slot_self_attend; /* 0 (default): slot query g_m does not read its own K/V;
                               1: it does (standard causal diagonal) */
    int   full_kv;          /* 1: also keep an uncompressed cache of max_seq_len
                               rows per (layer, sequence, kv head) for masw_full_attn */
    int   rollback_reserve; /* R extra ring rows; masw_rollback can undo up to R tokens */
} masw_opts_t;

typedef struct {
    int t;          /* raw tokens appended (host mirror) */
    int n_sink;     /* min(S, t) */
    int n_local;    /* tokens in the local window: clamp(t - S, 0, W) */
    int m;          /* slots in the chain (host mirror) */
    int dev_t;      /* device counters, read back synchronously; equal to t, m */
    int dev_m;      /*   unless a captured graph replay changed the state */
    int ring_rows;  /* W + R */
    int rows;       /* rows per (layer, sequence, kv head) block: S + W + R + M_max */
    int slot_capacity; /* M_max */
} masw_state_t;

/* ---- lifetime -------------------------------------------------------------- */

/* Create a pool for `layers` layers x opts->batch sequences x n_kv_heads heads
 * of head_dim, with S sink tokens (S >= 0), W local-window tokens (W >= 1) and
 * one slot per r evicted tokens (r >= 1) ([EN] §3.1 Eq. 4, §3.2 Algorithm 1).
 * head_dim must be 64 or 128.  opts may be NULL (batch 1, bf16, max_seq_len
 * 32768).  Allocates the pool (K and V: layers*batch*Hkv*(S+W+R+M_max)*D
 * elements each), the optional full-KV cache, counters and split scratch on
 * the current device.  On failure *out is NULL.
 * Every handle-owned device buffer carries a 4 KiB guard band on each side
 * (see masw_check_guards).  If the environment variable
 * MASW_DEVICE_MEMORY_LIMIT holds a byte count, create allocates at most that
 * much device memory in total (guards included) and otherwise fails with
 * MASW_ENOMEM, freeing what it had allocated: a way to exercise the
 * out-of-memory path without exhausting the device.  A limit below the pool's
 * own size is refused before any CUDA call.  If MASW_CHECK_SEGMENTS is "1" at
 * create, every bf16 decode launch of the handle first checks on the host that
 * each run of pool rows its CTAs will copy lies inside its own (layer,
 * sequence, kv head) block and region, and fails with MASW_EGUARD (nothing
 * launched) otherwise: a debug mode, whose host time per launch grows with
 * rows x kv heads. */
int masw_mem_create(int S, int W, int r, int n_kv_heads, int head_dim, int layers,
                    const masw_opts_t* opts, masw_mem_t** out);

/* Free everything the handle owns.  NULL is accepted.  Synchronises the device. */
int masw_mem_destroy(masw_mem_t* mem);

/* Out-of-bounds write check: synchronises the device, then reads back the guard
 * bands (4 KiB of 0xC3 before and after each handle-owned device buffer: the
 * pools, the full-KV cache, counters, slot ids, split partials and tickets)
 * and returns MASW_OK if all are intact, MASW_EGUARD otherwise (the message
 * names the buffer and the byte offset of the first changed guard byte; a
 * negative offset lies before the buffer).  Synchronous. */
int masw_check_guards(masw_mem_t* mem);

/* Message for the last failing call on `mem` (or on a NULL handle / stateless call). */
const char* masw_last_error(const masw_mem_t* mem);

/* ---- memory maintenance ---------------------------------------------------- */

/* Append one raw token to every active sequence of `layer` ([EN] §3.3
 * Algorithm 2): k, v are device [batch, Hkv, D] in the pool dtype.
 * Token i = t+1 goes to sink row i-1 if i <= S, else to ring row (i-S-1) mod
 * (W+R); that write is the eviction of [EN] §3.2 Algorithm 1.  With
 * full_kv it is also written to row i-1 of the full cache.  active: host
 * [batch] bytes, nonzero = append; NULL = all.  ECAPACITY when t would exceed
 * max_seq_len. */
int masw_append_kv(masw_mem_t* mem, int layer, const void* k, const void* v,
                   const uint8_t* active, masw_stream_t stream);

/* Memory-slot write at a compression boundary ([EN] §3.2 Algorithm 1)
 * for the n sequences in the host list seq_ids.  For each listed
 * sequence b, which must have t = tau_m = S + W + m*r for the next chain index
 * m (ESTATE otherwise):
 *   1. the slot query q_g attends, under the structured mask, to M_sink,
 *      M_local,tau_m and slots 1..m-1 (and to itself only with
 *      slot_self_attend); O_g and its LSE are returned;
 *   2. K_g, V_g (already projected by the caller's mirrored W_K,g / W_V,g)
 *      are appended as slot m;
 *   3. slot m gets position id tau_m (0-based id of the raw token after it).
 * q_g: device [n, n_q_heads, D]; k_g, v_g: device [n, Hkv, D]; o_g: device
 * float [n, n_q_heads, D]; lse_g: device float [n, n_q_heads] or NULL.
 * seq_ids must be distinct.  ECAPACITY when the chain is full.  Call it after
 * masw_draft_attn of the boundary step, so that the query at tau_m sees m-1
 * slots. */
int masw_materialize_slot(masw_mem_t* mem, int layer, const int* seq_ids, int n,
                          const void* q_g, const void* k_g, const void* v_g,
                          float* o_g, float* lse_g, int n_q_heads, masw_stream_t stream);

/* Draft prefill of one (layer, seq) under the structured write mask ([EN] §3.3
 * Algorithm 2, mask of §3.2 Algorithm 1): one attention pass over
 * a prefix of T raw tokens with the M = max(0, (T-S-W)/r) slot tokens
 * interleaved, then M_0 is stored as the sequence's memory (sink rows, the last
 * W+R raw tokens in their ring rows, slots 1..M with position ids tau_1..tau_M,
 * and the full cache with full_kv), so that decoding continues at t = T.
 *   raw token i (1-based) attends to sink tokens 1..min(S, i), raw tokens
 *   max(S+1, i-W+1)..i and slots m with tau_m < i;
 *   slot token g_m attends to the sink, raw tokens tau_m-W+1..tau_m and slots
 *   1..m-1 (1..m with slot_self_attend).
 * q_raw: device [T, n_q_heads, D]; k_raw, v_raw: device [T, Hkv, D];
 * q_slot: device [M, n_q_heads, D]; k_slot, v_slot: device [M, Hkv, D] (the
 * slot tokens' projections; may be NULL when M = 0); all bf16, 16-byte aligned.
 * o_raw: device float [T, n_q_heads, D]; lse_raw: device float [T, n_q_heads]
 * or NULL; o_slot, lse_slot likewise [M, ...].  bf16 pools with head_dim 128
 * only (EINVAL otherwise); ECAPACITY when T > max_seq_len or M exceeds the slot
 * chain.  The previous state of (layer, seq) is replaced; inputs must stay
 * valid until the stream reaches the call. */
int masw_prefill(masw_mem_t* mem, int layer, int seq, int T,
                 const void* q_raw, const void* k_raw, const void* v_raw,
                 const void* q_slot, const void* k_slot, const void* v_slot, int n_q_heads,
                 float* o_raw, float* lse_raw, float* o_slot, float* lse_slot,
                 masw_stream_t stream);

/* Undo the last t[b] - t_new[i] raw tokens of the listed sequences in every
 * layer ([EN] §3.3 Algorithm 2): counters go back to t_new and slots
 * with tau_m > t_new are dropped.  Needs 0 <= t - t_new <= R in every layer
 * (ESTATE otherwise), because the ring rows of the restored window must not
 * have been overwritten.  seq_ids, t_new: host arrays of n. */
int masw_rollback(masw_mem_t* mem, const int* seq_ids, const int* t_new, int n,
                  masw_stream_t stream);

/* ---- attention --------------------------------------------------------------- */

/* Draft decode attention over M_t ([EN] §2.3 Eq. 2 over the set of §3.1 Eq. 4):
 * O[b, h] = softmax(scale * q[b,h] . K_j) V_j over j in sink u window u slots
 * of (layer, b), kv head h / (n_q_heads / Hkv).  The segments are walked in
 * place (ring in physical row order; softmax does not depend on order).
 * q: device [batch, n_q_heads, D] (pool dtype); o: device float
 * [batch, n_q_heads, D]; lse: device float [batch, n_q_heads] or NULL.
 * A sequence with t = 0 gets O = 0 and LSE = -inf. */
int masw_draft_attn(masw_mem_t* mem, int layer, const void* q, int n_q_heads,
                    float* o, float* lse, masw_stream_t stream);

/* Full-KV decode attention over raw tokens 1..t ([EN] §2.3 Eq. 2 with the
 * whole prefix; the uncompressed draft the pages contrast against).  Same
 * arguments as masw_draft_attn.  ESTATE unless the pool was created with
 * full_kv = 1. */
int masw_full_attn(masw_mem_t* mem, int layer, const void* q, int n_q_heads,
                   float* o, float* lse, masw_stream_t stream);

/* One draft decode step of `layer` in a single launch: masw_append_kv followed
 * by masw_draft_attn ([EN] §3.3 Algorithm 2 -- the new token joins the
 * window, evicting the oldest, and the query at t+1 attends over M_{t+1}).
 * k, v: device [batch, Hkv, D] (the new token); q: device [batch, n_q_heads, D];
 * o, lse as in masw_draft_attn; active as in masw_append_kv (inactive
 * sequences are not appended and their query sees M_t).  The new row is read
 * straight from k/v by the attention and stored in the pool by the same launch.
 * Results equal the two separate calls up to fp32 summation order.  fp32
 * pools run the two calls as two launches. */
int masw_draft_step(masw_mem_t* mem, int layer, const void* q, const void* k, const void* v,
                    const uint8_t* active, int n_q_heads, float* o, float* lse,
                    masw_stream_t stream);

/* The draft step at a compression boundary in one launch: masw_draft_step
 * followed by masw_materialize_slot for the n listed sequences, which must each
 * be active and reach an unmaterialised boundary tau_m with this step's token
 * (ESTATE otherwise).  At tau_m the slot query's structured mask ([EN] §3.2
 * Algorithm 1: sink, window at tau_m, slots 1..m-1) is exactly the draft
 * query's working set M_{tau_m} (which does not yet hold g_m, [EN] §3.2
 * Algorithm 1), so both queries share every K/V row read.  Arguments:
 * those of masw_draft_step, then those of masw_materialize_slot.  fp32 pools,
 * more than 4 query heads per kv head, or slot_self_attend = 1 run the two
 * calls as two launches. */
int masw_draft_step_slot(masw_mem_t* mem, int layer, const void* q, const void* k, const void* v,
                         const uint8_t* active, int n_q_heads, float* o, float* lse,
                         const int* seq_ids, int n, const void* q_g, const void* k_g,
                         const void* v_g, float* o_g, float* lse_g, masw_stream_t stream);

/* The same fused step for the full-KV contrast: masw_append_kv followed by
 * masw_full_attn.  ESTATE unless the pool was created with full_kv = 1. */
int masw_full_step(masw_mem_t* mem, int layer, const void* q, const void* k, const void* v,
                   const uint8_t* active, int n_q_heads, float* o, float* lse,
                   masw_stream_t stream);

/* Target verify attention ([EN] §3.3 Algorithm 2), stateless: Lq query
 * positions per sequence against an uncompressed cache, causal inside the
 * block.  Query j (0-based) of sequence b sees keys 0 .. kv_len[b]-Lq+j
 * (kv_len counts the block's own Lq tokens).  bf16 only.
 * q: device [B, Lq, Hq, D]; k_cache, v_cache: device [B, Hkv, Tmax, D];
 * kv_len: device int [B], each in [Lq, Tmax]; o: device float [B, Lq, Hq, D];
 * lse: device float [B, Lq, Hq] or NULL; workspace: device scratch of at least
 * masw_verify_workspace_bytes() bytes, zero-filled by the caller before its
 * first use; every completed call leaves it zero-filled again (the last CTA of
 * each (sequence, kv head) resets its ticket), so a workspace is reused without
 * a memset between calls.  The int at byte offset
 * masw_verify_workspace_bytes() - 16 is a status word: 0, or MASW_ETIMEOUT
 * when a bounded wait inside the kernel gave up (that call's outputs are then
 * undefined, and the workspace must be zero-filled again before reuse).
 * It must not be shared by calls that overlap on the GPU.  scale 0 -> 1/sqrt(D).
 * D must be 128 and (Hq/Hkv) * Lq <= 32. */
int masw_verify_attn(const void* q, const void* k_cache, const void* v_cache,
                     const int* kv_len, int B, int Lq, int Hq, int Hkv, int D,
                     int Tmax, int dtype, float scale, float* o, float* lse,
                     void* workspace, size_t workspace_bytes, masw_stream_t stream);

/* Bytes of workspace masw_verify_attn needs for these sizes on the current device. */
int masw_verify_workspace_bytes(int B, int Lq, int Hq, int Hkv, int D, int Tmax,
                                size_t* bytes);

/* masw_verify_attn without a workspace argument and without allocating
 * anything.  The pages have no counterpart: this is a library convenience.
 * It is for callers that cannot hand over scratch memory or call cudaMalloc:
 * code that only receives input and output pointers (for example a plugin
 * slot in another inference engine), code whose device memory is owned by a
 * framework's own allocator, or a loop that cannot afford the device-wide
 * synchronisation a cudaMalloc may cause.  q, caches, kv_len, o, lse, scale
 * and the size rules are those of masw_verify_attn.  The split partials live
 * in a fixed array inside the library image (4 MiB + 16 KiB, held by every GPU
 * that loads the library until the process exits).
 * status: device int, or NULL.  When given, the call copies its status word
 * there on the stream once the kernel is done: 0, MASW_ETIMEOUT (a bounded wait
 * inside the kernel gave up; that call's O and LSE are undefined) or
 * MASW_EINVAL (the kernel found its shared memory misaligned).  With NULL such
 * a failure goes unreported, because the next call clears the word.
 * Limit: B * Hkv <= 4096 (EINVAL beyond, with a message).  Each call looks up
 * the array's device address with cudaGetSymbolAddress (no allocation); the
 * first call on a device also loads the library's device code there, so make
 * that first call before any stream capture on that device.  Every call reuses
 * the same array (tickets and status are cleared on the stream at the start of
 * each call), so calls that overlap on the GPU -- other streams, other host
 * threads -- race and must be serialised by the caller. */
int masw_verify_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                             const int* kv_len, int B, int Lq, int Hq, int Hkv, int D,
                             int Tmax, int dtype, float scale, float* o, float* lse,
                             int* status, masw_stream_t stream);

/* ---- speculative acceptance ------------------------------------------------------ */

/* Greedy acceptance of a speculative block ([EN] §2.2 and §3.3 Algorithm 2;
 * the pages' experiments decode greedily, temperature 0).  For each sequence b:
 * tokens[b][j] = argmax over v of logits[b][j][v] for j = 0..L (ties go to the
 * smallest id; NaN entries are skipped; +inf and -inf count as values; a row
 * whose entries are all NaN has no greedy token and gets -1); L_acc = the first
 * j < L with draft[b][j] != tokens[b][j], or L when all drafts match (drafts
 * are ids >= 0, so a -1 row rejects its draft); n_emit[b] = L_acc + 1, and the
 * emitted tokens are tokens[b][0 .. L_acc] (accepted drafts, then the target's
 * correction or bonus token; that last token is -1 when its row was all NaN,
 * which the caller must treat as "no token").
 * logits: device [B, L+1, V] (dtype MASW_BF16 or MASW_F32); draft: device int
 * [B, L]; tokens: device int [B, L+1]; n_emit: device int [B]; workspace:
 * device scratch of masw_greedy_workspace_bytes() bytes (16-byte aligned; zero-filled
 * by the caller before its first use, e.g. with cudaMemset; every completed call
 * leaves it zero-filled again, so it is cleared once per allocation; not shared by
 * overlapping calls). */
int masw_greedy_accept(const void* logits, const int* draft, int B, int L, int V, int dtype,
                       int* tokens, int* n_emit, void* workspace, size_t workspace_bytes,
                       masw_stream_t stream);

/* Bytes of workspace masw_greedy_accept needs for these sizes on the current device. */
int masw_greedy_workspace_bytes(int B, int L, int V, size_t* bytes);

/* Eq. 1 of [EN] §2.2: speedup over autoregressive decoding,
 * (l_acc + 1) / (l_draft * t_draft / t_target + 1), from the mean accepted
 * length and the per-token draft and target latencies.  Host only; returns -1
 * for invalid arguments. */
double masw_eq1_speedup(double l_acc, int l_draft, double t_draft, double t_target);

/* ---- plumbing for set-up, tests and benchmarks --------------------------------- */

/* Set (layer, seq) to the state after t raw tokens whose K/V are k_raw, v_raw
 * ([t, Hkv, D], host or device), with n_slots slots k_slots, v_slots
 * ([n_slots, Hkv, D], host or device) as if materialised at tau_1..tau_n.
 * EINVAL unless n_slots == max(0, (t-S-W)/r).  Synchronous. */
int masw_mem_load(masw_mem_t* mem, int layer, int seq, int t,
                  const void* k_raw, const void* v_raw,
                  const void* k_slots, const void* v_slots, int n_slots);

/* Copy the pool block of (layer, seq) -- K and V, each [Hkv, rows, D] with
 * rows = S + W + R + M_max -- into caller memory (host or device).  Optional
 * slot_pos: host int [M_max] receives the device-recorded 0-based position ids
 * (-1 where no slot was ever written).  Synchronous. */
int masw_mem_export(masw_mem_t* mem, int layer, int seq, void* k_out, void* v_out,
                    int* slot_pos);

/* Counters of (layer, seq): host mirror and device copy.  Synchronous. */
int masw_query(masw_mem_t* mem, int layer, int seq, masw_state_t* out);

/* Wait for the stream, then report any error recorded by a kernel since the
 * last masw_sync (MASW_ETIMEOUT; MASW_EGUARD when a decode kernel found its
 * segment table outside its block and skipped the copies; MASW_ECAPACITY) or
 * by the CUDA runtime (MASW_ECUDA). */
int masw_sync(masw_mem_t* mem, masw_stream_t stream);

/* Failure-detection self-test: launch a kernel whose bounded wait (the helper
 * every TMA/MMA wait of the library uses) waits `polls` polls, in [1, 2^20], on
 * a barrier nothing arrives on, runs out and records MASW_ETIMEOUT; the next
 * masw_sync returns MASW_ETIMEOUT and clears it.  Nothing is in flight when the
 * wait gives up, so the handle and the context stay usable. */
int masw_selftest_timeout(masw_mem_t* mem, int polls, masw_stream_t stream);

/* Host-side index model, exported so it can be checked without a GPU.
 * which: 0 = local-window lo (1-based), 1 = n_local, 2 = slot count m(t),
 * 3 = is_boundary(t), 4 = ring row of token t ((t-S-1) mod (W+R), -1 for a
 * sink token), 5 = working-set size.  Returns -1 for bad arguments. */
int masw_index(int which, int t, int S, int W, int r, int R);

/* Library version, "major.minor.patch". */
const char* masw_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MASW_H */
