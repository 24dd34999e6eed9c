"""Thin ctypes binding of libmasw (include/masw.h), same names as the C calls.

Argument marshalling only: torch tensors contribute device pointers, the
current CUDA stream is passed as the stream, and a non-zero status becomes a
MaswError carrying masw_last_error().  Every step of the computation runs in
the library's CUDA kernels; there is no fallback if the library is missing.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmasw.so")

MASW_OK, MASW_EINVAL, MASW_ENOMEM, MASW_ECAPACITY, MASW_ESTATE, MASW_ECUDA, MASW_ETIMEOUT = 0, -1, -2, -3, -4, -5, -6
MASW_EGUARD = -7
MASW_F32, MASW_BF16 = 0, 1
MASW_MAX_BATCH, MASW_MAX_GROUP = 512, 8

# every symbol include/masw.h declares
EXPORTS = [
    "masw_mem_create", "masw_mem_destroy", "masw_last_error", "masw_append_kv",
    "masw_materialize_slot", "masw_rollback", "masw_draft_attn", "masw_full_attn",
    "masw_draft_step", "masw_full_step", "masw_draft_step_slot",
    "masw_verify_attn", "masw_verify_workspace_bytes", "masw_verify_attn_noalloc", "masw_mem_load", "masw_mem_export",
    "masw_query", "masw_sync", "masw_index", "masw_version", "masw_check_guards",
    "masw_greedy_accept", "masw_greedy_workspace_bytes", "masw_eq1_speedup", "masw_prefill",
    "masw_selftest_timeout",
]


class MaswError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libmasw status {code}: {msg}")
        self.code = code


class masw_opts_t(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("dtype", ctypes.c_int), ("max_seq_len", ctypes.c_int),
                ("softmax_scale", ctypes.c_float), ("slot_self_attend", ctypes.c_int),
                ("full_kv", ctypes.c_int), ("rollback_reserve", ctypes.c_int)]


class masw_state_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("t", "n_sink", "n_local", "m", "dev_t", "dev_m",
                                            "ring_rows", "rows", "slot_capacity")]


_lib = None


def load() -> ctypes.CDLL:
    """Load the in-tree libmasw.so; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmasw.so not built at {LIB_PATH}; run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    IP = ctypes.POINTER(ctypes.c_int)
    sig = {
        "masw_mem_create": [I, I, I, I, I, I, ctypes.POINTER(masw_opts_t), ctypes.POINTER(P)],
        "masw_mem_destroy": [P],
        "masw_check_guards": [P],
        "masw_append_kv": [P, I, P, P, P, P],
        "masw_materialize_slot": [P, I, IP, I, P, P, P, P, P, I, P],
        "masw_rollback": [P, IP, IP, I, P],
        "masw_draft_attn": [P, I, P, I, P, P, P],
        "masw_full_attn": [P, I, P, I, P, P, P],
        "masw_draft_step": [P, I, P, P, P, P, I, P, P, P],
        "masw_full_step": [P, I, P, P, P, P, I, P, P, P],
        "masw_draft_step_slot": [P, I, P, P, P, P, I, P, P, IP, I, P, P, P, P, P, P],
        "masw_prefill": [P, I, I, I, P, P, P, P, P, P, I, P, P, P, P, P],
        "masw_selftest_timeout": [P, I, P],
        "masw_verify_attn": [P, P, P, P, I, I, I, I, I, I, I, F, P, P, P, Z, P],
        "masw_verify_workspace_bytes": [I, I, I, I, I, I, ctypes.POINTER(Z)],
        "masw_verify_attn_noalloc": [P, P, P, P, I, I, I, I, I, I, I, F, P, P, P, P],
        "masw_mem_load": [P, I, I, I, P, P, P, P, I],
        "masw_mem_export": [P, I, I, P, P, IP],
        "masw_query": [P, I, I, ctypes.POINTER(masw_state_t)],
        "masw_sync": [P, P],
        "masw_index": [I, I, I, I, I, I],
        "masw_greedy_accept": [P, P, I, I, I, I, P, P, P, Z, P],
        "masw_greedy_workspace_bytes": [I, I, I, ctypes.POINTER(Z)],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = I
    lib.masw_last_error.argtypes = [P]
    lib.masw_last_error.restype = ctypes.c_char_p
    lib.masw_eq1_speedup.argtypes = [ctypes.c_double, I, ctypes.c_double, ctypes.c_double]
    lib.masw_eq1_speedup.restype = ctypes.c_double
    lib.masw_version.argtypes = []
    lib.masw_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(rc: int, handle=None):
    if rc != MASW_OK:
        msg = load().masw_last_error(handle)
        raise MaswError(rc, msg.decode() if msg else "")


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is not None:
        return stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _int_array(xs):
    xs = [int(x) for x in xs]
    return (ctypes.c_int * len(xs))(*xs), len(xs)


# ---------------------------------------------------------------- lifetime --

def masw_mem_create(S, W, r, n_kv_heads, head_dim, layers, batch=1, dtype=MASW_BF16, max_seq_len=32768,
                    softmax_scale=0.0, slot_self_attend=False, full_kv=False, rollback_reserve=0):
    lib = load()
    opts = masw_opts_t(batch, dtype, max_seq_len, softmax_scale, int(slot_self_attend), int(full_kv),
                       rollback_reserve)
    h = ctypes.c_void_p()
    _check(lib.masw_mem_create(S, W, r, n_kv_heads, head_dim, layers, ctypes.byref(opts), ctypes.byref(h)))
    return h.value


def masw_mem_destroy(handle):
    _check(load().masw_mem_destroy(handle))


def masw_check_guards(handle):
    """Raise MaswError(MASW_EGUARD) if a guard band around one of the handle's
    device buffers was overwritten (synchronises the device)."""
    _check(load().masw_check_guards(handle), handle)


def masw_last_error(handle=None) -> str:
    msg = load().masw_last_error(handle)
    return msg.decode() if msg else ""


# ------------------------------------------------------------- maintenance --

def masw_append_kv(handle, layer, k, v, active=None, stream=None):
    act = None
    if active is not None:
        act = (ctypes.c_uint8 * len(active))(*[1 if a else 0 for a in active])
    _check(load().masw_append_kv(handle, layer, _ptr(k), _ptr(v),
                                 ctypes.cast(act, ctypes.c_void_p) if act is not None else None,
                                 _stream(stream)), handle)


def masw_materialize_slot(handle, layer, seq_ids, q_g, k_g, v_g, o_g, lse_g=None, stream=None):
    ids, n = _int_array(seq_ids)
    _check(load().masw_materialize_slot(handle, layer, ids, n, _ptr(q_g), _ptr(k_g), _ptr(v_g), _ptr(o_g),
                                        _ptr(lse_g), q_g.shape[1], _stream(stream)), handle)


def masw_rollback(handle, seq_ids, t_new, stream=None):
    ids, n = _int_array(seq_ids)
    tn, n2 = _int_array(t_new)
    if n != n2:
        raise ValueError("seq_ids and t_new differ in length")
    _check(load().masw_rollback(handle, ids, tn, n, _stream(stream)), handle)


# --------------------------------------------------------------- attention --

def masw_draft_attn(handle, layer, q, o, lse=None, stream=None):
    _check(load().masw_draft_attn(handle, layer, _ptr(q), q.shape[1], _ptr(o), _ptr(lse), _stream(stream)), handle)


def masw_full_attn(handle, layer, q, o, lse=None, stream=None):
    _check(load().masw_full_attn(handle, layer, _ptr(q), q.shape[1], _ptr(o), _ptr(lse), _stream(stream)), handle)


def _active(active):
    if active is None:
        return None, None
    arr = (ctypes.c_uint8 * len(active))(*[1 if a else 0 for a in active])
    return arr, ctypes.cast(arr, ctypes.c_void_p)


def masw_draft_step(handle, layer, q, k, v, o, lse=None, active=None, stream=None):
    keep, act = _active(active)
    _check(load().masw_draft_step(handle, layer, _ptr(q), _ptr(k), _ptr(v), act, q.shape[1], _ptr(o), _ptr(lse),
                                  _stream(stream)), handle)


def masw_full_step(handle, layer, q, k, v, o, lse=None, active=None, stream=None):
    keep, act = _active(active)
    _check(load().masw_full_step(handle, layer, _ptr(q), _ptr(k), _ptr(v), act, q.shape[1], _ptr(o), _ptr(lse),
                                 _stream(stream)), handle)


def masw_draft_step_slot(handle, layer, q, k, v, o, seq_ids, q_g, k_g, v_g, o_g, lse=None, lse_g=None,
                         active=None, stream=None):
    keep, act = _active(active)
    ids, n = _int_array(seq_ids)
    _check(load().masw_draft_step_slot(handle, layer, _ptr(q), _ptr(k), _ptr(v), act, q.shape[1], _ptr(o), _ptr(lse),
                                       ids, n, _ptr(q_g), _ptr(k_g), _ptr(v_g), _ptr(o_g), _ptr(lse_g),
                                       _stream(stream)), handle)


def masw_verify_workspace_bytes(B, Lq, Hq, Hkv, D, Tmax) -> int:
    out = ctypes.c_size_t()
    _check(load().masw_verify_workspace_bytes(B, Lq, Hq, Hkv, D, Tmax, ctypes.byref(out)))
    return out.value


def masw_verify_attn(q, k_cache, v_cache, kv_len, o, lse=None, workspace=None, scale=0.0, stream=None):
    """q [B, Lq, Hq, D] bf16, caches [B, Hkv, Tmax, D] bf16, kv_len [B] int32 -> o [B, Lq, Hq, D] fp32.
    A caller's workspace (uint8, at least masw_verify_workspace_bytes) must be zero-filled before its first
    use; every completed call leaves it zero-filled.  Without one, a zero-filled workspace is allocated."""
    B, Lq, Hq, D = q.shape
    Hkv, Tmax = k_cache.shape[1], k_cache.shape[2]
    need = masw_verify_workspace_bytes(B, Lq, Hq, Hkv, D, Tmax)
    if workspace is None:
        import torch
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)   # zero-filled before first use
    _check(load().masw_verify_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), B, Lq, Hq, Hkv, D, Tmax,
                                   MASW_BF16, scale, _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel(),
                                   _stream(stream)))


def masw_verify_attn_noalloc(q, k_cache, v_cache, kv_len, o, lse=None, scale=0.0, status=None, stream=None):
    """masw_verify_attn for callers that cannot allocate: no workspace, the
    library's own fixed device array holds the split partials.  status: an
    optional device int32 tensor that receives the call's status word."""
    B, Lq, Hq, D = q.shape
    Hkv, Tmax = k_cache.shape[1], k_cache.shape[2]
    _check(load().masw_verify_attn_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), B, Lq, Hq, Hkv, D,
                                           Tmax, MASW_BF16, scale, _ptr(o), _ptr(lse), _ptr(status),
                                           _stream(stream)))


def masw_greedy_accept(logits, draft, tokens, n_emit, workspace=None, stream=None):
    """logits [B, L+1, V] (bf16 or fp32), draft [B, L] int32 -> tokens [B, L+1], n_emit [B] (int32)."""
    import torch
    B, L1, V = logits.shape
    L = L1 - 1
    need = ctypes.c_size_t()
    _check(load().masw_greedy_workspace_bytes(B, L, V, ctypes.byref(need)))
    if workspace is None:   # zero-filled once; every call leaves it zero-filled
        workspace = torch.zeros(need.value, dtype=torch.uint8, device=logits.device)
    dt = MASW_BF16 if logits.dtype == torch.bfloat16 else MASW_F32
    _check(load().masw_greedy_accept(_ptr(logits), _ptr(draft), B, L, V, dt, _ptr(tokens), _ptr(n_emit),
                                     _ptr(workspace), workspace.numel(), _stream(stream)))


def masw_greedy_workspace_bytes(B, L, V) -> int:
    out = ctypes.c_size_t()
    _check(load().masw_greedy_workspace_bytes(B, L, V, ctypes.byref(out)))
    return out.value


def masw_eq1_speedup(l_acc, l_draft, t_draft, t_target) -> float:
    return load().masw_eq1_speedup(l_acc, l_draft, t_draft, t_target)


# ---------------------------------------------------------------- plumbing --

def masw_prefill(handle, layer, seq, q_raw, k_raw, v_raw, q_slot, k_slot, v_slot, o_raw, lse_raw=None,
                 o_slot=None, lse_slot=None, stream=None):
    """Prefill one (layer, seq): q_raw [T, Hq, D], k_raw/v_raw [T, Hkv, D], the slot
    tokens' q/k/v [M, ...] (None when M = 0), outputs fp32 o [.., Hq, D], lse [.., Hq]."""
    T, Hq = q_raw.shape[0], q_raw.shape[1]
    _check(load().masw_prefill(handle, layer, seq, T, _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(q_slot),
                               _ptr(k_slot), _ptr(v_slot), Hq, _ptr(o_raw), _ptr(lse_raw), _ptr(o_slot),
                               _ptr(lse_slot), _stream(stream)), handle)


def masw_selftest_timeout(handle, polls=1000, stream=None):
    """Launch the failure-detection self-test (a bounded wait that runs out);
    the next masw_sync raises MaswError with MASW_ETIMEOUT."""
    _check(load().masw_selftest_timeout(handle, polls, _stream(stream)), handle)


def masw_mem_load(handle, layer, seq, k_raw, v_raw, k_slots=None, v_slots=None):
    """k_raw, v_raw: [t, Hkv, D] torch tensors (CPU or CUDA), contiguous."""
    t = k_raw.shape[0]
    n = 0 if k_slots is None else k_slots.shape[0]
    for x in (k_raw, v_raw, k_slots, v_slots):
        if x is not None and not x.is_contiguous():
            raise ValueError("load inputs must be contiguous")
    _check(load().masw_mem_load(handle, layer, seq, t, _ptr(k_raw), _ptr(v_raw), _ptr(k_slots), _ptr(v_slots), n),
           handle)


def masw_mem_export(handle, layer, seq, k_out, v_out, slot_capacity=0):
    pos = (ctypes.c_int * max(1, slot_capacity))()
    _check(load().masw_mem_export(handle, layer, seq, _ptr(k_out), _ptr(v_out), pos), handle)
    return list(pos)[:slot_capacity]


def masw_query(handle, layer, seq) -> dict:
    st = masw_state_t()
    _check(load().masw_query(handle, layer, seq, ctypes.byref(st)), handle)
    return {name: getattr(st, name) for name, _ in masw_state_t._fields_}


def masw_sync(handle, stream=None):
    _check(load().masw_sync(handle, _stream(stream)), handle)


def masw_index(which, t, S, W, r, R=0) -> int:
    return load().masw_index(which, t, S, W, r, R)


def masw_version() -> str:
    return load().masw_version().decode()
