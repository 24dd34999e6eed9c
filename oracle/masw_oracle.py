"""CPU oracle for Memory-Augmented Sliding-Window (MASW) draft memory and attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything in this package.  The CUDA library never calls it and shares no code
with it (no kernels, headers, index helpers or constant tables).

What it computes is the plain definition, in float64, written so it can be read
against the pages:

* the working memory of Eq. 4, M_t = M_sink u M_local,t u M_slot,t, kept as the
  ENTIRE raw history plus the list of memory slots, and selected at every call
  by an explicitly materialised boolean mask row over
  ``[raw token 1..t] ++ [slot 1..m]``;
* softmax attention of Eq. 2, softmax(q K^T / sqrt(d)) V, over the masked
  columns, with numpy matrix-vector products as the only library primitive;
* the index bookkeeping (sink, local window, eviction, boundaries, slot position
  ids, which ring row holds which token) by a separate deque simulator that
  replays the appends one token at a time.

Pages cited (titles abbreviated):
  [EN]  "Strong Drafts Need Compact Memories: A Technical Review of
        Memory-Augmented Sliding-Window (MASW) Drafting for Long-Context
        Speculative Decoding" (zhongzhuzhou.org, 2026-09-06)
  [ZH]  "强推理草稿也要瘦身：长上下文投机解码的记忆增强滑窗（MASW）阅读笔记"
        (zhongzhuzhou.org, 2026-09-06), a translation of [EN] with extra notes
  [KO]  "Paper Review: Strong Drafts Need Compact Memories" (romaanj.github.io)

Readings taken where the pages are silent or garbled (each is pinned by a test
in tests/test_oracle_pins.py; none is "parity unpinned"):
  * slot count m(t) = max(0, floor((t - S - W) / r)): one slot for every r raw
    tokens that have fallen outside sink and window ([EN] §3.1, third bullet),
    not the looser floor(t / r) of the same section's closing sentence;
  * boundary tau_m = S + W + m*r (m >= 1): the step at which the (m*r)-th raw
    token has left the window ([EN] §3.2 Algorithm 1);
  * the slot query g_m reads the local window evaluated at t = tau_m, the sink
    and slots 1..m-1, and not itself ([EN] §3.2 Algorithm 1);
  * a draft query at step tau_m is issued before g_m is materialised, so it
    sees m-1 slots; the query at tau_m + 1 sees m (causal order of Algorithm 1: g_m follows raw token tau_m);
  * slot position id = tau_m + 1, the 1-based id of the raw token that follows
    g_m ([EN] §3.2 Algorithm 1);
  * GQA: query head h reads kv head floor(h / G), G = Hq / Hkv;
  * scale = 1 / sqrt(head_dim) unless overridden (Eq. 2 uses d for the head
    dimension; Eq. 3 reuses d for the hidden size);
  * verify: query j (0-based) of an Lq-query block whose last key is token
    kv_len sees keys 1 .. kv_len - Lq + 1 + j ([EN] §3.3 Algorithm 2);
  * rollback by k tokens needs k <= R extra ring rows; slots with tau <= t_new
    are kept ([EN] §3.3 Algorithm 2).
"""

from __future__ import annotations

import collections
import math

import numpy as np

__all__ = [
    "local_window", "n_local", "slot_count", "boundary", "is_boundary",
    "slot_pos_id", "working_set_size", "draft_mask", "slot_write_mask",
    "full_mask", "verify_mask", "attention", "IndexSim", "MaswOracle",
    "verify_attn", "greedy_token", "greedy_accept", "eq1_speedup", "prefill_attn",
]


# --------------------------------------------------------------------------
# Index closed forms, 1-based token ids as on the pages.
# --------------------------------------------------------------------------

def local_window(t: int, S: int, W: int) -> tuple[int, int]:
    """Inclusive 1-based bounds (lo, hi) of M_local,t.

    [EN] §3.1, second bullet under Eq. 4: the exact KV of tokens i with
    max(S+1, t-W+1) <= i <= t.  Empty (hi < lo) while t <= S.
    """
    lo = max(S + 1, t - W + 1)
    return lo, t


def n_local(t: int, S: int, W: int) -> int:
    lo, hi = local_window(t, S, W)
    return max(0, hi - lo + 1)


def slot_count(t: int, S: int, W: int, r: int) -> int:
    """Slots that exist once step t is complete: one per r raw tokens that have
    fallen outside sink and local window ([EN] §3.1, third bullet)."""
    return max(0, (t - S - W) // r)


def boundary(m: int, S: int, W: int, r: int) -> int:
    """tau_m, the raw step after which slot g_m is materialised (m >= 1)."""
    if m < 1:
        raise ValueError("boundaries are numbered from 1")
    return S + W + m * r


def is_boundary(t: int, S: int, W: int, r: int) -> bool:
    return t >= S + W + r and (t - S - W) % r == 0


def slot_pos_id(m: int, S: int, W: int, r: int) -> int:
    """RoPE position id of g_m: that of the raw token right after it
    ([EN] §3.2 Algorithm 1), i.e. tau_m + 1 (1-based)."""
    return boundary(m, S, W, r) + 1


def working_set_size(t: int, S: int, W: int, r: int) -> int:
    """|M_t| after step t: min(S, t) sink + window + slots ([EN] §3.1)."""
    return min(S, t) + n_local(t, S, W) + slot_count(t, S, W, r)


# --------------------------------------------------------------------------
# Explicit mask rows over [raw 1..t] ++ [slot 1..n_slots].
# --------------------------------------------------------------------------

def draft_mask(t: int, n_slots: int, S: int, W: int) -> np.ndarray:
    """Columns a draft query at step t may read: M_sink u M_local,t u every
    slot present at call time ([EN] §3.1 Eq. 4; §3.3 Algorithm 2)."""
    raw = np.zeros(t, dtype=bool)
    raw[:min(S, t)] = True
    lo, hi = local_window(t, S, W)
    if hi >= lo:
        raw[lo - 1:hi] = True
    return np.concatenate([raw, np.ones(n_slots, dtype=bool)])


def slot_write_mask(tau: int, m: int, S: int, W: int,
                    self_attend: bool = False) -> np.ndarray:
    """Columns slot token g_m may read at boundary tau ([EN] §3.2 Algorithm 1,
    the structured mask): M_sink, M_local,tau and M_slot,<m, and no other raw
    token.  Columns cover slots 1..m; slot m (g_m itself) is read
    only when ``self_attend``."""
    raw = np.zeros(tau, dtype=bool)
    raw[:min(S, tau)] = True
    lo, hi = local_window(tau, S, W)
    if hi >= lo:
        raw[lo - 1:hi] = True
    slots = np.zeros(m, dtype=bool)
    slots[:m - 1] = True
    if self_attend:
        slots[m - 1] = True
    return np.concatenate([raw, slots])


def full_mask(t: int) -> np.ndarray:
    """Full-KV decode: every raw token 1..t (Eq. 2 with K_{<=t})."""
    return np.ones(t, dtype=bool)


def verify_mask(kv_len: int, Lq: int) -> np.ndarray:
    """[Lq, kv_len] causal block: the cache holds kv_len tokens of which the last
    Lq are the block; query j sees keys 1..kv_len-Lq+1+j ([EN] §3.3
    Algorithm 2: one parallel target pass over the full cache)."""
    mask = np.zeros((Lq, kv_len), dtype=bool)
    for j in range(Lq):
        mask[j, :kv_len - Lq + 1 + j] = True
    return mask


# --------------------------------------------------------------------------
# Eq. 2 over masked columns.
# --------------------------------------------------------------------------

def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, mask: np.ndarray,
              scale: float) -> tuple[np.ndarray, np.ndarray]:
    """softmax(scale * q K^T) V over the columns where ``mask`` is True.

    q: [Hq, D]; K, V: [N, Hkv, D]; mask: [N] (shared by all heads) or [Hq, N].
    Query head h reads kv head h // (Hq // Hkv).  Returns O [Hq, D] and the
    natural-log normaliser LSE [Hq] = log sum_j exp(scale q.k_j).  An empty
    mask row gives O = 0, LSE = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Hq, D = q.shape
    Hkv = K.shape[1]
    if Hq % Hkv:
        raise ValueError("query heads must be a multiple of kv heads")
    G = Hq // Hkv
    mask = np.asarray(mask, dtype=bool)
    O = np.zeros((Hq, D))
    lse = np.full(Hq, -np.inf)
    for h in range(Hq):
        kv = h // G
        row = mask if mask.ndim == 1 else mask[h]
        if not row.any():
            continue
        s = (K[:, kv, :] @ q[h]) * scale
        s = np.where(row, s, -np.inf)
        mx = s.max()
        w = np.where(row, np.exp(s - mx), 0.0)
        z = w.sum()
        O[h] = (w @ V[:, kv, :]) / z
        lse[h] = mx + math.log(z)
    return O, lse


# --------------------------------------------------------------------------
# Deque simulator: replays appends one token at a time.
# --------------------------------------------------------------------------

class IndexSim:
    """Token bookkeeping of one (layer, sequence) by direct simulation.

    The sink is a list, the local window a ``deque(maxlen=W)`` of token ids, the
    ring an array of W + reserve rows written round-robin in arrival order of
    non-sink tokens.  Evictions are the ids the deque drops.  A boundary is
    declared when the number of tokens that have left the window reaches the
    next multiple of r.  Nothing here uses the closed forms above.
    """

    def __init__(self, S: int, W: int, r: int, reserve: int = 0):
        self.S, self.W, self.r, self.reserve = S, W, r, reserve
        self.t = 0
        self.sink: list[int] = []
        if W < 1 or r < 1 or S < 0 or reserve < 0:
            raise ValueError("need W >= 1, r >= 1, S >= 0, reserve >= 0")
        self.window: collections.deque[int] = collections.deque(maxlen=W)
        self.evicted: list[int] = []
        self.ring = [0] * (W + reserve)   # 0 = row never written
        self.cursor = 0
        self.slots: list[tuple[int, int]] = []   # (tau, pos_id), in chain order
        self.history: list[int] = []

    def append(self) -> int | None:
        """Add the next raw token; returns the id it evicted, if any."""
        self.t += 1
        i = self.t
        self.history.append(i)
        dropped = None
        if len(self.sink) < self.S:
            self.sink.append(i)
            return None
        if len(self.window) == self.W:
            dropped = self.window[0]
        self.window.append(i)
        self.ring[self.cursor] = i
        self.cursor = (self.cursor + 1) % len(self.ring)
        if dropped is not None:
            self.evicted.append(dropped)
        return dropped

    def boundary_due(self) -> bool:
        """True when the count of tokens that have left the window has just
        reached a multiple of r whose slot is the next one in the chain."""
        n = len(self.evicted)
        return n > 0 and n % self.r == 0 and len(self.slots) == n // self.r - 1

    def materialize(self) -> int:
        """Record g_m at the current step; returns its position id (the id of
        the raw token that will follow)."""
        if not self.boundary_due():
            raise RuntimeError("not at a compression boundary")
        pos = self.t + 1
        self.slots.append((self.t, pos))
        return pos

    def visible_raw(self) -> list[int]:
        return list(self.sink) + list(self.window)

    def rollback(self, t_new: int) -> None:
        """Discard raw tokens after t_new and slots made after it, rebuilding
        the window from ring rows; fails if a needed row was overwritten."""
        if t_new > self.t or t_new < 0:
            raise ValueError("bad rollback target")
        keep_hist = self.history[:t_new]
        self.sink = [i for i in keep_hist[:self.S]]
        nonsink = keep_hist[self.S:]
        want = nonsink[-self.W:]
        for i in want:
            if i not in self.ring:
                raise RuntimeError("rollback deeper than the ring reserve")
        self.window = collections.deque(want, maxlen=self.W)
        self.evicted = nonsink[:len(nonsink) - len(want)]
        self.slots = [(tau, pos) for (tau, pos) in self.slots if tau <= t_new]
        self.cursor = len(nonsink) % len(self.ring)
        self.history = keep_hist
        self.t = t_new

    def ring_map(self) -> list[int]:
        """Token id held by each ring row (0 = never written)."""
        return list(self.ring)


# --------------------------------------------------------------------------
# The oracle memory: full raw history + slot list, all float64.
# --------------------------------------------------------------------------

class MaswOracle:
    """Plain-definition model of the draft memory for `layers` x `batch`.

    K/V inputs are widened exactly to float64; every call rebuilds its mask row
    and evaluates Eq. 2 over the whole history with that mask.
    """

    def __init__(self, S: int, W: int, r: int, n_kv_heads: int, head_dim: int,
                 layers: int, batch: int = 1, scale: float | None = None,
                 slot_self_attend: bool = False, reserve: int = 0):
        self.S, self.W, self.r = S, W, r
        self.Hkv, self.D = n_kv_heads, head_dim
        self.layers, self.batch = layers, batch
        self.scale = (1.0 / math.sqrt(head_dim)) if not scale else float(scale)
        self.self_attend = slot_self_attend
        self.reserve = reserve
        empty = np.zeros((0, n_kv_heads, head_dim))
        self.raw_k = [[empty.copy() for _ in range(batch)] for _ in range(layers)]
        self.raw_v = [[empty.copy() for _ in range(batch)] for _ in range(layers)]
        self.slot_k = [[empty.copy() for _ in range(batch)] for _ in range(layers)]
        self.slot_v = [[empty.copy() for _ in range(batch)] for _ in range(layers)]
        self.slot_tau = [[[] for _ in range(batch)] for _ in range(layers)]
        self.sim = [[IndexSim(S, W, r, reserve) for _ in range(batch)] for _ in range(layers)]

    # -- state ------------------------------------------------------------
    def t(self, layer: int, seq: int) -> int:
        return self.raw_k[layer][seq].shape[0]

    def m(self, layer: int, seq: int) -> int:
        return self.slot_k[layer][seq].shape[0]

    def load(self, layer: int, seq: int, k_raw, v_raw, k_slots=None, v_slots=None):
        """Set a sequence's state after t raw tokens with the given slot K/V,
        as if slots had been materialised at every boundary tau_1..tau_n."""
        k_raw = np.asarray(k_raw, dtype=np.float64)
        v_raw = np.asarray(v_raw, dtype=np.float64)
        t = k_raw.shape[0]
        n = 0 if k_slots is None else np.asarray(k_slots).shape[0]
        if n != slot_count(t, self.S, self.W, self.r):
            raise ValueError("slot count must equal m(t)")
        self.raw_k[layer][seq] = k_raw.copy()
        self.raw_v[layer][seq] = v_raw.copy()
        shape = (0, self.Hkv, self.D)
        self.slot_k[layer][seq] = np.asarray(k_slots, dtype=np.float64).copy() if n else np.zeros(shape)
        self.slot_v[layer][seq] = np.asarray(v_slots, dtype=np.float64).copy() if n else np.zeros(shape)
        self.slot_tau[layer][seq] = [boundary(j, self.S, self.W, self.r) for j in range(1, n + 1)]
        sim = IndexSim(self.S, self.W, self.r, self.reserve)
        for _ in range(t):
            sim.append()
            if sim.boundary_due() and len(sim.slots) < n:
                sim.materialize()
        self.sim[layer][seq] = sim

    def append(self, layer: int, k, v, active=None):
        """Append one raw token per active sequence ([EN] §3.3 Algorithm 2;
        eviction is implicit in the window bounds)."""
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        for b in range(self.batch):
            if active is not None and not active[b]:
                continue
            self.raw_k[layer][b] = np.concatenate([self.raw_k[layer][b], k[b][None]], 0)
            self.raw_v[layer][b] = np.concatenate([self.raw_v[layer][b], v[b][None]], 0)
            self.sim[layer][b].append()

    # -- attention calls --------------------------------------------------
    def _columns(self, layer: int, seq: int):
        Kc = np.concatenate([self.raw_k[layer][seq], self.slot_k[layer][seq]], 0)
        Vc = np.concatenate([self.raw_v[layer][seq], self.slot_v[layer][seq]], 0)
        return Kc, Vc

    def draft_attn(self, layer: int, q):
        """Draft decode attention over M_t for every sequence: q [B, Hq, D]."""
        q = np.asarray(q, dtype=np.float64)
        B, Hq, D = q.shape
        O = np.zeros((B, Hq, D))
        L = np.full((B, Hq), -np.inf)
        for b in range(B):
            t, m = self.t(layer, b), self.m(layer, b)
            Kc, Vc = self._columns(layer, b)
            mask = draft_mask(t, m, self.S, self.W)
            O[b], L[b] = attention(q[b], Kc, Vc, mask, self.scale)
        return O, L

    def materialize_slot(self, layer: int, seq_ids, q_g, k_g, v_g):
        """Slot write at boundary tau_m for the listed sequences ([EN] §3.2
        Algorithm 1): g_m attends under the structured mask, then
        its K/V are appended to the chain.  Returns O_g [n, Hq, D] and LSE."""
        q_g = np.asarray(q_g, dtype=np.float64)
        k_g = np.asarray(k_g, dtype=np.float64)
        v_g = np.asarray(v_g, dtype=np.float64)
        n, Hq, D = q_g.shape
        O = np.zeros((n, Hq, D))
        L = np.full((n, Hq), -np.inf)
        for i, b in enumerate(seq_ids):
            tau = self.t(layer, b)
            if not is_boundary(tau, self.S, self.W, self.r):
                raise RuntimeError(f"sequence {b} is not at a compression boundary (t={tau})")
            m = slot_count(tau, self.S, self.W, self.r)
            if self.m(layer, b) != m - 1:
                raise RuntimeError("slot for this boundary already materialised")
            self.slot_k[layer][b] = np.concatenate([self.slot_k[layer][b], k_g[i][None]], 0)
            self.slot_v[layer][b] = np.concatenate([self.slot_v[layer][b], v_g[i][None]], 0)
            self.slot_tau[layer][b].append(tau)
            self.sim[layer][b].materialize()
            Kc, Vc = self._columns(layer, b)
            mask = slot_write_mask(tau, m, self.S, self.W, self.self_attend)
            O[i], L[i] = attention(q_g[i], Kc, Vc, mask, self.scale)
        return O, L

    def full_attn(self, layer: int, q):
        """Full-KV decode over all t raw tokens (the uncompressed contrast)."""
        q = np.asarray(q, dtype=np.float64)
        B, Hq, D = q.shape
        O = np.zeros((B, Hq, D))
        L = np.full((B, Hq), -np.inf)
        for b in range(B):
            t = self.t(layer, b)
            O[b], L[b] = attention(q[b], self.raw_k[layer][b], self.raw_v[layer][b],
                                   full_mask(t), self.scale)
        return O, L

    def rollback(self, seq_ids, t_new):
        """Discard raw tokens after t_new[i] and slots with tau > t_new[i] in
        every layer ([EN] §3.3 Algorithm 2)."""
        for i, b in enumerate(seq_ids):
            tn = int(t_new[i])
            for l in range(self.layers):
                t = self.t(l, b)
                if tn > t or t - tn > self.reserve:
                    raise RuntimeError("rollback deeper than the ring reserve")
                self.raw_k[l][b] = self.raw_k[l][b][:tn]
                self.raw_v[l][b] = self.raw_v[l][b][:tn]
                keep = [j for j, tau in enumerate(self.slot_tau[l][b]) if tau <= tn]
                self.slot_k[l][b] = self.slot_k[l][b][:len(keep)]
                self.slot_v[l][b] = self.slot_v[l][b][:len(keep)]
                self.slot_tau[l][b] = self.slot_tau[l][b][:len(keep)]
                self.sim[l][b].rollback(tn)


def verify_attn(q, k_cache, v_cache, kv_len, scale: float | None = None):
    """Target verify attention over an uncompressed cache ([EN] §3.3
    Algorithm 2).  q [B, Lq, Hq, D]; k/v_cache [B, Hkv, Tmax, D];
    kv_len [B] counts the block's own Lq tokens.  Returns O [B, Lq, Hq, D] and
    LSE [B, Lq, Hq]."""
    q = np.asarray(q, dtype=np.float64)
    B, Lq, Hq, D = q.shape
    scale = (1.0 / math.sqrt(D)) if not scale else float(scale)
    O = np.zeros((B, Lq, Hq, D))
    L = np.full((B, Lq, Hq), -np.inf)
    for b in range(B):
        n = int(kv_len[b])
        K = np.asarray(k_cache[b][:, :n, :], dtype=np.float64).transpose(1, 0, 2)
        V = np.asarray(v_cache[b][:, :n, :], dtype=np.float64).transpose(1, 0, 2)
        mask = verify_mask(n, Lq)
        for j in range(Lq):
            O[b, j], L[b, j] = attention(q[b, j], K, V, mask[j], scale)
    return O, L


# --------------------------------------------------------------------------
# Speculative acceptance and the speedup model.
# --------------------------------------------------------------------------

def greedy_token(row) -> int:
    """The target's greedy token for one logits row: the id of the largest
    value, the smallest id among ties, NaN entries ignored (+inf and -inf are
    values like any other).  A row with no value but NaN has no greedy token:
    -1.  (The pages decode at temperature 0 and say nothing of NaN logits;
    skipping them is this library's reading.)"""
    row = np.asarray(row, dtype=np.float64)
    ids = np.flatnonzero(~np.isnan(row))
    if ids.size == 0:
        return -1
    return int(ids[np.argmax(row[ids])])   # np.argmax: first position of the maximum


def greedy_accept(logits, draft):
    """Greedy speculative acceptance ([EN] §2.2, §3.3 Algorithm 2; the
    experiments use temperature 0).  logits [B, L+1, V], draft [B, L] ->
    tokens [B, L+1] (greedy_token of each row: argmax, first index among ties,
    NaN skipped, -1 for an all-NaN row) and n_emit [B] = L_acc + 1, L_acc =
    number of leading drafts equal to the target's tokens (a draft never equals
    -1, so an all-NaN row rejects its draft)."""
    logits = np.asarray(logits, dtype=np.float64)
    draft = np.asarray(draft)
    B, L1, V = logits.shape
    L = L1 - 1
    tokens = np.zeros((B, L1), dtype=np.int64)
    n_emit = np.zeros(B, dtype=np.int64)
    for b in range(B):
        for j in range(L1):
            tokens[b, j] = greedy_token(logits[b, j])
        l_acc = 0
        while l_acc < L and draft[b, l_acc] == tokens[b, l_acc]:
            l_acc += 1
        n_emit[b] = l_acc + 1
    return tokens, n_emit


def eq1_speedup(l_acc: float, l_draft: int, t_draft: float, t_target: float) -> float:
    """Eq. 1 of [EN] §2.2: (L_acc + 1) / (L_draft * t_d / t_t + 1)."""
    return (l_acc + 1.0) / (l_draft * (t_draft / t_target) + 1.0)


# --------------------------------------------------------------------------
# Draft prefill under the structured write mask.
# --------------------------------------------------------------------------

def prefill_row_mask(kind, idx, T, S, W, r, self_attend=False):
    """Mask row of one prefill query over the columns [raw 1..T] ++ [slot 1..M]
    ([EN] §3.3 Algorithm 2 with the structured mask of §3.2 Algorithm 1).
    kind "raw": raw token idx (1-based) reads the sink, its local window and
    the slots with tau_m < idx; kind "slot": slot g_idx reads what the slot
    write at tau_idx reads (sink, window at tau_idx, slots 1..idx-1)."""
    M = slot_count(T, S, W, r)
    mask = np.zeros(T + M, dtype=bool)
    if kind == "raw":
        i = idx
        mask[:i] = draft_mask(i, 0, S, W)            # raw columns 1..i
        mask[T:T + slot_count(i - 1, S, W, r)] = True   # slots with tau_m <= i-1
    else:
        m = idx
        tau = boundary(m, S, W, r)
        row = slot_write_mask(tau, m, S, W, self_attend)
        mask[:tau] = row[:tau]
        mask[T:T + m] = row[tau:]
    return mask


def prefill_attn(S, W, r, q_raw, k_raw, v_raw, q_slot, k_slot, v_slot, scale=None, self_attend=False,
                 raw_rows=None, slot_rows=None):
    """One layer of the draft prefill over T raw tokens with the M = m(T) slot
    tokens interleaved ([EN] §3.3 Algorithm 2, with the structured mask of
    §3.2 Algorithm 1): raw token i reads the sink, its local window and
    the slots materialised before it (tau_m < i); slot g_m reads the sink, the
    window at tau_m and slots 1..m-1.  Columns are [raw 1..T] ++ [slot 1..M].
    q_raw [T, Hq, D], k_raw/v_raw [T, Hkv, D], q_slot [M, Hq, D],
    k_slot/v_slot [M, Hkv, D].  Returns O_raw [T, Hq, D], LSE_raw [T, Hq],
    O_slot [M, Hq, D], LSE_slot [M, Hq].  raw_rows / slot_rows (1-based lists)
    restrict the evaluation to those rows (the others stay 0 / -inf)."""
    q_raw = np.asarray(q_raw, dtype=np.float64)
    k_raw = np.asarray(k_raw, dtype=np.float64)
    v_raw = np.asarray(v_raw, dtype=np.float64)
    T, Hq, D = q_raw.shape
    M = slot_count(T, S, W, r)
    q_slot = np.asarray(q_slot, dtype=np.float64).reshape(M, Hq, D)
    k_slot = np.asarray(k_slot, dtype=np.float64).reshape(M, k_raw.shape[1], D)
    v_slot = np.asarray(v_slot, dtype=np.float64).reshape(M, k_raw.shape[1], D)
    scale = (1.0 / math.sqrt(D)) if not scale else float(scale)
    K = np.concatenate([k_raw, k_slot], 0)
    V = np.concatenate([v_raw, v_slot], 0)
    o_raw = np.zeros((T, Hq, D))
    l_raw = np.full((T, Hq), -np.inf)
    for i in (range(1, T + 1) if raw_rows is None else raw_rows):
        mask = prefill_row_mask("raw", i, T, S, W, r)
        o_raw[i - 1], l_raw[i - 1] = attention(q_raw[i - 1], K, V, mask, scale)
    o_slot = np.zeros((M, Hq, D))
    l_slot = np.full((M, Hq), -np.inf)
    for m in (range(1, M + 1) if slot_rows is None else slot_rows):
        mask = prefill_row_mask("slot", m, T, S, W, r, self_attend)
        o_slot[m - 1], l_slot[m - 1] = attention(q_slot[m - 1], K, V, mask, scale)
    return o_raw, l_raw, o_slot, l_slot
