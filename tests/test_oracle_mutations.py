"""Plant plausible mistakes in the CPU oracle and check that the pins catch each.

Every mutation is applied to the oracle module on the CPU (monkeypatch) and
undone after the test; nothing here touches the CUDA library.
"""
import math

import numpy as np
import pytest

import oracle.masw_oracle as o
import oracle_pins as P


def _fails_some_pin():
    for pin in P.ALL_PINS:
        try:
            pin(o)
        except Exception:
            return pin.__name__
    return None


def _attention_variant(kv_of=None, use_scale=True, v_from_k=False, drop_max_in_lse=False):
    def attention(q, K, V, mask, scale):
        q = np.asarray(q, dtype=np.float64)
        K = np.asarray(K, dtype=np.float64)
        V = np.asarray(V, dtype=np.float64)
        Hq, D = q.shape
        Hkv = K.shape[1]
        G = Hq // Hkv
        mask = np.asarray(mask, dtype=bool)
        O = np.zeros((Hq, D))
        lse = np.full(Hq, -np.inf)
        for h in range(Hq):
            kv = kv_of(h, G, Hkv) if kv_of else h // G
            row = mask if mask.ndim == 1 else mask[h]
            if not row.any():
                continue
            s = (K[:, kv, :] @ q[h]) * (scale if use_scale else 1.0)
            s = np.where(row, s, -np.inf)
            mx = s.max()
            w = np.where(row, np.exp(s - mx), 0.0)
            z = w.sum()
            O[h] = (w @ (K if v_from_k else V)[:, kv, :]) / z
            lse[h] = (0.0 if drop_max_in_lse else mx) + math.log(z)
        return O, lse
    return attention


MUTATIONS = {
    "window_off_by_one": ("local_window", lambda t, S, W: (max(S + 1, t - W + 2), t)),
    "window_too_wide": ("local_window", lambda t, S, W: (max(S + 1, t - W), t)),
    "slot_count_floor_t_over_r": ("slot_count", lambda t, S, W, r: t // r),
    "slot_count_without_window": ("slot_count", lambda t, S, W, r: max(0, (t - S) // r)),
    "boundary_without_offset": ("is_boundary", lambda t, S, W, r: t >= r and t % r == 0),
    "slot_pos_id_same_as_tau": ("slot_pos_id", lambda m, S, W, r: S + W + m * r),
    "gqa_modulo_mapping": ("attention", _attention_variant(kv_of=lambda h, G, Hkv: h % Hkv)),
    "scale_missing": ("attention", _attention_variant(use_scale=False)),
    "v_replaced_by_k": ("attention", _attention_variant(v_from_k=True)),
    "lse_without_max": ("attention", _attention_variant(drop_max_in_lse=True)),
    "slot_reads_itself": ("slot_write_mask",
                          lambda tau, m, S, W, self_attend=False: _slot_mask_self(tau, m, S, W)),
    "verify_causal_shift": ("verify_mask", lambda kv_len, Lq: _verify_shift(kv_len, Lq)),
    "sink_dropped": ("draft_mask", lambda t, n_slots, S, W: _draft_no_sink(t, n_slots, S, W)),
    "accept_one_past_mismatch": ("greedy_accept", lambda logits, draft: _accept_off_by_one(logits, draft)),
    "greedy_argmax_returns_first_nan": ("greedy_token", lambda row: int(np.argmax(np.asarray(row, np.float64)))),
    "greedy_nan_as_minus_inf": ("greedy_token",
                                lambda row: int(np.argmax(np.nan_to_num(np.asarray(row, np.float64), nan=-np.inf)))),
    "prefill_raw_sees_slot_of_its_own_boundary": ("prefill_attn", lambda *a, **k: _prefill_slot_too_early(*a, **k)),
    "eq1_without_verify_cost": ("eq1_speedup", lambda l_acc, l_draft, t_d, t_t: (l_acc + 1.0) / (l_draft * t_d / t_t)
                                if t_d else l_acc + 1.0),
}

_orig_accept = o.greedy_accept


def _accept_off_by_one(logits, draft):
    tokens, n = _orig_accept(logits, draft)
    L = np.asarray(draft).shape[1]
    return tokens, np.minimum(n + 1, L + 1)

def _prefill_slot_too_early(S, W, r, q_raw, k_raw, v_raw, q_slot, k_slot, v_slot, scale=None, self_attend=False):
    """Raw token tau_m also reads slot m (the slot written at its own step)."""
    q_raw, k_raw, v_raw = (np.asarray(x, np.float64) for x in (q_raw, k_raw, v_raw))
    T, Hq, D = q_raw.shape
    M = o.slot_count(T, S, W, r)
    k_slot = np.asarray(k_slot, np.float64).reshape(M, k_raw.shape[1], D)
    v_slot = np.asarray(v_slot, np.float64).reshape(M, k_raw.shape[1], D)
    out = list(_orig_prefill(S, W, r, q_raw, k_raw, v_raw, q_slot, k_slot, v_slot, scale, self_attend))
    K, V = np.concatenate([k_raw, k_slot]), np.concatenate([v_raw, v_slot])
    sc = (1.0 / math.sqrt(D)) if not scale else float(scale)
    for i in range(1, T + 1):
        mask = np.zeros(T + M, dtype=bool)
        mask[:i] = o.draft_mask(i, 0, S, W)
        mask[T:T + o.slot_count(i, S, W, r)] = True
        out[0][i - 1], out[1][i - 1] = o.attention(q_raw[i - 1], K, V, mask, sc)
    return tuple(out)


_orig_prefill = o.prefill_attn
_orig = {name: getattr(o, name) for name in
         ("local_window", "slot_write_mask", "verify_mask", "draft_mask")}


def _slot_mask_self(tau, m, S, W):
    row = _orig["slot_write_mask"](tau, m, S, W)
    row[-1] = True
    return row


def _verify_shift(kv_len, Lq):
    mask = np.zeros((Lq, kv_len), dtype=bool)
    for j in range(Lq):
        mask[j, :kv_len - Lq + j] = True
    mask[0, 0] = True
    return mask


def _draft_no_sink(t, n_slots, S, W):
    row = _orig["draft_mask"](t, n_slots, S, W)
    lo, hi = _orig["local_window"](t, S, W)
    row[:min(S, t)] = False
    if hi >= lo:
        row[lo - 1:hi] = True
    return row


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(o, attr, fn)
    caught = _fails_some_pin()
    assert caught is not None, f"no pin caught the planted mistake {name}"
