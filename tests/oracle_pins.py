"""Checks that pin the CPU oracle to things other than itself.

Each ``pin_*`` takes the oracle module and raises AssertionError when the oracle
disagrees with what the pages or the mathematics fix: the hand-derived golden
trace, the deque simulator against the closed forms, textbook special cases,
pure-Python brute force on tiny inputs, and a library routine
(torch scaled_dot_product_attention in float64).  tests/test_oracle_mutations.py
plants plausible mistakes in the oracle and checks that some pin fails.
"""

from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers --

def _rng(seed):
    return np.random.default_rng(seed)


def _load_trace():
    rows, masks = [], []
    with open(os.path.join(GOLDEN, "index_trace_S2_W3_r2.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "mask":
                tau, m = int(parts[1]), int(parts[2])
                raw = [int(x) for x in parts[3].split(",")]
                slots = [] if parts[4] == "-" else [int(x) for x in parts[4].split(",")]
                masks.append((tau, m, raw, slots))
            else:
                rows.append([int(x) for x in parts])
    return rows, masks


def _brute_attention(q, cols_k, cols_v, scale):
    """Eq. 2 for one query head with pure-Python loops: q [D], cols [n][D]."""
    scores = [scale * sum(qi * ki for qi, ki in zip(q, k)) for k in cols_k]
    mx = max(scores)
    w = [math.exp(s - mx) for s in scores]
    z = sum(w)
    out = [sum(w[j] * cols_v[j][d] for j in range(len(w))) / z for d in range(len(q))]
    return out, mx + math.log(z)


# ------------------------------------------------------------------- pins --

def pin_golden_trace(o):
    """Hand-derived trace (tests/golden/index_trace_S2_W3_r2.txt)."""
    S, W, r = 2, 3, 2
    rows, masks = _load_trace()
    sim = o.IndexSim(S, W, r)
    for (t, nsink, lo, hi, evict, bnd, pos, m, r0, r1, r2, ws) in rows:
        dropped = sim.append()
        assert sim.t == t
        assert min(S, t) == nsink and len(sim.sink) == nsink
        assert o.local_window(t, S, W) == (lo, hi), (t, o.local_window(t, S, W))
        assert list(sim.window) == list(range(lo, hi + 1))
        assert (dropped or 0) == evict
        assert bool(o.is_boundary(t, S, W, r)) == bool(bnd)
        assert bool(sim.boundary_due()) == bool(bnd)
        if bnd:
            mm = o.slot_count(t, S, W, r)
            assert o.boundary(mm, S, W, r) == t
            assert o.slot_pos_id(mm, S, W, r) == pos
            assert sim.materialize() == pos
        assert o.slot_count(t, S, W, r) == m == len(sim.slots)
        assert sim.ring_map() == [r0, r1, r2]
        assert o.working_set_size(t, S, W, r) == ws
        assert int(o.draft_mask(t, m, S, W).sum()) == ws
    for tau, m, raw, slots in masks:
        row = o.slot_write_mask(tau, m, S, W)
        got_raw = [i + 1 for i in np.flatnonzero(row[:tau])]
        got_slots = [j + 1 for j in np.flatnonzero(row[tau:])]
        assert got_raw == raw, (tau, got_raw)
        assert got_slots == slots, (tau, got_slots)


def pin_sim_vs_closed_forms(o):
    """Deque simulator == closed forms on a grid of (S, W, r, reserve, t)."""
    for S in (0, 1, 4):
        for W in (1, 3, 8, 16):
            for r in (1, 2, 5, 16):
                for R in (0, 3):
                    sim = o.IndexSim(S, W, r, R)
                    for t in range(1, 3 * (S + W + r) + 2):
                        sim.append()
                        lo, hi = o.local_window(t, S, W)
                        assert list(sim.window) == list(range(lo, hi + 1))
                        assert sim.sink == list(range(1, min(S, t) + 1))
                        assert sim.evicted == list(range(S + 1, max(S + 1, t - W + 1)))
                        assert bool(sim.boundary_due()) == bool(o.is_boundary(t, S, W, r))
                        if sim.boundary_due():
                            mm = len(sim.slots) + 1
                            assert sim.materialize() == o.slot_pos_id(mm, S, W, r)
                        assert len(sim.slots) == o.slot_count(t, S, W, r)
                        assert [tau for tau, _ in sim.slots] == \
                            [o.boundary(j, S, W, r) for j in range(1, len(sim.slots) + 1)]
                        ring = sim.ring_map()
                        for i in range(lo, hi + 1):   # row of token i is (i-S-1) mod (W+R)
                            assert ring[(i - S - 1) % (W + R)] == i
                        mask = o.draft_mask(t, len(sim.slots), S, W)
                        assert [i + 1 for i in np.flatnonzero(mask[:t])] == sim.visible_raw()
                        assert int(mask.sum()) == o.working_set_size(t, S, W, r)


def pin_working_set_at_configs(o):
    """|M_t| = S + min(W, t-S) + floor((t-S-W)/r) at the benchmark shapes:
    4+256+6 = 266; 4+1024+13 = 1041; 4+1024+61 = 1089 (31740 // 512 = 61)."""
    assert o.working_set_size(2048, 4, 256, 256) == 266
    assert o.slot_count(2048, 4, 256, 256) == 6
    assert o.working_set_size(8192, 4, 1024, 512) == 1041
    assert o.slot_count(8192, 4, 1024, 512) == 13
    assert o.working_set_size(32768, 4, 1024, 512) == 1089
    assert o.working_set_size(4096, 4, 1024, 512) == 4 + 1024 + 5
    # the first boundary after an 8192-token prefix falls at step 8196
    assert o.is_boundary(8196, 4, 1024, 512) and o.boundary(14, 4, 1024, 512) == 8196
    assert o.is_boundary(32772, 4, 1024, 512)


def _random_memory(o, S, W, r, Hkv, D, t, batch=1, layers=1, seed=0, G=2):
    rng = _rng(seed)
    mem = o.MaswOracle(S, W, r, Hkv, D, layers, batch)
    for l in range(layers):
        for b in range(batch):
            n = o.slot_count(t, S, W, r)
            mem.load(l, b, rng.standard_normal((t, Hkv, D)), rng.standard_normal((t, Hkv, D)),
                     rng.standard_normal((n, Hkv, D)), rng.standard_normal((n, Hkv, D)))
    q = rng.standard_normal((batch, G * Hkv, D))
    return mem, q, rng


def pin_masw_equals_full_before_eviction(o):
    """No slots and t <= S+W: the draft working set is the whole prefix, so
    MASW attention must equal full attention exactly."""
    for (S, W) in ((4, 16), (0, 8), (3, 5)):
        for t in range(1, S + W + 1):
            mem, q, _ = _random_memory(o, S, W, 7, 2, 8, t, seed=t)
            a, la = mem.draft_attn(0, q)
            b, lb = mem.full_attn(0, q)
            assert np.array_equal(a, b) and np.array_equal(la, lb)
    # and one token past S+W the two differ (token S+1 has left the window)
    mem, q, _ = _random_memory(o, 2, 4, 100, 2, 8, 7, seed=1)
    a, _ = mem.draft_attn(0, q)
    b, _ = mem.full_attn(0, q)
    assert not np.allclose(a, b)


def pin_segments_combine(o):
    """Per-segment softmax (sink, window, slots taken from the simulator) merged
    with the log-sum-exp identity == the oracle's single masked softmax."""
    for seed, (S, W, r, t) in enumerate(((2, 5, 3, 30), (1, 4, 2, 40), (3, 8, 4, 21), (0, 6, 2, 25))):
        Hkv, D = 2, 6
        mem, q, _ = _random_memory(o, S, W, r, Hkv, D, t, seed=seed)
        sim = mem.sim[0][0]
        K, V = mem.raw_k[0][0], mem.raw_v[0][0]
        segs = []
        if sim.sink:
            idx = [i - 1 for i in sim.sink]
            segs.append((K[idx], V[idx]))
        if sim.window:
            idx = [i - 1 for i in sim.window]
            segs.append((K[idx], V[idx]))
        if mem.m(0, 0):
            segs.append((mem.slot_k[0][0], mem.slot_v[0][0]))
        want, want_l = mem.draft_attn(0, q)
        parts = [o.attention(q[0], k, v, np.ones(k.shape[0], bool), mem.scale) for k, v in segs]
        lses = np.stack([p[1] for p in parts])           # [nseg, Hq]
        M = lses.max(0)
        wts = np.exp(lses - M)
        comb = sum(wts[i][:, None] * parts[i][0] for i in range(len(parts))) / wts.sum(0)[:, None]
        assert np.allclose(comb, want[0], rtol=0, atol=1e-12)
        assert np.allclose(M + np.log(wts.sum(0)), want_l[0], rtol=0, atol=1e-12)


def pin_bruteforce_tiny(o):
    """Pure-Python loops over the simulator's visible set, for draft, slot
    write, full and verify, with GQA (Hkv=2, G=2) and a non-default scale."""
    S, W, r, Hkv, D, G = 2, 3, 2, 2, 4, 2
    rng = _rng(11)
    scale = 0.37
    mem = o.MaswOracle(S, W, r, Hkv, D, 1, 1, scale=scale)
    for t in range(1, 14):
        k = rng.standard_normal((1, Hkv, D))
        v = rng.standard_normal((1, Hkv, D))
        mem.append(0, k, v)
        q = rng.standard_normal((1, G * Hkv, D))
        got, got_l = mem.draft_attn(0, q)
        sim = mem.sim[0][0]
        for h in range(G * Hkv):
            kv = h // G
            ck = [list(mem.raw_k[0][0][i - 1, kv]) for i in sim.visible_raw()] + \
                 [list(x) for x in mem.slot_k[0][0][:, kv]]
            cv = [list(mem.raw_v[0][0][i - 1, kv]) for i in sim.visible_raw()] + \
                 [list(x) for x in mem.slot_v[0][0][:, kv]]
            want, wl = _brute_attention(list(q[0, h]), ck, cv, scale)
            assert np.allclose(got[0, h], want, rtol=0, atol=1e-12), (t, h)
            assert abs(got_l[0, h] - wl) < 1e-12
        got_f, _ = mem.full_attn(0, q)
        for h in range(G * Hkv):
            kv = h // G
            want, _ = _brute_attention(list(q[0, h]), [list(x) for x in mem.raw_k[0][0][:, kv]],
                                       [list(x) for x in mem.raw_v[0][0][:, kv]], scale)
            assert np.allclose(got_f[0, h], want, rtol=0, atol=1e-12)
        if o.is_boundary(t, S, W, r):
            qg = rng.standard_normal((1, G * Hkv, D))
            kg = rng.standard_normal((1, Hkv, D))
            vg = rng.standard_normal((1, Hkv, D))
            prev_k = mem.slot_k[0][0].copy()
            prev_v = mem.slot_v[0][0].copy()
            vis = list(sim.visible_raw())
            got_g, _ = mem.materialize_slot(0, [0], qg, kg, vg)
            for h in range(G * Hkv):
                kv = h // G
                ck = [list(mem.raw_k[0][0][i - 1, kv]) for i in vis] + [list(x) for x in prev_k[:, kv]]
                cv = [list(mem.raw_v[0][0][i - 1, kv]) for i in vis] + [list(x) for x in prev_v[:, kv]]
                want, _ = _brute_attention(list(qg[0, h]), ck, cv, scale)
                assert np.allclose(got_g[0, h], want, rtol=0, atol=1e-12)
    # verify: B=1, Lq=3, kv_len=7 in a cache of 9 rows
    Lq, n, Tmax = 3, 7, 9
    qv = rng.standard_normal((1, Lq, G * Hkv, D))
    kc = rng.standard_normal((1, Hkv, Tmax, D))
    vc = rng.standard_normal((1, Hkv, Tmax, D))
    got_v, _ = o.verify_attn(qv, kc, vc, [n], scale)
    for j in range(Lq):
        for h in range(G * Hkv):
            kv = h // G
            keys = n - Lq + 1 + j
            want, _ = _brute_attention(list(qv[0, j, h]), [list(kc[0, kv, i]) for i in range(keys)],
                                       [list(vc[0, kv, i]) for i in range(keys)], scale)
            assert np.allclose(got_v[0, j, h], want, rtol=0, atol=1e-12)


def pin_q_zero_and_single(o):
    """q = 0: uniform weights, O = mean of V over exactly the visible set and
    LSE = log |set|.  A single visible column: O = that V exactly."""
    S, W, r, Hkv, D = 3, 5, 2, 2, 8
    mem, q, _ = _random_memory(o, S, W, r, Hkv, D, 23, seed=5)
    q[:] = 0.0
    got, lse = mem.draft_attn(0, q)
    sim = mem.sim[0][0]
    for h in range(q.shape[1]):
        kv = h // (q.shape[1] // Hkv)
        rows = [mem.raw_v[0][0][i - 1, kv] for i in sim.visible_raw()] + list(mem.slot_v[0][0][:, kv])
        assert np.allclose(got[0, h], np.mean(rows, axis=0), rtol=0, atol=1e-13)
        assert abs(lse[0, h] - math.log(len(rows))) < 1e-13
    mem1, q1, _ = _random_memory(o, 4, 8, 2, 2, 8, 1, seed=6)
    got1, lse1 = mem1.draft_attn(0, q1)
    for h in range(q1.shape[1]):
        kv = h // (q1.shape[1] // 2)
        assert np.array_equal(got1[0, h], mem1.raw_v[0][0][0, kv])
        assert abs(lse1[0, h] - mem1.scale * float(q1[0, h] @ mem1.raw_k[0][0][0, kv])) < 1e-13


def pin_one_hot_exclusion(o):
    """V_i = e_i: O is the weight vector.  Every raw token outside sink and
    window (and, for a slot write, g_m itself) gets weight exactly 0; every
    visible column gets a positive weight."""
    S, W, r, Hkv = 2, 4, 3, 1
    t = 17
    n = o.slot_count(t, S, W, r)
    D = t + n + 1
    rng = _rng(3)
    mem = o.MaswOracle(S, W, r, Hkv, D, 1, 1)
    eye = np.eye(D)
    mem.load(0, 0, rng.standard_normal((t, Hkv, D)), eye[:t, None, :],
             rng.standard_normal((n, Hkv, D)), eye[t:t + n, None, :])
    q = rng.standard_normal((1, 2, D)) * 0.1
    got, _ = mem.draft_attn(0, q)
    vis = set(mem.sim[0][0].visible_raw())
    for h in range(2):
        for i in range(1, t + 1):
            if i in vis:
                assert got[0, h, i - 1] > 0
            else:
                assert got[0, h, i - 1] == 0.0
        assert np.all(got[0, h, t:t + n] > 0)
    # advance to the next boundary and write slot n+1 with V = e_{t+n}
    while not o.is_boundary(mem.t(0, 0), S, W, r):
        mem.append(0, rng.standard_normal((1, Hkv, D)), np.zeros((1, Hkv, D)))
    tau = mem.t(0, 0)
    vis = set(mem.sim[0][0].visible_raw())
    vg = np.zeros((1, Hkv, D))
    vg[0, 0, D - 1] = 1.0
    got_g, _ = mem.materialize_slot(0, [0], q, rng.standard_normal((1, Hkv, D)), vg)
    assert got_g[0, 0, D - 1] == 0.0                  # g_m does not read itself
    for i in range(1, t + 1):                          # original one-hot tokens
        if i not in vis:
            assert got_g[0, 0, i - 1] == 0.0
    assert np.all(got_g[0, 0, t:t + n] > 0)            # every earlier slot is read
    assert tau == o.boundary(n + 1, S, W, r)


def pin_sdpa(o):
    """torch.nn.functional.scaled_dot_product_attention in float64 with an
    explicit boolean mask and GQA, default scale 1/sqrt(D), for full decode and
    for causal verify."""
    import torch
    import torch.nn.functional as F
    rng = _rng(9)
    B, Hkv, G, D, T = 2, 2, 3, 16, 29
    mem = o.MaswOracle(4, 8, 4, Hkv, D, 1, B)
    kr = rng.standard_normal((B, T, Hkv, D))
    vr = rng.standard_normal((B, T, Hkv, D))
    for b in range(B):
        n = o.slot_count(T, 4, 8, 4)
        mem.load(0, b, kr[b], vr[b], np.zeros((n, Hkv, D)), np.zeros((n, Hkv, D)))
    q = rng.standard_normal((B, G * Hkv, D))
    got, _ = mem.full_attn(0, q)
    qt = torch.from_numpy(q)[:, :, None, :]                        # [B, Hq, 1, D]
    kt = torch.from_numpy(kr).permute(0, 2, 1, 3)                   # [B, Hkv, T, D]
    vt = torch.from_numpy(vr).permute(0, 2, 1, 3)
    ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.ones(1, T, dtype=torch.bool),
                                         enable_gqa=True)[:, :, 0, :]
    assert np.allclose(got, ref.numpy(), rtol=0, atol=1e-12)
    # draft attention == SDPA with the draft mask row
    got_d, _ = mem.draft_attn(0, q)
    m = o.slot_count(T, 4, 8, 4)
    row = torch.from_numpy(o.draft_mask(T, m, 4, 8))
    kc = torch.cat([kt, torch.zeros(B, Hkv, m, D, dtype=torch.float64)], 2)
    vc = torch.cat([vt, torch.zeros(B, Hkv, m, D, dtype=torch.float64)], 2)
    ref_d = F.scaled_dot_product_attention(qt, kc, vc, attn_mask=row[None, :], enable_gqa=True)[:, :, 0, :]
    assert np.allclose(got_d, ref_d.numpy(), rtol=0, atol=1e-12)
    # verify
    Lq, Tmax = 5, 40
    kv_len = [37, 12]
    qv = rng.standard_normal((B, Lq, G * Hkv, D))
    kc = rng.standard_normal((B, Hkv, Tmax, D))
    vc = rng.standard_normal((B, Hkv, Tmax, D))
    got_v, _ = o.verify_attn(qv, kc, vc, kv_len)
    for b in range(B):
        n = kv_len[b]
        causal = torch.ones(Lq, n, dtype=torch.bool).tril(diagonal=n - Lq)
        ref_v = F.scaled_dot_product_attention(torch.from_numpy(qv[b]).permute(1, 0, 2),
                                               torch.from_numpy(kc[b, :, :n]), torch.from_numpy(vc[b, :, :n]),
                                               attn_mask=causal, enable_gqa=True)
        assert np.allclose(got_v[b], ref_v.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def pin_permutation(o):
    """Softmax attention is invariant to the order of its columns (so a ring
    may be read in physical row order)."""
    rng = _rng(4)
    N, Hkv, D = 23, 2, 8
    K = rng.standard_normal((N, Hkv, D))
    V = rng.standard_normal((N, Hkv, D))
    mask = rng.random(N) < 0.6
    q = rng.standard_normal((4, D))
    a, la = o.attention(q, K, V, mask, 0.3)
    p = rng.permutation(N)
    b, lb = o.attention(q, K[p], V[p], mask[p], 0.3)
    assert np.allclose(a, b, rtol=0, atol=1e-13) and np.allclose(la, lb, rtol=0, atol=1e-13)


def pin_verify_rows_are_decodes(o):
    """Verify row j equals a full-KV decode over the first kv_len-Lq+1+j keys."""
    rng = _rng(8)
    B, Hkv, G, D, Lq, Tmax = 1, 2, 2, 8, 6, 50
    kc = rng.standard_normal((B, Hkv, Tmax, D))
    vc = rng.standard_normal((B, Hkv, Tmax, D))
    q = rng.standard_normal((B, Lq, G * Hkv, D))
    n = 44
    got, got_l = o.verify_attn(q, kc, vc, [n])
    for j in range(Lq):
        keys = n - Lq + 1 + j
        want, wl = o.attention(q[0, j], kc[0, :, :keys].transpose(1, 0, 2), vc[0, :, :keys].transpose(1, 0, 2),
                               np.ones(keys, bool), 1 / math.sqrt(D))
        assert np.allclose(got[0, j], want, rtol=0, atol=1e-13)
        assert np.allclose(got_l[0, j], wl, rtol=0, atol=1e-13)


def pin_rollback(o):
    """Rolling back k <= R tokens and re-appending the same tokens reproduces
    the state and outputs; slots made after the rollback point are dropped;
    rolling back deeper than R is refused."""
    S, W, r, R, Hkv, D = 2, 4, 3, 3, 1, 4
    rng = _rng(12)
    mem = o.MaswOracle(S, W, r, Hkv, D, 2, 1, reserve=R)
    toks = [(rng.standard_normal((1, Hkv, D)), rng.standard_normal((1, Hkv, D))) for _ in range(30)]
    slotkv = [(rng.standard_normal((1, 2, D)), rng.standard_normal((1, Hkv, D)), rng.standard_normal((1, Hkv, D)))
              for _ in range(30)]
    q = rng.standard_normal((1, 2, D))

    def run(lo, hi):
        for t in range(lo, hi):
            for l in range(2):
                mem.append(l, *toks[t])
                if o.is_boundary(mem.t(l, 0), S, W, r):
                    mem.materialize_slot(l, [0], *slotkv[t])
    run(0, 20)
    ref = [mem.draft_attn(l, q)[0] for l in range(2)]
    run(20, 23)     # crosses tau_5 = 2+4+15 = 21
    assert mem.m(0, 0) == 5
    mem.rollback([0], [20])
    assert mem.t(0, 0) == 20 and mem.m(0, 0) == 4
    for l in range(2):
        assert np.array_equal(mem.draft_attn(l, q)[0], ref[l])
    assert list(mem.sim[0][0].window) == list(range(17, 21))
    run(20, 23)
    mem.rollback([0], [20])
    for l in range(2):
        assert np.array_equal(mem.draft_attn(l, q)[0], ref[l])
    try:
        run(20, 24)
        mem.rollback([0], [20])
    except RuntimeError:
        pass
    else:
        raise AssertionError("rollback by 4 > R=3 must be refused")


def pin_greedy_accept(o):
    """Greedy acceptance against a hand loop on tiny logits, with the special
    cases: all drafts accepted (bonus token), first draft rejected, ties going
    to the smallest id, NaN entries skipped, +-inf rows, and an all-NaN row
    (token -1, which rejects the draft at that position)."""
    rng = _rng(21)
    B, L, V = 5, 4, 11
    logits = rng.standard_normal((B, L + 1, V))
    arg = logits.argmax(-1)
    draft = arg[:, :L].copy()
    draft[1, 0] = (arg[1, 0] + 1) % V           # first rejected
    draft[2, 2] = (arg[2, 2] + 3) % V           # two accepted
    draft[3, 3] = (arg[3, 3] + 1) % V           # three accepted
    tokens, n_emit = o.greedy_accept(logits, draft)
    for b in range(B):
        want_tok = []
        for j in range(L + 1):
            best, bi = -math.inf, -1
            for v in range(V):
                if logits[b, j, v] > best:
                    best, bi = logits[b, j, v], v
            want_tok.append(bi)
        k = 0
        while k < L and draft[b, k] == want_tok[k]:
            k += 1
        assert list(tokens[b]) == want_tok
        assert n_emit[b] == k + 1
    assert list(n_emit) == [L + 1, 1, 3, 4, L + 1]
    tied = np.zeros((1, 2, 6))
    tied[0, 0, [2, 4]] = 1.0
    tok, n = o.greedy_accept(tied, np.array([[2]]))
    assert tok[0, 0] == 2 and n[0] == 2 and tok[0, 1] == 0
    # NaN entries are skipped, +-inf are values, an all-NaN row has no token
    # (-1), which no draft equals; expected ids written out by hand
    nan, inf = math.nan, math.inf
    rows = [[1.0, nan, 3.0, nan, 3.0, 0.0],          # -> 2 (NaN skipped, tie to the smaller id)
            [nan, nan, nan, nan, nan, nan],          # -> -1
            [-inf, nan, -inf, -inf, nan, -inf],      # -> 0 (-inf is a value)
            [nan, -inf, 5.0, inf, inf, nan],         # -> 3
            [nan, nan, nan, nan, nan, -2.5]]         # -> 5
    tok, n = o.greedy_accept(np.array([rows]), np.array([[2, 1, 0, 3]]))
    assert list(tok[0]) == [2, -1, 0, 3, 5] and n[0] == 2
    tok, n = o.greedy_accept(np.array([[rows[3], rows[4], rows[1]]]), np.array([[3, 5]]))
    assert list(tok[0]) == [3, 5, -1] and n[0] == 3


def pin_eq1(o):
    """Eq. 1 limits: a free draft gives L_acc + 1; with t_d = t_t and nothing
    accepted the speedup is 1 / (L_draft + 1)."""
    assert o.eq1_speedup(5, 5, 0.0, 1.0) == 6.0
    assert abs(o.eq1_speedup(0, 5, 1.0, 1.0) - 1.0 / 6.0) < 1e-15
    assert abs(o.eq1_speedup(3.0, 5, 0.1, 1.0) - 4.0 / 1.5) < 1e-15


def pin_prefill_equals_incremental(o):
    """Prefill under the structured mask == appending the same tokens one by one
    with a draft query after each append and the slot write at each boundary
    (the decode-time definitions); a plain causal prefill differs."""
    S, W, r, Hkv, G, D, T = 2, 5, 3, 2, 2, 4, 26
    rng = _rng(31)
    M = o.slot_count(T, S, W, r)
    qr, kr, vr = rng.standard_normal((T, G * Hkv, D)), rng.standard_normal((T, Hkv, D)), rng.standard_normal((T, Hkv, D))
    qs, ks, vs = rng.standard_normal((M, G * Hkv, D)), rng.standard_normal((M, Hkv, D)), rng.standard_normal((M, Hkv, D))
    o_raw, l_raw, o_slot, l_slot = o.prefill_attn(S, W, r, qr, kr, vr, qs, ks, vs)
    mem = o.MaswOracle(S, W, r, Hkv, D, 1, 1)
    m = 0
    for i in range(T):
        mem.append(0, kr[i][None], vr[i][None])
        got, gl = mem.draft_attn(0, qr[i][None])
        assert np.allclose(got[0], o_raw[i], rtol=0, atol=1e-12) and np.allclose(gl[0], l_raw[i], rtol=0, atol=1e-12)
        if o.is_boundary(i + 1, S, W, r):
            gs, gsl = mem.materialize_slot(0, [0], qs[m][None], ks[m][None], vs[m][None])
            assert np.allclose(gs[0], o_slot[m], rtol=0, atol=1e-12)
            m += 1
    assert m == M
    causal, _ = o.attention(qr[-1], kr, vr, np.ones(T, bool), 1 / math.sqrt(D))
    assert not np.allclose(causal, o_raw[-1])


ALL_PINS = [
    pin_golden_trace, pin_sim_vs_closed_forms, pin_working_set_at_configs,
    pin_masw_equals_full_before_eviction, pin_segments_combine, pin_bruteforce_tiny,
    pin_q_zero_and_single, pin_one_hot_exclusion, pin_sdpa, pin_permutation,
    pin_verify_rows_are_decodes, pin_rollback, pin_greedy_accept, pin_eq1, pin_prefill_equals_incremental,
]
