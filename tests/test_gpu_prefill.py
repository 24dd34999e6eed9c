"""Draft prefill (masw_prefill) against the oracle's prefill under the structured
write mask, then decoding continued from the stored memory M_0."""
import pytest
import torch

import oracle.masw_oracle as orc
from compressed_draft_kv_gb300 import capi

from gpu_helpers import DEV, Pair

pytestmark = pytest.mark.gpu

# (S, W, r, Hkv, G, T): several 128-row tiles of the interleaved order with
# ragged tails, r > W (one slot per tile), no sink, prefixes inside the sink and
# inside the first window, r = 1 (a slot after every raw token past S + W: half
# the rows of a tile are slot rows, and slot prefixes below and above the 56 a
# merged sink + slot block holds), the paper's S = W = 128 with r = 4
CASES = [
    (4, 8, 1, 2, 4, 200),
    (1, 3, 2, 1, 2, 140),
    (4, 16, 4, 2, 4, 100),
    (4, 16, 4, 1, 8, 257),
    (0, 32, 8, 2, 2, 200),
    (8, 16, 4, 2, 4, 5),
    (4, 64, 16, 2, 4, 60),
    (4, 8, 16, 1, 4, 150),
    (2, 40, 3, 2, 1, 333),
    (128, 128, 4, 2, 4, 1024),
]


@pytest.mark.parametrize("S,W,r,Hkv,G,T", CASES)
def test_prefill_matches_oracle(S, W, r, Hkv, G, T):
    p = Pair(S, W, r, Hkv, 128, layers=2, batch=3, dtype="bf16", Hq=Hkv * G, max_seq_len=T + 64,
             tag=f"prefill{S}_{W}_{r}_{T}")
    try:
        p.prefill(1, 2, T)
        p.check_state(1, 2)
    finally:
        p.close()


def test_prefill_self_attend_and_scale():
    p = Pair(4, 16, 4, 2, 128, layers=1, batch=1, dtype="bf16", Hq=8, max_seq_len=256, self_attend=True,
             scale=0.05, tag="prefill_sa")
    try:
        p.prefill(0, 0, 130)
        p.check_state(0, 0)
    finally:
        p.close()


def test_decode_continues_after_prefill():
    """Prefill every sequence to a different length, then fused draft steps (with
    slot writes at the boundaries), a rollback and more steps, all against the
    oracle; the full-KV cache written by the prefill is checked too."""
    S, W, r, Hkv, G, R = 4, 24, 4, 2, 4, 6
    B = 3
    p = Pair(S, W, r, Hkv, 128, layers=1, batch=B, dtype="bf16", Hq=Hkv * G, max_seq_len=400, full_kv=True,
             reserve=R, tag="prefill_cont")
    try:
        lens = [37, 64, 29]            # one mid-window, one on a boundary, one just past S+W
        for b, t in enumerate(lens):
            p.prefill(0, b, t, seed=b)
            p.check_state(0, b)
        for step in range(12):
            p.step = step
            due = [b for b in range(B) if orc.is_boundary(p.ref.t(0, b) + 1, S, W, r)]
            if due:
                p.fstep_slot(0, due)
            else:
                p.fstep(0)
            p.draft(0, full=True)
        for b in range(B):
            p.check_state(0, b)
        t_new = [p.ref.t(0, b) - k for b, k in enumerate((R, 1, 3))]
        capi.masw_rollback(p.h, list(range(B)), t_new)
        p.ref.rollback(list(range(B)), t_new)
        for step in range(12, 20):
            p.step = step
            due = [b for b in range(B) if orc.is_boundary(p.ref.t(0, b) + 1, S, W, r)]
            if due:
                p.fstep_slot(0, due)
            else:
                p.fstep(0)
        for b in range(B):
            p.check_state(0, b)
    finally:
        p.close()


def test_prefill_rejects_bad_calls():
    p = Pair(4, 16, 4, 2, 128, layers=1, batch=1, dtype="bf16", Hq=8, max_seq_len=64, tag="prefill_bad")
    q = torch.zeros(65, 8, 128, dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros(65, 2, 128, dtype=torch.bfloat16, device=DEV)
    o = torch.empty(65, 8, 128, device=DEV)
    try:
        with pytest.raises(capi.MaswError):        # T > max_seq_len
            capi.masw_prefill(p.h, 0, 0, q, kv, kv, q, kv, kv, o)
        with pytest.raises(capi.MaswError):        # slots needed but none given
            capi.masw_prefill(p.h, 0, 0, q[:40], kv[:40], kv[:40], None, None, None, o)
        with pytest.raises(capi.MaswError):        # seq out of range
            capi.masw_prefill(p.h, 0, 1, q[:8], kv[:8], kv[:8], None, None, None, o)
    finally:
        p.close()
    f = Pair(4, 16, 4, 2, 64, layers=1, batch=1, dtype="f32", Hq=8, max_seq_len=64, tag="prefill_f32")
    try:
        q32 = torch.zeros(8, 8, 64, device=DEV)
        kv32 = torch.zeros(8, 2, 64, device=DEV)
        with pytest.raises(capi.MaswError):        # bf16 / head_dim 128 pools only
            capi.masw_prefill(f.h, 0, 0, q32, kv32, kv32, None, None, None, torch.empty(8, 8, 64, device=DEV))
    finally:
        f.close()


def test_prefill_full_size_sampled_rows():
    """The benchmark's launch configuration (3B-draft attention shape, 32K prefix,
    S = 4, W = 1024, r = 512, 61 slots): raw rows (sink, first window, first
    boundaries, middle, last, and one in every 128-row query tile) and every
    slot row against the oracle's per-row evaluation, and the stored memory bit
    for bit."""
    import numpy as np
    from compressed_draft_kv_gb300 import synth
    S, W, r, Hkv, G, T, D = 4, 1024, 512, 8, 3, 32768, 128
    Hq = Hkv * G
    p = Pair(S, W, r, Hkv, D, layers=1, batch=1, dtype="bf16", Hq=Hq, max_seq_len=T + 64, reserve=16,
             tag="prefill_full")
    try:
        M = orc.slot_count(T, S, W, r)
        g = lambda shape, name: synth.normal(shape, "bf16", "prefill_full", name)
        qr, kr, vr = g((T, Hq, D), "q"), g((T, Hkv, D), "k"), g((T, Hkv, D), "v")
        qs, ks, vs = g((M, Hq, D), "qs"), g((M, Hkv, D), "ks"), g((M, Hkv, D), "vs")
        o_r = torch.empty(T, Hq, D, device=DEV)
        l_r = torch.empty(T, Hq, device=DEV)
        o_s = torch.empty(M, Hq, D, device=DEV)
        l_s = torch.empty(M, Hq, device=DEV)
        capi.masw_prefill(p.h, 0, 0, qr.to(DEV), kr.to(DEV), vr.to(DEV), qs.to(DEV), ks.to(DEV), vs.to(DEV),
                          o_r, l_r, o_s, l_s)
        capi.masw_sync(p.h)
        rng = np.random.default_rng(17)
        # the special rows, one seeded row in every 128-row query tile of the
        # launch, and every slot row
        per_tile = [int(rng.integers(j + 1, min(j + 128, T) + 1)) for j in range(0, T, 128)]
        raw_rows = sorted(set([1, 3, 4, 5, 64, 129, S + W, S + W + 1, S + W + r, S + W + r + 1, 16384, T - 1, T]
                              + per_tile))
        slot_rows = list(range(1, M + 1))
        want = orc.prefill_attn(S, W, r, qr.float().numpy(), kr.float().numpy(), vr.float().numpy(),
                                qs.float().numpy(), ks.float().numpy(), vs.float().numpy(),
                                raw_rows=raw_rows, slot_rows=slot_rows)
        ri = [i - 1 for i in raw_rows]
        si = [m - 1 for m in slot_rows]
        from gpu_helpers import assert_close
        assert_close(o_r[ri], want[0][ri], "bf16", "full-size prefill O_raw")
        assert_close(l_r[ri], want[1][ri], "bf16", "full-size prefill LSE_raw")
        assert_close(o_s[si], want[2][si], "bf16", "full-size prefill O_slot")
        assert_close(l_s[si], want[3][si], "bf16", "full-size prefill LSE_slot")
        # every row of the launch, not only the sampled ones, is finite
        assert torch.isfinite(o_r).all() and torch.isfinite(l_r).all() and torch.isfinite(o_s).all()
        p.ref.load(0, 0, kr.float().numpy(), vr.float().numpy(), ks.float().numpy(), vs.float().numpy())
        p.check_state(0, 0)
    finally:
        p.close()
