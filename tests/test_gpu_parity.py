"""GPU parity: every C-ABI call against the CPU oracle on the same seeded inputs.

Indices (counters, ring placement, slot ids) are compared bit for bit; attention
outputs within the stated tolerance (fp32 inputs: 2e-5 absolute; bf16 inputs:
max abs <= 1e-2 and relative L2 <= 5e-3).
"""
import numpy as np
import pytest
import torch

import oracle.masw_oracle as orc
from compressed_draft_kv_gb300 import capi, synth
from gpu_helpers import DEV, Guarded, Pair, assert_close, to_np
from libmasw_fixture import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    torch.cuda.set_device(DEV)


def test_tiny_f32_single_layer():
    """8q/2kv heads, D=64, fp32, t=2048, S=4, W=256, r=256 (6 slots): a draft
    step, appends up to tau_7 = 2052, the slot write there and eviction."""
    p = Pair(4, 256, 256, 2, 64, 1, 1, "f32", 8, max_seq_len=4096, full_kv=True, tag="tiny")
    try:
        p.load(0, 0, 2048, seed=0)
        assert p.ref.m(0, 0) == 6
        p.check_state(0, 0)
        p.draft(0)
        p.draft(0, full=True)
        for step in range(2049, 2054):
            p.step = step
            p.append(0)
            p.draft(0)
            p.draft(0, full=True)
            if orc.is_boundary(step, 4, 256, 256):
                assert step == 2052
                p.materialize(0, [0])
            p.check_state(0, 0)
        assert p.ref.m(0, 0) == 7
    finally:
        p.close()


def test_draft3b_shape_one_layer_8k():
    """24q/8kv heads, D=128, bf16, t=8192 (13 slots), S=4, W=1024, r=512: five
    draft steps; the boundary tau_14 = 8196 is crossed at the fourth."""
    p = Pair(4, 1024, 512, 8, 128, 1, 1, "bf16", 24, max_seq_len=8192 + 16, full_kv=True, tag="cfg2")
    try:
        p.load(0, 0, 8192, seed=1)
        assert p.ref.m(0, 0) == 13
        p.draft(0)
        for step in range(8193, 8198):
            p.step = step
            p.append(0)
            p.draft(0)
            p.draft(0, full=True)
            if step == 8196:
                p.materialize(0, [0])
        p.check_state(0, 0)
        assert p.ref.m(0, 0) == 14
    finally:
        p.close()


@pytest.mark.parametrize("dtype,D,G", [("f32", 64, 4), ("bf16", 128, 3), ("bf16", 64, 8), ("f32", 128, 1)])
def test_masw_equals_full_before_eviction(dtype, D, G):
    """No slots and t <= S+W: the draft working set is the whole prefix."""
    S, W = 5, 100
    p = Pair(S, W, 16, 2, D, 1, 1, dtype, 2 * G, max_seq_len=256, full_kv=True, tag="eq")
    try:
        for t in range(1, S + W + 1):
            p.step = t
            p.append(0)
            if t in (1, S, S + 1, 37, S + W):
                q = p.rand((1, 2 * G, D), "q")
                o1, l1, want, _ = p.draft(0, q=q)
                o2, l2, want_f, _ = p.draft(0, q=q, full=True)
                assert np.array_equal(want, want_f)
                assert_close(o1, to_np(o2), "f32", f"draft vs full t={t}")
        p.check_state(0, 0)
    finally:
        p.close()


def test_one_hot_values_show_exact_exclusion():
    """V_i = e_i: the output is the weight vector.  Raw tokens outside sink and
    window get exactly 0 on the GPU, every visible column a positive weight;
    the slot query reads neither evicted tokens nor itself."""
    S, W, r, D = 2, 8, 4, 64
    t = 40
    p = Pair(S, W, r, 1, D, 1, 1, "f32", 2, max_seq_len=64, tag="onehot")
    try:
        n = orc.slot_count(t, S, W, r)
        eye = torch.eye(D, dtype=torch.float32)
        kr = synth.normal((t, 1, D), "f32", "onehot", "k") * 0.2
        vr = eye[:t, None, :].contiguous()
        ks = synth.normal((n, 1, D), "f32", "onehot", "ks") * 0.2
        vs = eye[t:t + n, None, :].contiguous()
        capi.masw_mem_load(p.h, 0, 0, kr, vr, ks, vs)
        p.ref.load(0, 0, kr.numpy(), vr.numpy(), ks.numpy(), vs.numpy())
        q = synth.normal((1, 2, D), "f32", "onehot", "q") * 0.2
        o, _, want, _ = p.draft(0, q=q)
        o = to_np(o)
        vis = set(p.ref.sim[0][0].visible_raw())
        for i in range(1, t + 1):
            if i in vis:
                assert (o[0, :, i - 1] > 0).all()
            else:
                assert (o[0, :, i - 1] == 0).all(), f"evicted token {i} has weight {o[0, :, i - 1]}"
        assert (o[0, :, t:t + n] > 0).all()
        # advance to the next boundary (tau_8 = 2 + 8 + 32 = 42); new tokens carry V = 0
        for i in range(t + 1, 43):
            k = synth.normal((1, 1, D), "f32", "onehot", "k", i) * 0.2
            v = torch.zeros(1, 1, D)
            capi.masw_append_kv(p.h, 0, k.to(DEV), v.to(DEV))
            p.ref.append(0, k.numpy(), v.numpy())
        assert orc.is_boundary(42, S, W, r)
        vis = set(p.ref.sim[0][0].visible_raw())
        qg = synth.normal((1, 2, D), "f32", "onehot", "qg") * 0.2
        kg = synth.normal((1, 1, D), "f32", "onehot", "kg") * 0.2
        vg = torch.zeros(1, 1, D)
        vg[0, 0, D - 1] = 1.0
        og = torch.empty(1, 2, D, device=DEV)
        capi.masw_materialize_slot(p.h, 0, [0], qg.to(DEV), kg.to(DEV), vg.to(DEV), og)
        want_g, _ = p.ref.materialize_slot(0, [0], qg.numpy(), kg.numpy(), vg.numpy())
        og = to_np(og)
        assert_close(og, want_g, "f32", "slot one-hot")
        assert (og[0, :, D - 1] == 0).all(), "slot query read its own K/V"
        for i in range(1, t + 1):
            if i not in vis:
                assert (og[0, :, i - 1] == 0).all()
        assert (og[0, :, t:t + n] > 0).all()
    finally:
        p.close()


def test_ragged_batch_active_mask_and_edges():
    """Three sequences at different points (empty, sink-only, past several
    boundaries), appends with an active mask, G = 8, D = 64, S = 0 excluded."""
    S, W, r = 3, 40, 7
    p = Pair(S, W, r, 2, 64, 2, 3, "bf16", 16, max_seq_len=400, full_kv=True, tag="ragged")
    try:
        for l in range(2):
            p.load(l, 1, 2, seed=l)        # inside the sink
            p.load(l, 2, 150, seed=l)      # 15 slots
        o, lse, want, want_l = p.draft(0)
        assert np.isneginf(want_l[0]).all() and (to_np(o)[0] == 0).all() and torch.isinf(lse[0]).all()
        for step in range(1, 30):
            p.step = step
            active = [1, step % 2, 1]
            for l in range(2):
                p.append(l, active=active)
                p.draft(l)
                due = [b for b in range(3) if orc.is_boundary(p.ref.t(l, b), S, W, r)
                       and p.ref.m(l, b) == orc.slot_count(p.ref.t(l, b), S, W, r) - 1]
                if due:
                    p.materialize(l, due)
            if step % 7 == 0:
                p.draft(1, full=True)
        for l in range(2):
            for b in range(3):
                p.check_state(l, b)
    finally:
        p.close()


def test_maximum_batch_ragged_active_and_boundaries():
    """The largest batch a handle holds (MASW_MAX_BATCH = 512 sequences), every
    sequence at its own prefix: fused steps with an active mask over all 16
    words of the mask, and at each step the fused slot write for exactly the
    sequences that reach a boundary (row ids up to 511); every sequence's
    output is compared with the oracle at every step, and a sample of memories
    row by row."""
    S, W, r, Hkv, G, D = 2, 6, 3, 1, 3, 64
    B = capi.MASW_MAX_BATCH
    p = Pair(S, W, r, Hkv, D, 1, B, "bf16", Hkv * G, max_seq_len=64, tag="maxbatch")
    try:
        for b in range(B):
            p.load(0, b, b % 23, seed=1)
        for step in range(6):
            p.step = step
            active = [int((b + step) % 5 != 0) for b in range(B)]
            due = [b for b in range(B) if active[b] and orc.is_boundary(p.ref.t(0, b) + 1, S, W, r)
                   and p.ref.m(0, b) == orc.slot_count(p.ref.t(0, b) + 1, S, W, r) - 1]
            if due:
                p.fstep_slot(0, due, active=active)
            else:
                p.fstep(0, active=active)
        capi.masw_sync(p.h)
        for b in (0, 1, 255, 256, 510, 511):
            p.check_state(0, b)
    finally:
        p.close()


@pytest.mark.parametrize("S,W,r,dtype", [(0, 1, 1, "bf16"), (1, 1, 1, "f32"), (0, 2, 3, "bf16"), (3, 1, 5, "f32")])
def test_degenerate_windows_and_rates(S, W, r, dtype):
    """Degenerate memories: a one-token window, a slot for every evicted token
    (r = 1), no sink, a slot rate above the window: fused steps from an empty
    memory through many boundaries, the fused slot write at each, checked
    against the oracle at every step and row by row at the end."""
    Hkv, G, D = 2, 2, 64
    B, T = 2, 40
    p = Pair(S, W, r, Hkv, D, 1, B, dtype, Hkv * G, max_seq_len=T + 4, tag=f"degen{S}{W}{r}")
    try:
        for step in range(T):
            p.step = step
            due = [b for b in range(B) if orc.is_boundary(p.ref.t(0, b) + 1, S, W, r)]
            if due and dtype == "bf16":
                p.fstep_slot(0, due)
            else:
                p.fstep(0)
                if due:
                    p.materialize(0, due)
        capi.masw_sync(p.h)
        for b in range(B):
            assert p.ref.m(0, b) == orc.slot_count(T, S, W, r)
            p.check_state(0, b)
    finally:
        p.close()


def test_no_sink_r_larger_than_w_and_scale():
    """S = 0 (pure window plus slots), r > W, an explicit softmax scale."""
    p = Pair(0, 16, 40, 2, 128, 1, 2, "bf16", 4, max_seq_len=600, scale=0.05, tag="nosink")
    try:
        p.load(0, 0, 300, seed=3)
        p.load(0, 1, 57, seed=4)
        for step in range(60):
            p.step = step
            p.append(0)
            p.draft(0)
            due = [b for b in range(2) if orc.is_boundary(p.ref.t(0, b), 0, 16, 40)]
            if due:
                p.materialize(0, due)
        p.check_state(0, 0)
        p.check_state(0, 1)
    finally:
        p.close()


def test_slot_self_attend_option():
    p = Pair(2, 8, 4, 2, 64, 1, 1, "f32", 4, max_seq_len=64, self_attend=True, tag="selfatt")
    try:
        p.load(0, 0, 21, seed=0)
        for step in range(6):
            p.step = step
            p.append(0)
            p.draft(0)
            if orc.is_boundary(p.ref.t(0, 0), 2, 8, 4):
                p.materialize(0, [0])
        p.check_state(0, 0)
    finally:
        p.close()


def test_rollback_restores_state_and_refuses_too_deep():
    S, W, r, R = 4, 32, 8, 6
    p = Pair(S, W, r, 2, 128, 2, 2, "bf16", 6, max_seq_len=512, reserve=R, full_kv=True, tag="rb")
    try:
        for l in range(2):
            p.load(l, 0, 66, seed=l)
            p.load(l, 1, 100, seed=l + 9)
        q = p.rand((2, 6, 128), "qfixed")
        before = [to_np(p.draft(l, q=q)[0]) for l in range(2)]
        for step in range(1, 6):          # seq 0 crosses tau_4 = 68 at step 2
            p.step = step
            for l in range(2):
                p.append(l)
                p.draft(l)
                due = [b for b in range(2) if orc.is_boundary(p.ref.t(l, b), S, W, r)]
                if due:
                    p.materialize(l, due)
        assert p.ref.m(0, 0) == orc.slot_count(71, S, W, r)
        capi.masw_rollback(p.h, [0, 1], [66, 100])
        p.ref.rollback([0, 1], [66, 100])
        for l in range(2):
            after = to_np(p.draft(l, q=q)[0])
            assert np.array_equal(after, before[l])
            for b in range(2):
                p.check_state(l, b)
        for step in range(7):
            p.step = 100 + step
            for l in range(2):
                p.append(l)
        with pytest.raises(capi.MaswError) as ei:
            capi.masw_rollback(p.h, [0], [66])
        assert ei.value.code == capi.MASW_ESTATE
    finally:
        p.close()


@pytest.mark.parametrize("dtype,D,G", [("bf16", 128, 3), ("bf16", 64, 4), ("f32", 64, 2)])
def test_fused_step_from_empty_through_boundaries(dtype, D, G):
    """masw_draft_step (append + attention in one launch for bf16 pools) from
    t = 0: the sink phase, window growth, ring wrap with a rollback reserve,
    several boundaries with slot writes, a ragged active mask; the full-KV
    step alongside."""
    S, W, r, R, Hkv = 3, 20, 6, 4, 2
    p = Pair(S, W, r, Hkv, D, 2, 3, dtype, G * Hkv, max_seq_len=128, full_kv=True, reserve=R, tag="fstep")
    try:
        for step in range(1, 70):
            p.step = step
            active = [1, 1 if step % 3 else 0, 1 if step > 10 else 0]
            for l in range(2):
                p.fstep(l, active=active)
                due = [b for b in range(3) if orc.is_boundary(p.ref.t(l, b), S, W, r)
                       and p.ref.m(l, b) == orc.slot_count(p.ref.t(l, b), S, W, r) - 1]
                if due:
                    p.materialize(l, due)
            if step % 9 == 0:
                p.draft(0, full=True)
        for l in range(2):
            for b in range(3):
                p.check_state(l, b)
    finally:
        p.close()


@pytest.mark.parametrize("dtype,G,self_attend", [("bf16", 3, False), ("bf16", 4, False), ("bf16", 8, False),
                                                  ("f32", 2, False), ("bf16", 2, True)])
def test_fused_boundary_step(dtype, G, self_attend):
    """masw_draft_step_slot: the slot write rides in the draft step's launch
    (bf16, G <= 4) or falls back to two launches; ragged batch, some rows at a
    boundary, some not, an inactive row."""
    S, W, r, Hkv, D = 2, 24, 8, 2, 128 if dtype == "bf16" else 64
    p = Pair(S, W, r, Hkv, D, 2, 4, dtype, G * Hkv, max_seq_len=256, reserve=3, self_attend=self_attend,
             tag=f"fbnd{G}{int(self_attend)}")
    try:
        for l in range(2):
            p.load(l, 0, 40, seed=1)
            p.load(l, 1, 53, seed=2)
            p.load(l, 3, 9, seed=3)
        for step in range(1, 40):
            p.step = step
            active = [1, 1, 1 if step % 4 else 0, 1 if step > 5 else 0]
            for l in range(2):
                due = [b for b in range(4) if active[b] and orc.is_boundary(p.ref.t(l, b) + 1, S, W, r)
                       and p.ref.m(l, b) == orc.slot_count(p.ref.t(l, b) + 1, S, W, r) - 1]
                if due:
                    p.fstep_slot(l, due, active=active)
                else:
                    p.fstep(l, active=active)
        for l in range(2):
            for b in range(4):
                p.check_state(l, b)
    finally:
        p.close()


def test_fused_full_step():
    p = Pair(4, 16, 8, 2, 128, 1, 2, "bf16", 8, max_seq_len=300, full_kv=True, tag="ffull")
    try:
        p.load(0, 0, 150, seed=1)
        p.load(0, 1, 7, seed=2)
        for step in range(12):
            p.step = step
            p.fstep(0, full=True)
        p.check_state(0, 0)
        p.check_state(0, 1)
    finally:
        p.close()


@pytest.mark.parametrize("r", [4, 8])
def test_paper_configuration_many_slots(r):
    """The pages' configuration S = W = 128 with r = 4 / 8: the slot chain holds
    most of the working set (hundreds of slots); boundaries every r steps."""
    S = W = 128
    p = Pair(S, W, r, 8, 128, 1, 2, "bf16", 24, max_seq_len=1400, reserve=8, full_kv=True, tag=f"paper{r}")
    try:
        p.load(0, 0, 1200, seed=1)
        p.load(0, 1, 701, seed=2)
        assert p.ref.m(0, 0) == (1200 - 256) // r
        for step in range(1, 3 * r + 2):
            p.step = step
            due = [b for b in range(2) if orc.is_boundary(p.ref.t(0, b) + 1, S, W, r)
                   and p.ref.m(0, b) == orc.slot_count(p.ref.t(0, b) + 1, S, W, r) - 1]
            if due:
                p.fstep_slot(0, due)
            else:
                p.fstep(0)
            if step % 3 == 0:
                p.draft(0, full=True)
        p.check_state(0, 0)
        p.check_state(0, 1)
    finally:
        p.close()


@pytest.mark.parametrize("dtype,B,L,V", [("bf16", 4, 5, 128256), ("f32", 3, 5, 1000), ("bf16", 2, 0, 77),
                                         ("f32", 7, 9, 32003)])
def test_greedy_accept(dtype, B, L, V):
    """Greedy acceptance on seeded synthetic logits, bit-exact against the
    oracle: a mix of fully accepted, partly accepted and rejected blocks, ties."""
    logits = synth.normal((B, L + 1, V), dtype, "accept", B, L, V)
    lf = logits.float().numpy()
    arg = lf.argmax(-1)
    draft = arg[:, :L].copy()
    for b in range(B):
        if L and b % 3 == 1:
            draft[b, (b * 7) % L] = (arg[b, (b * 7) % L] + 1) % V
        if L and b % 3 == 2:
            draft[b, 0] = (arg[b, 0] + 5) % V
    if V > 10:   # a tie at the top of row (0, 0): the smaller id must win
        top = int(arg[0, 0])
        other = (top + 7) % V
        logits[0, 0, other] = logits[0, 0, top]
        lf = logits.float().numpy()
    want_tok, want_n = orc.greedy_accept(lf, draft)
    dl = logits.to(DEV)
    dd = torch.from_numpy(np.ascontiguousarray(draft, dtype=np.int32)).to(DEV)
    gws = Guarded((capi.masw_greedy_workspace_bytes(B, L, V),), torch.uint8)
    ws = gws.t
    gtok = Guarded((B, L + 1), torch.int32)
    gn = Guarded((B,), torch.int32)
    tok, n = gtok.t, gn.t
    for call in range(3):   # one zero-filled workspace, reused: every call leaves its tickets at zero
        tok.fill_(-7)
        n.fill_(-7)
        capi.masw_greedy_accept(dl, dd, tok, n, workspace=ws)
        torch.cuda.synchronize()
        assert np.array_equal(tok.cpu().numpy(), want_tok), call
        assert np.array_equal(n.cpu().numpy(), want_n), call
    assert not ws[-4 * B:].any()   # the per-sequence tickets (the workspace's last B words) are zero again
    for g_, name in ((gws, "workspace"), (gtok, "tokens"), (gn, "n_emit")):
        g_.check(f"greedy {name}")


@pytest.mark.parametrize("dtype,V", [("bf16", 128256), ("f32", 3001)])
def test_greedy_accept_nan_and_inf(dtype, V):
    """NaN entries are skipped, +-inf are values, an all-NaN row gives token -1
    (rejecting its draft; as the bonus row it is emitted as -1), bit-exact
    against the oracle; bf16 over many vocabulary chunks, f32 on the unaligned
    (scalar) path."""
    B, L = 3, 4
    logits = synth.normal((B, L + 1, V), dtype, "accept-nan", V).float()
    nan, inf = float("nan"), float("inf")
    x = logits
    x[0, 0, ::97] = nan                                   # NaN sprinkled over a normal row
    x[0, 0, 5] = 40.0
    x[0, 0, 3] = nan                                      # NaN before the maximum
    x[0, 1, :] = nan                                      # all NaN: no token
    x[1, 0, :] = -inf
    x[1, 0, ::3] = nan                                    # -inf and NaN only: first -inf id
    x[1, 1, V // 2] = inf
    x[1, 1, V - 1] = inf                                  # +inf tie: the smaller id
    x[1, 1, 7] = nan
    x[1, 2, :] = nan
    x[1, 2, V - 1] = -inf                                 # NaN but for one -inf at the end
    top = int(x[1, 3].argmax())
    x[1, 3, top] = nan                                    # NaN where the maximum was
    x[1, 4, :] = nan                                      # the bonus row all NaN
    logits = x.to(torch.bfloat16) if dtype == "bf16" else x
    lf = logits.float().numpy()
    want_tok, _ = orc.greedy_accept(lf, np.zeros((B, L), dtype=np.int64))
    draft = np.array(want_tok[:, :L], dtype=np.int64)
    draft[0, 1] = 11                                      # row (0, 1) has no token: rejected anyway
    draft[2, 2] = (want_tok[2, 2] + 1) % V                # an ordinary rejection
    want_tok, want_n = orc.greedy_accept(lf, draft)
    assert want_tok[0, 1] == -1 and want_tok[1, 4] == -1 and want_tok[1, 0] == 1
    assert list(want_n) == [2, L + 1, 3]
    dl = logits.contiguous().to(DEV)
    dd = torch.from_numpy(np.ascontiguousarray(draft, dtype=np.int32)).to(DEV)
    tok = torch.full((B, L + 1), -7, dtype=torch.int32, device=DEV)
    n = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    ws = torch.zeros(capi.masw_greedy_workspace_bytes(B, L, V), dtype=torch.uint8, device=DEV)
    for call in range(2):
        capi.masw_greedy_accept(dl, dd, tok, n, workspace=ws)
        torch.cuda.synchronize()
        assert np.array_equal(tok.cpu().numpy(), want_tok), call
        assert np.array_equal(n.cpu().numpy(), want_n), call


def test_allocation_limit_frees_what_create_had_allocated(monkeypatch):
    """With MASW_DEVICE_MEMORY_LIMIT above the pools' size but below the full-KV
    cache, create allocates the two pools, is refused the cache, returns
    MASW_ENOMEM and frees the pools: device free memory is unchanged."""
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info(DEV)[0]
    monkeypatch.setenv("MASW_DEVICE_MEMORY_LIMIT", str(200 << 20))   # pools: ~143 MB; cache: ~4.3 GB
    with pytest.raises(capi.MaswError) as ei:
        capi.masw_mem_create(4, 1024, 512, 8, 128, 4, batch=8, dtype=capi.MASW_BF16, max_seq_len=32768,
                             full_kv=True)
    assert ei.value.code == capi.MASW_ENOMEM
    torch.cuda.synchronize()
    assert abs(torch.cuda.mem_get_info(DEV)[0] - free0) < (8 << 20)
    monkeypatch.delenv("MASW_DEVICE_MEMORY_LIMIT")
    h = capi.masw_mem_create(4, 1024, 512, 8, 128, 4, batch=8, dtype=capi.MASW_BF16, max_seq_len=32768)
    capi.masw_check_guards(h)
    capi.masw_mem_destroy(h)


def test_state_errors():
    p = Pair(2, 8, 4, 2, 64, 1, 1, "f32", 4, max_seq_len=18, tag="err")
    try:
        p.load(0, 0, 13, seed=0)          # m(13) = 0; tau_1 = 14
        qg = torch.zeros(1, 4, 64, device=DEV)
        kg = torch.zeros(1, 2, 64, device=DEV)
        og = torch.empty(1, 4, 64, device=DEV)
        with pytest.raises(capi.MaswError) as ei:
            capi.masw_materialize_slot(p.h, 0, [0], qg, kg, kg, og)
        assert ei.value.code == capi.MASW_ESTATE
        with pytest.raises(capi.MaswError) as ei:
            capi.masw_full_attn(p.h, 0, qg, og)
        assert ei.value.code == capi.MASW_ESTATE
        with pytest.raises(capi.MaswError) as ei:
            capi.masw_draft_attn(p.h, 0, torch.zeros(1, 10, 64, device=DEV), torch.empty(1, 10, 64, device=DEV))
        assert ei.value.code == capi.MASW_EINVAL
        for step in range(5):
            p.step = step
            p.append(0)
        with pytest.raises(capi.MaswError) as ei:
            p.append(0)
        assert ei.value.code == capi.MASW_ECAPACITY
        with pytest.raises(capi.MaswError) as ei:
            capi.masw_draft_attn(p.h, 1, qg, og)
        assert ei.value.code == capi.MASW_EINVAL
        capi.masw_sync(p.h)
    finally:
        p.close()


def _verify_case(B, Lq, Hq, Hkv, Tmax, kv_len, seed, scale=0.0, qscale=1.0):
    D = 128
    q = synth.normal((B, Lq, Hq, D), "bf16", "verify", seed, "q", scale=qscale)
    k = synth.normal((B, Hkv, Tmax, D), "bf16", "verify", seed, "k")
    v = synth.normal((B, Hkv, Tmax, D), "bf16", "verify", seed, "v")
    kl = torch.tensor(kv_len, dtype=torch.int32)
    o = torch.empty(B, Lq, Hq, D, device=DEV)
    lse = torch.empty(B, Lq, Hq, device=DEV)
    capi.masw_verify_attn(q.to(DEV), k.to(DEV), v.to(DEV), kl.to(DEV), o, lse, scale=scale)
    torch.cuda.synchronize()
    want, want_l = orc.verify_attn(q.float().numpy(), k.float().numpy(), v.float().numpy(), kv_len, scale or None)
    assert_close(o, want, "bf16", f"verify O {B}x{Lq}x{Hq}/{Hkv}")
    assert_close(lse, want_l, "bf16", "verify LSE")


@pytest.mark.parametrize("B,Lq,Hq,Hkv,Tmax,kv_len", [
    (2, 6, 32, 8, 700, [700, 333]),       # 8B-target shape, ragged, several splits
    (1, 5, 24, 8, 97, [64]),              # NQ = 15: padded N tile
    (3, 1, 8, 8, 300, [1, 17, 300]),      # G = 1, Lq = 1: plain decode; a 1-key cache
    (1, 8, 32, 8, 4096, [4000]),          # NQ = 32: the largest block
])
def test_verify_against_oracle(B, Lq, Hq, Hkv, Tmax, kv_len):
    _verify_case(B, Lq, Hq, Hkv, Tmax, kv_len, seed=B * 100 + Lq)


def test_verify_workspace_reuse_leaves_tickets_zero():
    """A zero-filled workspace is reused across calls with no memset between
    them: every call leaves its (sequence, kv head) tickets at zero, and the
    results of each call match the oracle."""
    B, Lq, Hq, Hkv, Tmax, D = 2, 6, 32, 8, 1500, 128
    need = capi.masw_verify_workspace_bytes(B, Lq, Hq, Hkv, D, Tmax)
    gws = Guarded((need,), torch.uint8)          # zero-filled, with guard bands on both sides
    ws = gws.t
    for call, kv_len in enumerate([[1500, 900], [1200, 1500], [64, 700]]):
        seed = 900 + call
        q = synth.normal((B, Lq, Hq, D), "bf16", "verify", seed, "q")
        k = synth.normal((B, Hkv, Tmax, D), "bf16", "verify", seed, "k")
        v = synth.normal((B, Hkv, Tmax, D), "bf16", "verify", seed, "v")
        kl = torch.tensor(kv_len, dtype=torch.int32)
        go = Guarded((B, Lq, Hq, D), torch.float32)
        gl = Guarded((B, Lq, Hq), torch.float32)
        capi.masw_verify_attn(q.to(DEV), k.to(DEV), v.to(DEV), kl.to(DEV), go.t, gl.t, workspace=ws)
        torch.cuda.synchronize()
        want, want_l = orc.verify_attn(q.float().numpy(), k.float().numpy(), v.float().numpy(), kv_len, None)
        assert_close(go.t, want, "bf16", f"verify call {call}")
        assert_close(gl.t, want_l, "bf16", f"verify LSE call {call}")
        tail = ws[need - 16 - B * Hkv * 4:].view(torch.int32)   # tickets, then the status word
        assert int(tail.abs().sum()) == 0, f"call {call} left tickets/status {tail.tolist()}"
        for g_, name in ((gws, "workspace"), (go, "O"), (gl, "LSE")):
            g_.check(f"verify call {call} {name}")


def test_verify_peaky_softmax_and_scale():
    _verify_case(2, 6, 32, 8, 512, [512, 200], seed=7, qscale=4.0)
    _verify_case(1, 6, 32, 8, 256, [250], seed=8, scale=0.2)


@pytest.mark.slow
def test_verify_full_size():
    """8B-target verify at full size: B=4, Lq=6, 32q/8kv, 32768 + 6 keys."""
    T = 32768 + 6
    _verify_case(4, 6, 32, 8, T, [T] * 4, seed=3)


@pytest.mark.slow
def test_draft3b_full_size_sampled():
    """The benchmark's launch shape: batch 8, 24q/8kv, 32K prefix (61 slots),
    S=4, W=1024, r=512.  Two sequences of the batch carry CPU-seeded data and
    are checked against the oracle; the rest are filled on the device.  The
    launch grid and split count depend on batch, heads and working-set length,
    not on the number of layers, so two layers stand for 28."""
    S, W, r, t0 = 4, 1024, 512, 32768
    B, L, Hkv, D, Hq = 8, 2, 8, 128, 24
    p = Pair(S, W, r, Hkv, D, L, B, "bf16", Hq, max_seq_len=t0 + 16, full_kv=True, tag="cfg3")
    sampled = {(0, 3), (1, 7)}
    try:
        g = torch.Generator(device=DEV)
        g.manual_seed(1234)
        n = orc.slot_count(t0, S, W, r)
        for l in range(L):
            for b in range(B):
                if (l, b) in sampled:
                    p.load(l, b, t0, seed=2)
                else:                               # unchecked rows: device-filled, K != V
                    kr = torch.randn(t0, Hkv, D, generator=g, device=DEV).to(torch.bfloat16)
                    vr = torch.randn(t0, Hkv, D, generator=g, device=DEV).to(torch.bfloat16)
                    ks = torch.randn(n, Hkv, D, generator=g, device=DEV).to(torch.bfloat16)
                    vs = torch.randn(n, Hkv, D, generator=g, device=DEV).to(torch.bfloat16)
                    capi.masw_mem_load(p.h, l, b, kr, vr, ks, vs)
                    del kr, vr, ks, vs
        for step in range(1, 6):
            p.step = step
            for l in range(L):
                k = p.rand((B, Hkv, D), "k", l)
                v = p.rand((B, Hkv, D), "v", l)
                capi.masw_append_kv(p.h, l, k.to(DEV), v.to(DEV))
                q = p.rand((B, Hq, D), "q", l)
                o = torch.empty(B, Hq, D, device=DEV)
                lse = torch.empty(B, Hq, device=DEV)
                capi.masw_draft_attn(p.h, l, q.to(DEV), o, lse)
                of = torch.empty(B, Hq, D, device=DEV)
                capi.masw_full_attn(p.h, l, q.to(DEV), of)
                for (sl, sb) in sampled:
                    if sl != l:
                        continue
                    p.ref.append(l, k.float().numpy(), v.float().numpy(),
                                 active=[bb == sb for bb in range(B)])
                    qb = q.float().numpy()[sb:sb + 1]
                    Kc, Vc = p.ref._columns(l, sb)
                    mask = orc.draft_mask(p.ref.t(l, sb), p.ref.m(l, sb), S, W)
                    wo, wl = orc.attention(qb[0], Kc, Vc, mask, p.ref.scale)
                    assert_close(o[sb], wo, "bf16", f"cfg3 draft l={l} b={sb} step={step}")
                    assert_close(lse[sb], wl, "bf16", "cfg3 draft LSE")
                    fo, _ = orc.attention(qb[0], p.ref.raw_k[l][sb], p.ref.raw_v[l][sb],
                                          orc.full_mask(p.ref.t(l, sb)), p.ref.scale)
                    assert_close(of[sb], fo, "bf16", f"cfg3 full l={l} b={sb}")
                if step == 4:       # tau_62 = 4 + 1024 + 62*512 = 32772 for every sequence
                    assert orc.is_boundary(t0 + 4, S, W, r)
                    qg = p.rand((B, Hq, D), "qg", l)
                    kg = p.rand((B, Hkv, D), "kg", l)
                    vg = p.rand((B, Hkv, D), "vg", l)
                    og = torch.empty(B, Hq, D, device=DEV)
                    capi.masw_materialize_slot(p.h, l, list(range(B)), qg.to(DEV), kg.to(DEV), vg.to(DEV), og)
                    for (sl, sb) in sampled:
                        if sl != l:
                            continue
                        w, _ = p.ref.materialize_slot(l, [sb], qg.float().numpy()[sb:sb + 1],
                                                      kg.float().numpy()[sb:sb + 1], vg.float().numpy()[sb:sb + 1])
                        assert_close(og[sb:sb + 1], w, "bf16", f"cfg3 slot l={l} b={sb}")
        capi.masw_sync(p.h)
        for (sl, sb) in sampled:
            p.check_state(sl, sb)
    finally:
        p.close()


@pytest.mark.slow
@pytest.mark.parametrize("prefix", [4096, 8192, 16384, 24576, 32768])
def test_config3_every_pair_at_each_prefix(prefix):
    """The 28-layer, batch-8 sweep's launch shape (24q/8kv heads, S=4, W=1024,
    r=512) at every prefix of the sweep, 4K..32K, whose working sets (1033 to
    1089 keys) give different split and cluster plans.  Two layers stand for 28
    (the grid does not depend on the layer count).  Every (layer, row) pair
    carries CPU-seeded data; the five fused steps of the benchmark's iteration
    run in its order (the boundary tau = prefix + 4 is crossed at step 4 by
    every sequence, so step 4 is the fused boundary step with all eight slot
    queries), and at steps 4 and 5 every pair's draft output, and at step 4
    every slot output, is compared with the oracle; then every pair's memory is
    checked row by row."""
    S, W, r, t0 = 4, 1024, 512, prefix
    B, L, Hkv, D, Hq = 8, 2, 8, 128, 24
    assert orc.is_boundary(t0 + 4, S, W, r)
    p = Pair(S, W, r, Hkv, D, L, B, "bf16", Hq, max_seq_len=t0 + 16, reserve=16, tag=f"cfg3_{prefix}")
    try:
        for l in range(L):
            for b in range(B):
                p.load(l, b, t0, seed=5)
        for step in range(1, 6):
            p.step = step
            for l in range(L):
                if step == 4:
                    p.fstep_slot(l, list(range(B)))
                else:
                    p.fstep(l, check=step == 5)
        capi.masw_sync(p.h)
        for l in range(L):
            for b in range(B):
                assert p.ref.m(l, b) == orc.slot_count(t0 + 5, S, W, r)
                p.check_state(l, b)
    finally:
        p.close()


@pytest.mark.slow
def test_swa_special_case_full_size():
    """Sliding-window attention, the pages' SWA baseline, as a special case of
    the memory: S = 0, no slots (r beyond the longest sequence), W = 1024, on
    the 3B-draft launch shape (batch 8, 24q/8kv, 32K prefix, ring reserve 16).
    Every (layer, row) pair carries CPU-seeded data; five fused steps, every
    pair's output compared with the oracle at the first and last step, and every
    pair's memory checked row by row (no slot is ever written)."""
    S, W, r, t0 = 0, 1024, 1 << 20, 32768
    B, L, Hkv, D, Hq = 8, 2, 8, 128, 24
    p = Pair(S, W, r, Hkv, D, L, B, "bf16", Hq, max_seq_len=t0 + 16, reserve=16, tag="swa")
    try:
        for l in range(L):
            for b in range(B):
                p.load(l, b, t0, seed=6)
        for step in range(1, 6):
            p.step = step
            for l in range(L):
                p.fstep(l, check=step in (1, 5))
        capi.masw_sync(p.h)
        for l in range(L):
            for b in range(B):
                assert p.ref.m(l, b) == 0 and orc.working_set_size(t0 + 5, S, W, r) == W
                p.check_state(l, b)
    finally:
        p.close()


@pytest.mark.parametrize("Hq,B", [(24, 8), (32, 8), (24, 4), (32, 4), (32, 2)])
def test_fused_steps_full_size_sampled(Hq, B):
    """The fused step and the fused boundary step at the benchmark's launch
    shape (batch 8, 8 kv heads, 32K prefix, S=4, W=1024, r=512) and at batch 4
    and 2: every split of a (row, head) pair is a CTA of one thread-block
    cluster (6, 10 and 12 CTAs; with 10 the last rank finalises a shorter slice
    of the output), so the shared-memory merge runs with G = 3 or 4 query
    columns per pair, and with 2G = 6 or 8 at the boundary step, where the slot
    queries of all sequences ride in the same launch.  The new token's row is
    stored by the split whose keys include it.  Two (layer, row) pairs carry
    CPU-seeded data and are checked against the oracle; the other rows are
    filled on the device."""
    S, W, r, t0 = 4, 1024, 512, 32768
    L, Hkv, D = 2, 8, 128
    p = Pair(S, W, r, Hkv, D, L, B, "bf16", Hq, max_seq_len=t0 + 16, tag=f"fsz{Hq}_{B}")
    sampled = {(0, B // 4), (1, B - 2)}
    try:
        g = torch.Generator(device=DEV)
        g.manual_seed(4321)
        n = orc.slot_count(t0, S, W, r)
        for l in range(L):
            for b in range(B):
                if (l, b) in sampled:
                    p.load(l, b, t0, seed=3)
                else:                               # unchecked rows: device-filled, K != V
                    kr = torch.randn(t0, Hkv, D, generator=g, device=DEV).to(torch.bfloat16)
                    vr = torch.randn(t0, Hkv, D, generator=g, device=DEV).to(torch.bfloat16)
                    ks = torch.randn(n, Hkv, D, generator=g, device=DEV).to(torch.bfloat16)
                    vs = torch.randn(n, Hkv, D, generator=g, device=DEV).to(torch.bfloat16)
                    capi.masw_mem_load(p.h, l, b, kr, vr, ks, vs)
                    del kr, vr, ks, vs
        for step in range(1, 7):
            p.step = step
            boundary = step == 4          # tau_62 = 4 + 1024 + 62*512 = 32772 for every sequence
            for l in range(L):
                k = p.rand((B, Hkv, D), "k", l)
                v = p.rand((B, Hkv, D), "v", l)
                q = p.rand((B, Hq, D), "q", l)
                o = torch.empty(B, Hq, D, device=DEV)
                lse = torch.empty(B, Hq, device=DEV)
                if boundary:
                    assert orc.is_boundary(t0 + 4, S, W, r)
                    qg = p.rand((B, Hq, D), "qg", l)
                    kg = p.rand((B, Hkv, D), "kg", l)
                    vg = p.rand((B, Hkv, D), "vg", l)
                    og = torch.empty(B, Hq, D, device=DEV)
                    lg = torch.empty(B, Hq, device=DEV)
                    capi.masw_draft_step_slot(p.h, l, q.to(DEV), k.to(DEV), v.to(DEV), o, list(range(B)),
                                              qg.to(DEV), kg.to(DEV), vg.to(DEV), og, lse, lg)
                else:
                    capi.masw_draft_step(p.h, l, q.to(DEV), k.to(DEV), v.to(DEV), o, lse)
                for (sl, sb) in sampled:
                    if sl != l:
                        continue
                    p.ref.append(l, k.float().numpy(), v.float().numpy(), active=[bb == sb for bb in range(B)])
                    Kc, Vc = p.ref._columns(l, sb)
                    mask = orc.draft_mask(p.ref.t(l, sb), p.ref.m(l, sb), S, W)
                    wo, wl = orc.attention(q.float().numpy()[sb], Kc, Vc, mask, p.ref.scale)
                    assert_close(o[sb], wo, "bf16", f"fused step Hq={Hq} l={l} b={sb} step={step}")
                    assert_close(lse[sb], wl, "bf16", "fused step LSE")
                    if boundary:
                        w, wlg = p.ref.materialize_slot(l, [sb], qg.float().numpy()[sb:sb + 1],
                                                        kg.float().numpy()[sb:sb + 1], vg.float().numpy()[sb:sb + 1])
                        assert_close(og[sb:sb + 1], w, "bf16", f"fused slot Hq={Hq} l={l} b={sb}")
                        assert_close(lg[sb:sb + 1], wlg, "bf16", "fused slot LSE")
        capi.masw_sync(p.h)
        for (sl, sb) in sampled:
            p.check_state(sl, sb)
    finally:
        p.close()


@pytest.mark.parametrize("Hq", [24, 32])
def test_fused_steps_one_sequence(Hq):
    """One sequence (8 kv heads, 8K prefix, S=4, W=1024, r=512): each (sequence,
    head) pair runs as a cluster of 12 CTAs merging in shared memory; fused
    steps, and at tau_14 = 8196 the fused boundary step (2G = 6 or 8 query
    columns per pair), across two layers, all rows checked against the oracle."""
    S, W, r, t0 = 4, 1024, 512, 8192
    B, L, Hkv, D = 1, 2, 8, 128
    p = Pair(S, W, r, Hkv, D, L, B, "bf16", Hq, max_seq_len=t0 + 16, tag=f"fs1_{Hq}")
    try:
        for l in range(L):
            p.load(l, 0, t0, seed=4 + l)
        for step in range(1, 7):
            p.step = step
            for l in range(L):
                if orc.is_boundary(p.ref.t(l, 0) + 1, S, W, r):
                    p.fstep_slot(l, [0])
                else:
                    p.fstep(l)
        for l in range(L):
            p.check_state(l, 0)
            assert p.ref.m(l, 0) == 14
    finally:
        p.close()


def test_draft8b_large_batch_every_sequence():
    """The large-batch launch shape (batch 32, 32q/8kv, W = 2048, r = 1024,
    ragged prefixes 16K..32K, each snapped down as the benchmark does so that
    sequence b reaches its compression boundary at draft step b mod 8 + 1): one
    split per (sequence, head) streams ~2080 keys, which selects the three-stage
    kernel.  Eight fused steps with per-sequence slot writes.  Every sequence
    carries CPU-seeded data; every sequence's draft output and slot output at
    its boundary step, and every draft output at the last step, are compared
    with the oracle's mask and attention over that sequence's columns (kept
    here in preallocated arrays, so the 32 histories are not re-copied at each
    append); two sequences' memories are also checked row by row."""
    S, W, r, steps = 4, 2048, 1024, 8
    B, Hkv, D, G = 32, 8, 128, 4
    Hq = Hkv * G
    prefixes = []
    for b, p0 in enumerate(synth.ragged_prefixes(B, 16384, 32768, "long-runs")):
        t = p0
        while not orc.is_boundary(t + b % steps + 1, S, W, r):
            t -= 1
        prefixes.append(t)
    tracked = [5, 17]
    p = Pair(S, W, r, Hkv, D, 1, B, "bf16", Hq, max_seq_len=32768 + 64, reserve=16, tag="cfg5all")
    try:
        raw_k, raw_v, slot_k, slot_v, t_of, m_of = [], [], [], [], [], []
        for b in range(B):
            t = prefixes[b]
            n = orc.slot_count(t, S, W, r)
            kr, vr = (synth.normal((t, Hkv, D), "bf16", p.tag, nm, b) for nm in ("k", "v"))
            ks, vs = (synth.normal((n, Hkv, D), "bf16", p.tag, nm, b) for nm in ("ks", "vs"))
            capi.masw_mem_load(p.h, 0, b, kr, vr, ks if n else None, vs if n else None)
            rk, rv = np.zeros((t + steps, Hkv, D), np.float32), np.zeros((t + steps, Hkv, D), np.float32)
            rk[:t], rv[:t] = kr.float().numpy(), vr.float().numpy()
            sk, sv = np.zeros((n + 1, Hkv, D), np.float32), np.zeros((n + 1, Hkv, D), np.float32)
            sk[:n], sv[:n] = ks.float().numpy(), vs.float().numpy()
            raw_k.append(rk), raw_v.append(rv), slot_k.append(sk), slot_v.append(sv)
            t_of.append(t), m_of.append(n)
            if b in tracked:
                p.ref.load(0, b, rk[:t], rv[:t], sk[:n], sv[:n])
            del kr, vr, ks, vs

        def columns(b, t, m):
            return (np.concatenate([raw_k[b][:t], slot_k[b][:m]]), np.concatenate([raw_v[b][:t], slot_v[b][:m]]))

        checked_slots = 0
        for step in range(steps):
            p.step = step
            due = [b for b in range(B) if orc.is_boundary(t_of[b] + 1, S, W, r)]
            assert due == [b for b in range(B) if b % steps == step]
            k, v, q = p.rand((B, Hkv, D), "k"), p.rand((B, Hkv, D), "v"), p.rand((B, Hq, D), "q")
            o = torch.empty(B, Hq, D, device=DEV)
            lse = torch.empty(B, Hq, device=DEV)
            n = len(due)
            qg, kg, vg = p.rand((n, Hq, D), "qg"), p.rand((n, Hkv, D), "kg"), p.rand((n, Hkv, D), "vg")
            og = torch.empty(n, Hq, D, device=DEV)
            lg = torch.empty(n, Hq, device=DEV)
            capi.masw_draft_step_slot(p.h, 0, q.to(DEV), k.to(DEV), v.to(DEV), o, due, qg.to(DEV), kg.to(DEV),
                                      vg.to(DEV), og, lse, lg)
            capi.masw_sync(p.h)
            kf, vf, qf = k.float().numpy(), v.float().numpy(), q.float().numpy()
            qgf, kgf, vgf = qg.float().numpy(), kg.float().numpy(), vg.float().numpy()
            for b in range(B):
                raw_k[b][t_of[b]], raw_v[b][t_of[b]] = kf[b], vf[b]
                t_of[b] += 1
            p.ref.append(0, kf, vf, active=[b in tracked for b in range(B)])
            for b in sorted(set(due) | (set(range(B)) if step == steps - 1 else set())):
                Kc, Vc = columns(b, t_of[b], m_of[b])
                wo, wl = orc.attention(qf[b], Kc, Vc, orc.draft_mask(t_of[b], m_of[b], S, W), p.ref.scale)
                assert_close(o[b], wo, "bf16", f"cfg5 draft b={b} step={step}")
                assert_close(lse[b], wl, "bf16", f"cfg5 draft LSE b={b} step={step}")
            for i, b in enumerate(due):
                tau, m = t_of[b], m_of[b] + 1
                slot_k[b][m - 1], slot_v[b][m - 1] = kgf[i], vgf[i]
                m_of[b] = m
                Kc, Vc = columns(b, tau, m)
                wo, wl = orc.attention(qgf[i], Kc, Vc, orc.slot_write_mask(tau, m, S, W), p.ref.scale)
                assert_close(og[i], wo, "bf16", f"cfg5 slot b={b} step={step}")
                assert_close(lg[i], wl, "bf16", f"cfg5 slot LSE b={b} step={step}")
                checked_slots += 1
                if b in tracked:
                    p.ref.materialize_slot(0, [b], qgf[i:i + 1], kgf[i:i + 1], vgf[i:i + 1])
        assert checked_slots == B
        assert all(m_of[b] == orc.slot_count(prefixes[b] + steps, S, W, r) for b in range(B))
        for b in tracked:
            p.check_state(0, b)
    finally:
        p.close()


def test_graph_replay_matches_eager():
    """A captured speculative iteration (appends, draft attention, a slot
    write at the boundary, rollback) replays with the same results: the
    counters live on the device, so the graph's net effect is identity."""
    S, W, r, R = 4, 64, 16, 8
    B, L, Hq, Hkv, D = 2, 2, 6, 2, 128
    p = Pair(S, W, r, Hkv, D, L, B, "bf16", Hq, max_seq_len=1024, reserve=R, tag="graph")
    try:
        t0 = S + W + 5 * r - 2     # boundary after 2 appends
        for l in range(L):
            for b in range(B):
                p.load(l, b, t0, seed=l * 10 + b)
        steps = 4
        ks = [[p.rand((B, Hkv, D), "k", s, l).to(DEV) for l in range(L)] for s in range(steps)]
        vs = [[p.rand((B, Hkv, D), "v", s, l).to(DEV) for l in range(L)] for s in range(steps)]
        qs = [[p.rand((B, Hq, D), "q", s, l).to(DEV) for l in range(L)] for s in range(steps)]
        qg = p.rand((B, Hq, D), "qg").to(DEV)
        kg = p.rand((B, Hkv, D), "kg").to(DEV)
        outs = [[torch.empty(B, Hq, D, device=DEV) for _ in range(L)] for _ in range(steps)]
        og = torch.empty(B, Hq, D, device=DEV)

        def iteration():
            for s in range(steps):
                for l in range(L):
                    capi.masw_append_kv(p.h, l, ks[s][l], vs[s][l])
                    capi.masw_draft_attn(p.h, l, qs[s][l], outs[s][l])
                    if s == 1:
                        capi.masw_materialize_slot(p.h, l, list(range(B)), qg, kg, kg, og)
            capi.masw_rollback(p.h, list(range(B)), [t0] * B)

        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            iteration()
        torch.cuda.synchronize()
        eager = [[o.clone() for o in row] for row in outs]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            iteration()
        for _ in range(3):
            for row in outs:
                for o in row:
                    o.zero_()
            graph.replay()
            torch.cuda.synchronize()
            for s in range(steps):
                for l in range(L):
                    assert torch.equal(outs[s][l], eager[s][l])
        capi.masw_sync(p.h)
        st = capi.masw_query(p.h, 0, 0)
        assert st["dev_t"] == st["t"] == t0 and st["dev_m"] == st["m"] == orc.slot_count(t0, S, W, r)
    finally:
        p.close()


@pytest.mark.parametrize("D,G", [(128, 3), (64, 4)])
def test_graph_replays_from_a_later_state_rebuild_the_segment_table(D, G):
    """A captured fused step replayed without a rollback: every replay after the
    first starts from a state the launches were not captured in, so the
    speculative segment table each CTA builds from the counters known at
    capture is wrong; the kernel must find that out from the device counters,
    rebuild the table and run its loop again.  Outputs are checked against the
    oracle at every replay, and the device counters advance by one per replay."""
    S, W, r, Hkv = 4, 64, 16, 2
    B, L, Hq = 2, 2, Hkv * G
    p = Pair(S, W, r, Hkv, D, L, B, "bf16", Hq, max_seq_len=1024, tag=f"replay{D}")
    try:
        t0 = S + W + 3 * r + 1       # the next boundary is 15 tokens away
        for l in range(L):
            for b in range(B):
                p.load(l, b, t0, seed=l * 10 + b)
        k = [p.rand((B, Hkv, D), "k", l) for l in range(L)]
        v = [p.rand((B, Hkv, D), "v", l) for l in range(L)]
        q = [p.rand((B, Hq, D), "q", l) for l in range(L)]
        kd, vd, qd = ([x.to(DEV) for x in xs] for xs in (k, v, q))
        outs = [torch.empty(B, Hq, D, device=DEV) for _ in range(L)]

        def step():
            for l in range(L):
                capi.masw_draft_step(p.h, l, qd[l], kd[l], vd[l], outs[l])

        def oracle_step(what):
            for l in range(L):
                p.ref.append(l, k[l].float().numpy(), v[l].float().numpy())
                want, _ = p.ref.draft_attn(l, q[l].float().numpy())
                assert_close(outs[l], want, "bf16", f"{what} l={l}")

        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            step()                   # eager: kernels configured, state t0 + 1
        torch.cuda.synchronize()
        oracle_step("eager")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()                   # captured from the host's view of state t0 + 1
        for rep in range(4):
            for o in outs:
                o.zero_()
            graph.replay()
            torch.cuda.synchronize()
            oracle_step(f"replay {rep}")
            st = capi.masw_query(p.h, 0, 0)
            assert st["dev_t"] == t0 + 2 + rep and st["dev_m"] == orc.slot_count(t0 + 2 + rep, S, W, r)
        capi.masw_sync(p.h)
    finally:
        p.close()


def test_bounded_wait_timeout_is_reported_and_the_context_survives():
    """Failure detection without a fault: a bounded wait on a barrier nothing
    arrives on runs out, masw_sync reports MASW_ETIMEOUT (once), and the same
    handle keeps working afterwards."""
    p = Pair(4, 16, 4, 2, 64, 1, 1, "f32", 8, max_seq_len=64, tag="timeout")
    try:
        p.load(0, 0, 30, seed=1)
        capi.masw_selftest_timeout(p.h, polls=1000)
        with pytest.raises(capi.MaswError) as ei:
            capi.masw_sync(p.h)
        assert ei.value.code == capi.MASW_ETIMEOUT
        capi.masw_sync(p.h)          # reported once, then cleared
        p.step = 0
        p.append(0)
        p.draft(0)                   # attention still matches the oracle
        p.check_state(0, 0)
    finally:
        p.close()
