"""Shared helpers for the GPU parity tests: seeded state set-up mirrored into the
CPU oracle, and the tolerance checks."""
from __future__ import annotations

import numpy as np
import torch

import oracle.masw_oracle as orc
from compressed_draft_kv_gb300 import capi, synth

DEV = torch.device("cuda:0")

# fp32 inputs: both sides are exact up to fp32 summation order
F32_ATOL = 2e-5
# bf16 inputs, fp32 accumulation (the stated tolerance for this path)
BF16_ATOL = 1e-2
BF16_REL_L2 = 5e-3


def to_np(x: torch.Tensor) -> np.ndarray:
    return x.detach().to("cpu", torch.float64).numpy()


def assert_close(got, want, dtype: str, what: str = ""):
    got = to_np(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: non-finite pattern differs"
    err = np.abs(got[fin] - want[fin])
    max_abs = float(err.max()) if err.size else 0.0
    if dtype == "f32":
        assert max_abs <= F32_ATOL, f"{what}: max abs {max_abs:.3e} > {F32_ATOL}"
    else:
        rel = float(np.linalg.norm(got[fin] - want[fin]) / max(np.linalg.norm(want[fin]), 1e-30))
        assert max_abs <= BF16_ATOL, f"{what}: max abs {max_abs:.3e} > {BF16_ATOL}"
        assert rel <= BF16_REL_L2, f"{what}: rel L2 {rel:.3e} > {BF16_REL_L2}"
    return max_abs


class Pair:
    """A libmasw pool and the oracle fed the same seeded inputs."""

    def __init__(self, S, W, r, Hkv, D, layers, batch, dtype, Hq, max_seq_len, full_kv=False,
                 reserve=0, self_attend=False, scale=0.0, tag="pair"):
        self.S, self.W, self.r, self.Hkv, self.D = S, W, r, Hkv, D
        self.layers, self.batch, self.dtype, self.Hq = layers, batch, dtype, Hq
        self.tag = tag
        self.h = capi.masw_mem_create(S, W, r, Hkv, D, layers, batch=batch,
                                      dtype=capi.MASW_BF16 if dtype == "bf16" else capi.MASW_F32,
                                      max_seq_len=max_seq_len, full_kv=full_kv, rollback_reserve=reserve,
                                      slot_self_attend=self_attend, softmax_scale=scale)
        self.ref = orc.MaswOracle(S, W, r, Hkv, D, layers, batch, scale=scale or None,
                                  slot_self_attend=self_attend, reserve=reserve)
        self.step = 0

    def close(self):
        if self.h:
            try:
                capi.masw_sync(self.h)           # no device-side error (segment tables in bounds, ...)
                capi.masw_check_guards(self.h)   # no kernel wrote outside a handle-owned buffer
            finally:
                capi.masw_mem_destroy(self.h)
                self.h = None

    def load(self, layer, seq, t, seed=0):
        n = orc.slot_count(t, self.S, self.W, self.r)
        kr = synth.normal((t, self.Hkv, self.D), self.dtype, self.tag, seed, "k", layer, seq)
        vr = synth.normal((t, self.Hkv, self.D), self.dtype, self.tag, seed, "v", layer, seq)
        ks = synth.normal((n, self.Hkv, self.D), self.dtype, self.tag, seed, "ks", layer, seq)
        vs = synth.normal((n, self.Hkv, self.D), self.dtype, self.tag, seed, "vs", layer, seq)
        capi.masw_mem_load(self.h, layer, seq, kr, vr, ks if n else None, vs if n else None)
        self.ref.load(layer, seq, kr.float().numpy(), vr.float().numpy(), ks.float().numpy(), vs.float().numpy())

    def prefill(self, layer, seq, t, seed=0):
        """masw_prefill of a t-token prefix; checks O/LSE of every raw and slot
        row against the oracle's prefill and mirrors the resulting memory into it."""
        n = orc.slot_count(t, self.S, self.W, self.r)
        g = lambda shape, name: synth.normal(shape, self.dtype, self.tag, "prefill", seed, name, layer, seq)
        qr, kr, vr = g((t, self.Hq, self.D), "q"), g((t, self.Hkv, self.D), "k"), g((t, self.Hkv, self.D), "v")
        qs, ks, vs = g((n, self.Hq, self.D), "qs"), g((n, self.Hkv, self.D), "ks"), g((n, self.Hkv, self.D), "vs")
        o_r = torch.empty(t, self.Hq, self.D, device=DEV)
        l_r = torch.empty(t, self.Hq, device=DEV)
        o_s = torch.empty(max(n, 1), self.Hq, self.D, device=DEV)
        l_s = torch.empty(max(n, 1), self.Hq, device=DEV)
        dev = [x.to(DEV) if x.numel() else None for x in (qr, kr, vr, qs, ks, vs)]
        capi.masw_prefill(self.h, layer, seq, *dev, o_r, l_r, o_s if n else None, l_s if n else None)
        want = orc.prefill_attn(self.S, self.W, self.r, qr.float().numpy(), kr.float().numpy(), vr.float().numpy(),
                                qs.float().numpy(), ks.float().numpy(), vs.float().numpy(),
                                scale=self.ref.scale, self_attend=self.ref.self_attend)
        capi.masw_sync(self.h)
        assert_close(o_r, want[0], self.dtype, f"prefill O_raw l={layer} b={seq}")
        assert_close(l_r, want[1], self.dtype, "prefill LSE_raw")
        if n:
            assert_close(o_s[:n], want[2], self.dtype, f"prefill O_slot l={layer} b={seq}")
            assert_close(l_s[:n], want[3], self.dtype, "prefill LSE_slot")
        self.ref.load(layer, seq, kr.float().numpy(), vr.float().numpy(), ks.float().numpy(), vs.float().numpy())

    def rand(self, shape, *name, scale=1.0):
        return synth.normal(shape, self.dtype, self.tag, "io", self.step, *name, scale=scale)

    def append(self, layer, active=None):
        k = self.rand((self.batch, self.Hkv, self.D), "k", layer)
        v = self.rand((self.batch, self.Hkv, self.D), "v", layer)
        capi.masw_append_kv(self.h, layer, k.to(DEV), v.to(DEV), active=active)
        self.ref.append(layer, k.float().numpy(), v.float().numpy(), active=active)

    def draft(self, layer, q=None, check=True, full=False):
        if q is None:
            q = self.rand((self.batch, self.Hq, self.D), "q", layer)
        o = torch.empty(self.batch, self.Hq, self.D, device=DEV)
        lse = torch.empty(self.batch, self.Hq, device=DEV)
        (capi.masw_full_attn if full else capi.masw_draft_attn)(self.h, layer, q.to(DEV), o, lse)
        want, want_l = (self.ref.full_attn if full else self.ref.draft_attn)(layer, q.float().numpy())
        if check:
            capi.masw_sync(self.h)
            assert_close(o, want, self.dtype, f"{'full' if full else 'draft'} O l={layer} step={self.step}")
            assert_close(lse, want_l, self.dtype, f"{'full' if full else 'draft'} LSE l={layer}")
        return o, lse, want, want_l

    def fstep(self, layer, active=None, full=False, check=True):
        """Fused append + attention (masw_draft_step / masw_full_step)."""
        k = self.rand((self.batch, self.Hkv, self.D), "k", layer)
        v = self.rand((self.batch, self.Hkv, self.D), "v", layer)
        q = self.rand((self.batch, self.Hq, self.D), "q", layer)
        o = torch.empty(self.batch, self.Hq, self.D, device=DEV)
        lse = torch.empty(self.batch, self.Hq, device=DEV)
        fn = capi.masw_full_step if full else capi.masw_draft_step
        fn(self.h, layer, q.to(DEV), k.to(DEV), v.to(DEV), o, lse, active=active)
        self.ref.append(layer, k.float().numpy(), v.float().numpy(), active=active)
        if check:
            want, want_l = (self.ref.full_attn if full else self.ref.draft_attn)(layer, q.float().numpy())
            capi.masw_sync(self.h)
            assert_close(o, want, self.dtype, f"{'full' if full else 'draft'} step O l={layer} step={self.step}")
            assert_close(lse, want_l, self.dtype, "step LSE")
        return o

    def fstep_slot(self, layer, seqs, active=None):
        """Fused draft step + slot write at a boundary (masw_draft_step_slot)."""
        B, n = self.batch, len(seqs)
        k = self.rand((B, self.Hkv, self.D), "k", layer)
        v = self.rand((B, self.Hkv, self.D), "v", layer)
        q = self.rand((B, self.Hq, self.D), "q", layer)
        qg = self.rand((n, self.Hq, self.D), "qg", layer)
        kg = self.rand((n, self.Hkv, self.D), "kg", layer)
        vg = self.rand((n, self.Hkv, self.D), "vg", layer)
        o = torch.empty(B, self.Hq, self.D, device=DEV)
        lse = torch.empty(B, self.Hq, device=DEV)
        og = torch.empty(n, self.Hq, self.D, device=DEV)
        lg = torch.empty(n, self.Hq, device=DEV)
        capi.masw_draft_step_slot(self.h, layer, q.to(DEV), k.to(DEV), v.to(DEV), o, seqs, qg.to(DEV), kg.to(DEV),
                                  vg.to(DEV), og, lse, lg, active=active)
        self.ref.append(layer, k.float().numpy(), v.float().numpy(), active=active)
        want, want_l = self.ref.draft_attn(layer, q.float().numpy())
        want_g, want_gl = self.ref.materialize_slot(layer, seqs, qg.float().numpy(), kg.float().numpy(),
                                                    vg.float().numpy())
        capi.masw_sync(self.h)
        assert_close(o, want, self.dtype, f"step_slot O l={layer} step={self.step}")
        assert_close(lse, want_l, self.dtype, "step_slot LSE")
        assert_close(og, want_g, self.dtype, f"step_slot O_g l={layer}")
        assert_close(lg, want_gl, self.dtype, "step_slot LSE_g")

    def materialize(self, layer, seqs):
        n = len(seqs)
        qg = self.rand((n, self.Hq, self.D), "qg", layer)
        kg = self.rand((n, self.Hkv, self.D), "kg", layer)
        vg = self.rand((n, self.Hkv, self.D), "vg", layer)
        og = torch.empty(n, self.Hq, self.D, device=DEV)
        lg = torch.empty(n, self.Hq, device=DEV)
        capi.masw_materialize_slot(self.h, layer, seqs, qg.to(DEV), kg.to(DEV), vg.to(DEV), og, lg)
        want, want_l = self.ref.materialize_slot(layer, seqs, qg.float().numpy(), kg.float().numpy(),
                                                 vg.float().numpy())
        capi.masw_sync(self.h)
        assert_close(og, want, self.dtype, f"slot O l={layer}")
        assert_close(lg, want_l, self.dtype, f"slot LSE l={layer}")
        return og

    def check_state(self, layer, seq):
        """Counters, slot position ids and every visible row's placement, bit-exact."""
        st = capi.masw_query(self.h, layer, seq)
        t, m = self.ref.t(layer, seq), self.ref.m(layer, seq)
        assert (st["t"], st["m"], st["dev_t"], st["dev_m"]) == (t, m, t, m), (st, t, m)
        sim = self.ref.sim[layer][seq]
        rows, cap = st["rows"], st["slot_capacity"]
        tdt = synth.torch_dtype(self.dtype)
        kb = torch.empty(self.Hkv, rows, self.D, dtype=tdt)
        vb = torch.empty(self.Hkv, rows, self.D, dtype=tdt)
        pos = capi.masw_mem_export(self.h, layer, seq, kb, vb, cap)
        kb = kb.float().numpy()
        vb = vb.float().numpy()
        raw_k, raw_v = self.ref.raw_k[layer][seq], self.ref.raw_v[layer][seq]
        Wc = st["ring_rows"]
        for i in sim.sink:
            assert np.array_equal(kb[:, i - 1], raw_k[i - 1]) and np.array_equal(vb[:, i - 1], raw_v[i - 1])
        ring = sim.ring_map()
        for i in sim.window:
            row = ring.index(i)
            assert row == (i - self.S - 1) % Wc
            assert np.array_equal(kb[:, self.S + row], raw_k[i - 1]), f"token {i} not in ring row {row}"
            assert np.array_equal(vb[:, self.S + row], raw_v[i - 1])
        for j in range(m):
            assert np.array_equal(kb[:, self.S + Wc + j], self.ref.slot_k[layer][seq][j])
            assert np.array_equal(vb[:, self.S + Wc + j], self.ref.slot_v[layer][seq][j])
            # library ids are 0-based: tau_j, the id of the raw token after g_j
            assert pos[j] == self.ref.slot_tau[layer][seq][j] == orc.slot_pos_id(j + 1, self.S, self.W, self.r) - 1


GUARD_BYTES = 4096
GUARD_BYTE = 0xC3


class Guarded:
    """A caller-owned device buffer with a guard band of GUARD_BYTES (0xC3) on
    each side, for out-of-bounds write checks of the handle-less calls (their
    workspaces and outputs).  `.t` is the buffer, viewed as dtype and shape."""

    def __init__(self, shape, dtype, zero=True):
        n = 1
        for x in shape:
            n *= x
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((nbytes + 2 * GUARD_BYTES,), GUARD_BYTE, dtype=torch.uint8, device=DEV)
        mid = self.raw[GUARD_BYTES:GUARD_BYTES + nbytes]
        if zero:
            mid.zero_()
        self.nbytes = nbytes
        self.t = mid.view(dtype).view(*shape) if n else mid.view(dtype)

    def check(self, what=""):
        torch.cuda.synchronize()
        lo = self.raw[:GUARD_BYTES]
        hi = self.raw[GUARD_BYTES + self.nbytes:]
        assert bool((lo == GUARD_BYTE).all()) and bool((hi == GUARD_BYTE).all()), f"{what}: guard band overwritten"
