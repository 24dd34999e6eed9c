"""The allocation-free verify entry point (masw_verify_attn_noalloc).

It exists for callers that cannot give the library scratch memory or call
cudaMalloc -- code that only receives input and output pointers, code whose
device memory belongs to another allocator, or a loop that cannot afford the
device-wide synchronisation an allocation may cause.  This test calls it through
the C ABI twice in a row, with different shapes, and checks each result against
masw_verify_attn (which takes a caller workspace) and against the CPU oracle,
within the tolerance the other bf16 tests use, and that the status word the call
copies out is 0.  (Both shapes run the usual split count: at one CTA per SM the
partials stay far below the fixed array on this GPU.)

The file name makes pytest collect it last, so a run that stops at the first
failure has run every other test before this one.
"""
import pytest
import torch

import oracle.masw_oracle as orc
from compressed_draft_kv_gb300 import capi, synth
from gpu_helpers import DEV, assert_close
from libmasw_fixture import ensure_built

pytestmark = pytest.mark.gpu


def _inputs(B, Lq, Hq, Hkv, Tmax, kv_len, seed):
    D = 128
    q = synth.normal((B, Lq, Hq, D), "bf16", "noalloc", seed, "q").to(DEV)
    k = synth.normal((B, Hkv, Tmax, D), "bf16", "noalloc", seed, "k").to(DEV)
    v = synth.normal((B, Hkv, Tmax, D), "bf16", "noalloc", seed, "v").to(DEV)
    kl = torch.tensor(kv_len, dtype=torch.int32, device=DEV)
    return q, k, v, kl


def test_noalloc_verify_matches_workspace_verify_twice():
    ensure_built()
    torch.cuda.set_device(DEV)
    cases = [
        (2, 6, 32, 8, 700, [700, 333], 1),
        (4, 6, 32, 8, 8192, [8192, 5000, 7001, 64], 2),
    ]
    for B, Lq, Hq, Hkv, Tmax, kv_len, seed in cases:
        q, k, v, kl = _inputs(B, Lq, Hq, Hkv, Tmax, kv_len, seed)
        o_ref = torch.empty(B, Lq, Hq, 128, device=DEV)
        l_ref = torch.empty(B, Lq, Hq, device=DEV)
        capi.masw_verify_attn(q, k, v, kl, o_ref, l_ref)
        o = torch.full((B, Lq, Hq, 128), float("nan"), device=DEV)
        lse = torch.full((B, Lq, Hq), float("nan"), device=DEV)
        status = torch.full((1,), -99, dtype=torch.int32, device=DEV)
        capi.masw_verify_attn_noalloc(q, k, v, kl, o, lse, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == capi.MASW_OK
        assert_close(o, o_ref.double().cpu().numpy(), "bf16", f"noalloc O vs workspace B={B} T={Tmax}")
        assert_close(lse, l_ref.double().cpu().numpy(), "bf16", f"noalloc LSE vs workspace B={B} T={Tmax}")
        o_or, l_or = orc.verify_attn(q.float().cpu().numpy(), k.float().cpu().numpy(), v.float().cpu().numpy(),
                                     kv_len)
        assert_close(o, o_or, "bf16", f"noalloc O vs oracle B={B} T={Tmax}")
        assert_close(lse, l_or, "bf16", f"noalloc LSE vs oracle B={B} T={Tmax}")


def test_noalloc_rejects_sizes_beyond_its_limit():
    ensure_built()
    torch.cuda.set_device(DEV)
    q = torch.zeros(1, 1, 4097, 128, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(1, 4097, 1, 128, dtype=torch.bfloat16, device=DEV)
    kl = torch.ones(1, dtype=torch.int32, device=DEV)
    o = torch.empty(1, 1, 4097, 128, device=DEV)
    with pytest.raises(capi.MaswError) as ei:
        capi.masw_verify_attn_noalloc(q, k, k, kl, o)
    assert ei.value.code == capi.MASW_EINVAL
    assert "static scratch limit" in str(ei.value)
