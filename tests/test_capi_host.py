"""The C-ABI library without a GPU: it loads, exports every declared symbol,
its host-side index model matches the oracle's simulator bit for bit, and its
argument checks fail with the documented codes."""
import ctypes
import os
import re

import pytest

import oracle.masw_oracle as o
from compressed_draft_kv_gb300 import capi
from libmasw_fixture import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "masw.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(masw_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = ensure_built()
    names = _declared()
    assert len(names) >= 16
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(capi.EXPORTS) == names
    assert capi.masw_version().count(".") == 2


def test_index_model_matches_simulator():
    ensure_built()
    for S in (0, 1, 4):
        for W in (1, 3, 8):
            for r in (1, 2, 5):
                for R in (0, 2):
                    sim = o.IndexSim(S, W, r, R)
                    for t in range(1, 3 * (S + W + r) + 2):
                        sim.append()
                        lo, _ = o.local_window(t, S, W)
                        assert capi.masw_index(0, t, S, W, r, R) == lo
                        assert capi.masw_index(1, t, S, W, r, R) == len(sim.window)
                        assert capi.masw_index(3, t, S, W, r, R) == int(sim.boundary_due())
                        if sim.boundary_due():
                            sim.materialize()
                        assert capi.masw_index(2, t, S, W, r, R) == len(sim.slots)
                        assert capi.masw_index(5, t, S, W, r, R) == len(sim.visible_raw()) + len(sim.slots)
                        row = capi.masw_index(4, t, S, W, r, R)
                        if t <= S:
                            assert row == -1
                        else:
                            assert sim.ring_map()[row] == t


def test_index_at_workload_sizes():
    ensure_built()
    assert capi.masw_index(5, 2048, 4, 256, 256, 0) == 266
    assert capi.masw_index(5, 8192, 4, 1024, 512, 0) == 1041
    assert capi.masw_index(5, 32768, 4, 1024, 512, 0) == 1089
    assert capi.masw_index(3, 8196, 4, 1024, 512, 0) == 1
    assert capi.masw_index(3, 32772, 4, 1024, 512, 0) == 1
    assert capi.masw_index(0, 5, -1, 3, 2, 0) == -1


def test_argument_errors_are_reported():
    lib = ensure_built()
    h = ctypes.c_void_p()
    opts = capi.masw_opts_t(1, capi.MASW_BF16, 1024, 0.0, 0, 0, 0)
    assert lib.masw_mem_create(4, 0, 8, 2, 64, 1, ctypes.byref(opts), ctypes.byref(h)) == capi.MASW_EINVAL
    assert h.value is None
    assert lib.masw_mem_create(4, 8, 8, 2, 96, 1, ctypes.byref(opts), ctypes.byref(h)) == capi.MASW_EINVAL
    assert "head_dim" in capi.masw_last_error(None)
    bad = capi.masw_opts_t(capi.MASW_MAX_BATCH + 1, capi.MASW_BF16, 1024, 0.0, 0, 0, 0)
    assert lib.masw_mem_create(4, 8, 8, 2, 64, 1, ctypes.byref(bad), ctypes.byref(h)) == capi.MASW_EINVAL
    # NULL handles are rejected, not dereferenced
    assert lib.masw_draft_attn(None, 0, None, 8, None, None, None) == capi.MASW_EINVAL
    assert lib.masw_append_kv(None, 0, None, None, None, None) == capi.MASW_EINVAL
    assert lib.masw_mem_destroy(None) == capi.MASW_OK
    out = ctypes.c_size_t()
    assert lib.masw_verify_workspace_bytes(4, 6, 32, 8, 64, 1024, ctypes.byref(out)) == capi.MASW_EINVAL
    assert lib.masw_verify_workspace_bytes(4, 16, 32, 8, 128, 1024, ctypes.byref(out)) == capi.MASW_EINVAL
    assert lib.masw_verify_attn(None, None, None, None, 1, 1, 8, 8, 128, 16, 1, 0.0, None, None, None, 0,
                                None) == capi.MASW_EINVAL


def test_create_without_gpu_fails_cleanly():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib = ensure_built()
    h = ctypes.c_void_p()
    rc = lib.masw_mem_create(4, 8, 8, 2, 64, 1, None, ctypes.byref(h))
    assert rc in (capi.MASW_ECUDA, capi.MASW_ENOMEM)
    assert h.value is None
    assert capi.masw_last_error(None)


def test_eq1_speedup_matches_oracle():
    ensure_built()
    for args in [(5, 5, 0.0, 1.0), (0, 5, 1.0, 1.0), (3.65, 5, 13.94, 40.0), (4.72, 5, 0.2, 1.0)]:
        assert abs(capi.masw_eq1_speedup(*args) - o.eq1_speedup(*args)) < 1e-12
    assert capi.masw_eq1_speedup(1, 5, 1.0, 0.0) == -1.0


def test_allocation_limit_refuses_before_any_cuda_call(monkeypatch):
    """MASW_DEVICE_MEMORY_LIMIT below the pool's size: create fails with
    MASW_ENOMEM before touching the device (so this runs without a GPU), the
    handle stays NULL and the message names the limit."""
    lib = ensure_built()
    monkeypatch.setenv("MASW_DEVICE_MEMORY_LIMIT", "1048576")
    opts = capi.masw_opts_t(8, capi.MASW_BF16, 32768, 0.0, 0, 0, 16)
    h = ctypes.c_void_p(1234)
    rc = lib.masw_mem_create(4, 1024, 512, 8, 128, 28, ctypes.byref(opts), ctypes.byref(h))
    assert rc == capi.MASW_ENOMEM
    assert h.value is None
    assert b"MASW_DEVICE_MEMORY_LIMIT" in lib.masw_last_error(None)


def test_check_guards_rejects_a_null_handle():
    lib = ensure_built()
    assert lib.masw_check_guards(None) == capi.MASW_EINVAL
