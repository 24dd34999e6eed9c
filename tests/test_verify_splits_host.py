"""The split plans of the verify kernel on the host (masw_splits.h, compiled
with the host compiler): the allocation-free entry point's reduction is not
reached with one CTA per SM on a 152-SM GPU, and where larger resident-slot
counts reach it, it keeps the largest split count whose partials fit in the
4 MiB static array (or one split, which writes no partials)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CAP = 4 << 20


def partial_bytes(pairs, nq, n):
    # per pair and split: NQ rows of 128 outputs + max + sum, 4-byte floats, rounded up to 256 B
    b = pairs * n * nq * 130 * 4
    return (b + 255) // 256 * 256


def test_noalloc_split_reduction(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if not cxx:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path / "verify_splits_host")
    subprocess.run([cxx, "-std=c++17", "-O1", os.path.join(HERE, "verify_splits_host.cpp"), "-o", exe], check=True)
    lines = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split("\n")
    rows = [tuple(map(int, ln.split())) for ln in lines if ln.strip()]
    assert len(rows) == 13 * 6 * 3 * 4
    reduced = 0
    for pairs, nq, tmax, slots, plan, n in rows:
        # the usual plan: one wave of the slots, >= 256 keys per split, <= 64 splits
        assert plan == max(1, min(slots // pairs, max(1, (tmax + 255) // 256), 64))
        if slots == 152:
            assert n == plan, (pairs, nq, tmax)          # not reached with one CTA per SM on 152 SMs
        assert 1 <= n <= plan
        assert n == 1 or partial_bytes(pairs, nq, n) <= CAP
        # the largest count that fits: one more split would not
        assert n == plan or partial_bytes(pairs, nq, n + 1) > CAP
        reduced += n < plan
    assert reduced > 0                                    # larger slot counts do reach the reduction
    # a worked case: 5 pairs, 32 rows, 304 slots -> plan 60 (4.99 MB), cut to 50 (4.16 MB)
    assert (5, 32, 32768, 304, 60, 50) in rows
