"""The decode kernels' segment-table bounds test, on the host: every table the
index model builds from in-range counters lies inside its (layer, sequence,
kv head) block, and tables with a planted fault are refused; and the prefill's
interleaved row order matches a brute-force construction.

The library runs this test on every decode launch's speculative tables when a
handle is created with MASW_CHECK_SEGMENTS=1 (the GPU tests set it), and the
fp32 decode kernel runs it on the device; this file checks the test itself.
It compiles tests/segment_check_host.cu (host code only) with nvcc."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))

EXPECTED = {
    # in-range counters: no table fails
    "draft_in_range_failures": 0,
    "step_in_range_failures": 0,
    "slot_in_range_failures": 0,
    "nosink_in_range_failures": 0,
    "full_in_range_failures": 0,
    # counters past capacity
    "full_t_past_capacity_ok": 0,
    "slot_count_past_capacity_ok": 0,
    "slot_count_at_capacity_ok": 1,
    # sink, window wrapped around the ring (two runs), slot chain, new row
    "reference_table_runs": 5,
    "reference_table_ok": 1,
    # planted faults
    "sink_run_into_ring_ok": 0,
    "slot_run_past_block_ok": 0,
    "overlapping_runs_ok": 0,
    "foreign_caller_row_ok": 0,
    "v_offset_mismatch_ok": 0,
    "empty_run_ok": 0,
    "other_heads_block_ok": 0,
    "six_runs_ok": 0,
    # the prefill's interleaved query order (raw tokens, slot m right after raw
    # token tau_m) against brute force over 1200 (S, W, r, T) shapes
    "interleaved_rows": 745024,
    "interleaved_mismatches": 0,
}


def test_segment_bounds_check_accepts_the_index_model_and_refuses_planted_faults(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "segment_check_host")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                    os.path.join(HERE, "segment_check_host.cu"), "-o", exe], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    got = {k: int(v) for k, v in (line.split() for line in out.strip().splitlines())}
    assert got == EXPECTED
