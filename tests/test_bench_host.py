"""Host-side helpers of bench.py (no GPU): the code hash that gates the
recorded DRAM traffic of the fused-step kernel."""
import os
import re

import bench


def test_code_only_ignores_comments_and_blank_lines():
    a = "int f(int x) {\n    return x + 1;   // add one\n}\n"
    b = "/* a header\n   comment */\nint f(int x) {\n\n    return x + 1;\n}   \n"
    assert bench._code_only(a) == bench._code_only(b)


def test_code_only_sees_code_changes():
    a = "int f(int x) { return x + 1; }\n"
    b = "int f(int x) { return x + 2; }\n"
    assert bench._code_only(a) != bench._code_only(b)


def test_recorded_traffic_is_the_profile_figure_or_null():
    with open(os.path.join(bench.ROOT, "profiles", "decode_mma_step_b8_32k.md")) as f:
        rec = int(re.search(r"traffic_bytes_per_launch: (\d+)", f.read()).group(1))
    assert bench._recorded_traffic() in (None, rec)
