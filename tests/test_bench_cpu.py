# Host-side pieces of bench.py: the code-only kernel hash that keys the ncu
# capture sidecars (a comment edit must keep a capture valid, a code edit must
# not) and the sidecar lookup itself.
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_keeps_literals():
    src = ('int a = 1;  // trailing\n'
           '/* block\n   comment */ const char *s = "a//b /* c */";\n'
           '\n'
           "char c = '/'; char d = '\\'';\n"
           '    int b;   \n')
    out = bench.code_only(src)
    assert "trailing" not in out and "block" not in out
    assert '"a//b /* c */"' in out
    assert "'/'" in out and "'\\''" in out
    assert all(line.strip() for line in out.splitlines())  # no empty lines
    assert all(line == line.rstrip() for line in out.splitlines())


def test_comment_edit_keeps_the_hash_and_code_edit_changes_it():
    code = "__device__ int f(int x) { return x + 1; }\n"
    a = bench.code_only("// one comment\n" + code)
    b = bench.code_only("/* another\n comment */\n" + code + "\n\n// tail\n")
    c = bench.code_only(code.replace("+ 1", "+ 2"))
    assert a == b
    assert a != c


SIDECARS = {("bf16", "hy3_tp8"): 1.5e8, ("bf16", "skewed"): 2.17e9, ("e4m3", "fp8"): 3.97e8}


def test_sidecars_are_well_formed():
    for (dtype, wl), algorithmic in SIDECARS.items():
        name = f"attn_{dtype.replace('e4m3', 'fp8')}_{wl}.json"
        with open(os.path.join(ROOT, "profiles", name)) as f:
            d = json.load(f)
        assert len(d["kernel_source_sha256"]) == 64
        # DRAM traffic of one launch: the algorithmic bytes and a little more
        assert algorithmic <= d["dram_bytes_per_launch"] <= 1.05 * algorithmic, name


def test_profiled_traffic_reads_only_a_matching_sidecar():
    assert bench.profiled_traffic("0" * 64, "bf16", "skewed") is None
    h = bench.kernel_source_hash()
    assert bench.profiled_traffic(h, "bf16", "no_such_workload") is None
    with open(os.path.join(ROOT, "profiles", "attn_bf16_skewed.json")) as f:
        captured = json.load(f)["kernel_source_sha256"]
    if captured != h:
        pytest.skip("the skewed capture was taken on other kernel code (traffic is reported as null)")
    assert bench.profiled_traffic(h, "bf16", "skewed") > 2.0e9
    assert bench.profiled_traffic(h, "e4m3", "fp8") > 3.9e8
