"""Host-side pieces of bench.py (no GPU): the code hash that keys the recorded DRAM
traffic, and the traffic lookup."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_code_only_drops_comments_and_blank_space():
    src = "int a; // note\n/* block\n comment */ int  b;\n\n  asm(\"fma.rn.f32x2 %0;\");\n"
    assert bench.code_only(src) == 'int a; int b; asm("fma.rn.f32x2 %0;");'


def test_code_hash_ignores_comments_but_not_code():
    base = {n: "x = 1; // c\n" for n in bench.KERNEL_SOURCES}
    edited = dict(base)
    edited[bench.KERNEL_SOURCES[0]] = "x = 1; // another comment\n/* more */\n"
    changed = dict(base)
    changed[bench.KERNEL_SOURCES[0]] = "x = 2;\n"
    h = bench.kernel_sources_hash(base.__getitem__)
    assert h == bench.kernel_sources_hash(edited.__getitem__)
    assert h != bench.kernel_sources_hash(changed.__getitem__)


def test_recorded_traffic_needs_a_matching_entry_and_workload():
    assert bench.recorded_traffic("no_such_entry", "sgemm_4096") is None
    assert bench.recorded_traffic("256x128x64_t8x16_s2_f2_v4", "no_such_workload") is None


def test_reference_arm_prints_the_gpu_arms_config(capsys):
    """Both arms of a workload carry the same `config` (the GPU-only details of the
    plan go to `plan`), so their lines can be matched key for key."""
    import argparse
    import json
    w = bench.WORKLOADS["sgemm_256"]
    args = argparse.Namespace(steps=1, warmup=0, gpus=1)
    assert bench.run_reference(args, w) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"] == bench.workload_config(w, 1)
    assert set(line["config"]) == {"workload", "M", "N", "K", "l2", "parallelism"}
