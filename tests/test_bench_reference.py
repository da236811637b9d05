"""The reference arm of bench.py (the CPU oracle timed on the host cores) runs
without a GPU and prints one JSON line with the fields the bench contract
names: the same metric and unit as the GPU arm, an oracle cpu_baseline whose
value is the line's (plus the one-core figure and the host's CPU), and an e2e
entry that moves no bytes."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == "tree nodes verified/sec (attn+verify)" and d["unit"] == "nodes/s"
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 3
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    # The default workload is the largest single-GPU one, and the config is the
    # very dict the GPU arm prints for it (so the two arms compare equal).
    assert bench.DEFAULT_WORKLOAD == "batch32-P2048-n16"
    assert d["value"] > 0 and d["config"] == bench.config_of(W.SPECS[bench.DEFAULT_WORKLOAD])
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    # ... and the same oracle on one core, with the host it ran on.
    one = cb["single_core"]
    assert one["cores"] == 1 and one["unit"] == d["unit"] and 0 < one["value"]
    assert cb["nproc"] >= 1 and cb["cpu_model"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_cpu_baseline_entry_of_the_gpu_arm():
    """The GPU arm builds its cpu_baseline with the same helper, on the
    workload's own inputs; here on the tiny workload with a one-pass sample."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    spec = W.SPECS["tiny-f32-P128-n16"]
    trees, att, gi, si = bench.workload_inputs(spec)
    n = int(trees.node_offsets[-1])
    cb = bench.oracle_baseline(spec, trees, att, gi, si, 0.0, bench.choose_heads_sample(spec, trees), n)
    assert cb["kind"] == "oracle" and cb["unit"] == "nodes/s" and cb["value"] > 0 and cb["cores"] >= 1
    assert cb["single_core"]["cores"] == 1 and cb["single_core"]["value"] > 0
    import oracle
    assert oracle.num_threads() == cb["cores"]  # the thread count is restored


def test_cpu_model_on_arm_and_x86(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    arm = tmp_path / "arm"
    arm.write_text("processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU part\t: 0xd4f\n\n"
                   "processor\t: 1\nCPU implementer\t: 0x41\nCPU part\t: 0xd4f\n")
    assert "implementer 0x41, part 0xd4f" in bench.host_cpu_model(str(arm))
    x86 = tmp_path / "x86"
    x86.write_text("processor\t: 0\nvendor_id\t: GenuineIntel\nmodel name\t: Some CPU @ 2.00GHz\n")
    assert bench.host_cpu_model(str(x86)) == "Some CPU @ 2.00GHz"
    assert bench.host_cpu_model(str(tmp_path / "missing")) is not None
