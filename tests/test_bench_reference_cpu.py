"""bench.py's reference arm on the CPU: `--impl reference` times the oracle on a
bounded sample of the AlexNet step (host cores only, no GPU) and prints one
JSON line with the keys the measurement contract asks for.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1", "--ref-batch", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["warmup"] >= 3                      # at least three untimed warm-up steps, always
    assert d["value"] > 0 and d["unit"] == "TFLOP/s"
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_step_profile_states_gemm_traffic():
    """bench.py reads the GEMM kernels' DRAM bytes per step (its roofline
    `traffic`) from the committed launch-list summary; the line must be there
    and plausible: about the sum of the GEMMs' own inputs and outputs (1.26 GB)."""
    import re
    with open(os.path.join(ROOT, "profiles", "launch_list_alexnet_b128_step.md")) as f:
        m = re.search(r"conv_gemm_dram_bytes_per_step = (\d+)", f.read())
    assert m, "launch-list summary lacks the conv_gemm_dram_bytes_per_step line"
    assert 1.0e9 < int(m.group(1)) < 1.6e9
