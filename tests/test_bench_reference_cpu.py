"""bench.py's reference arm on the CPU: `--impl reference` times the oracle on a
bounded sample of the AlexNet step (host cores only, no GPU) and prints one
JSON line with the keys the measurement contract asks for.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


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


def test_step_traffic_record():
    """bench.py reports the GEMM kernels' DRAM bytes per step (its roofline
    `traffic`) from the stored ncu counters, and only while the GEMM sources
    are the ones they were taken on.  The record must be plausible (about the
    sum of the GEMMs' own inputs and outputs, 1.26 GB), and a changed source
    must make the figure null."""
    import json
    bench = _bench()
    with open(bench.STEP_TRAFFIC) as f:
        rec = json.load(f)
    assert 1.0e9 < rec["conv_gemm_dram_bytes_per_step"] < 1.6e9
    t = bench.gemm_traffic_per_step()
    assert t is None or t == rec["conv_gemm_dram_bytes_per_step"]
    assert bench.gemm_sources_digest(rec["gemm_sources"][:-1]) != rec["gemm_sources_sha256"]
