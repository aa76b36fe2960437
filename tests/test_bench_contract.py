"""bench.py's host side on CPU: the reference arm's JSON line (the FP64 oracle timed
on the host cores) and the names that tie the per-kernel byte model to the
library's timing records.  No GPU work."""
import json
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line_with_the_contract_keys():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "kda_tiny", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "kda_tiny" and d["steps"] == 1
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == d["value"] and cpu["sample"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["e2e"]["d2h_bytes_per_step"] == 0


def test_byte_model_names_are_the_library_timing_names():
    sys.path.insert(0, ROOT)
    import bench
    src = open(os.path.join(ROOT, "gated_delta_rule_varlen_gb300", "csrc", "gdr_api.cu")).read()
    timed = set(re.findall(r'ProfScope ps\("(\w+)"', src))
    assert set(bench.KERNEL_MODEL) <= timed, set(bench.KERNEL_MODEL) - timed
    for name, (b, f) in bench.KERNEL_MODEL.items():
        assert b > 0 and f > 0, name
