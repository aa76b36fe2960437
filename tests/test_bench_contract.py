"""bench.py's host side on CPU: the reference arm's JSON line (the FP64 oracle timed
on the host cores), the names that tie the per-kernel byte model to the
library's timing records, and the binding roofline's minimal-I/O arithmetic.
No GPU work."""
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


def test_binding_roofline_counts_the_minimal_io():
    # Minimal I/O per token: every input read once and every output written
    # once at the ABI's precisions.  KDA per (token, head): q, k, v, out BF16
    # (4 x 256 B), g FP32 (512 B), beta BF16 (2 B) in the forward = 1,538 B;
    # the backward reads the same inputs and dout (1,538 B) and writes dq, dk,
    # dv (BF16), dg (FP32), dbeta (BF16) (1,282 B): 4,358 B in all.
    sys.path.insert(0, ROOT)
    import bench
    fwd, bwd = bench.io_bytes("kda", 16, 16)
    assert (fwd, bwd) == (1538 * 16, 2820 * 16)
    # Grouped GDN (16, 48): q, k once per Q/K head, scalar FP32 gate and beta.
    fwd, bwd = bench.io_bytes("gdn", 16, 48)
    qk, vrow, sc = 2 * 16 * 128 * 2, 48 * 128 * 2, 48 * 4
    assert (fwd, bwd) == (qk + 2 * vrow + 2 * sc, (qk + 2 * vrow + 2 * sc) + (qk + vrow + 2 * sc))
    # The whole step's fraction: the HBM time of the minimal bytes over the
    # step time when HBM binds (KDA, T = 261,392, H = 16 at 6,707.5 GB/s).
    pk = {"hbm_gbs": 6707.5, "bf16_tflops_sustained": 1783.0}
    r = bench.binding_roofline("kda", 261392, 16, 16, 18.19, pk)
    assert r["bound"] == "hbm"
    assert abs(r["alg_bytes"] - 4358 * 16 * 261392) < 1
    assert abs(r["frac"] - 4358 * 16 * 261392 / 6707.5e9 * 1e3 / 18.19) < 1e-12
    assert abs(r["frac"] - 0.1494) < 5e-4
