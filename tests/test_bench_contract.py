"""The benchmark's reference arm on CPU: `bench.py --impl reference` times the
oracle on the host cores and prints one JSON line with the keys of the
benchmark contract (its own arm needs a GPU and is checked there)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    d = json.loads(lines[0])
    for key, typ in (("impl", str), ("metric", str), ("value", float), ("unit", str), ("n_gpus", int),
                     ("steps", int), ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool),
                     ("scaling", str), ("dtype", str), ("data", str), ("config", dict),
                     ("cpu_baseline", dict), ("e2e", dict)):
        assert isinstance(d[key], typ), (key, d[key])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["vs_baseline"] is None and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_grouped_attainable_bound_limits():
    """The grouped GEMM's attainable time is, per expert, the larger of its
    compute time at the tensor peak and the time to stream its weights,
    activations and BF16 output: one expert holding every row is the plain
    compute time; experts of one row each are bound by their weight stream."""
    import types
    sys.path.insert(0, ROOT)
    import bench
    K, N = 7168, 2048
    pk = {"hbm_gbs": 1000.0, "fp8_tflops": 1000.0, "fp4_tflops": 3000.0}
    for fp4, code, peak in ((False, 1.0, 1000.0), (True, 0.5, 3000.0)):
        step = types.SimpleNamespace(moe_counts=[32768], moe_kn=(K, N))
        r = bench.attainable(step, 1.0, pk, fp4)
        t_fl = 2.0 * 32768 * N * K / (peak * 1e12)
        t_by = (N * K * (code + 1 / 32) + 32768 * K * (code + 1 / 32) + 32768 * N * 2) / 1e12
        assert abs(r["attainable_ms"] - round(max(t_fl, t_by) * 1e3, 4)) < 1e-9
        step = types.SimpleNamespace(moe_counts=[1] * 64, moe_kn=(K, N))
        r = bench.attainable(step, 2.0, pk, fp4)
        t_w = 64 * (N * K * (code + 1 / 32) + K * (code + 1 / 32) + N * 2) / 1e12
        assert abs(r["attainable_ms"] - round(t_w * 1e3, 4)) < 1e-9
        assert abs(r["frac_attainable"] - r["attainable_ms"] / 2.0) <= 1e-4
