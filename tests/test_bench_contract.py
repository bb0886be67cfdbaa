"""The reference arm of bench.py (the fp64 oracle on the host cores) runs without a GPU and
prints one JSON line with the keys the benchmark contract names."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "full_h16_d128"


def test_varlen_workload_recipe():
    """The packed-batch timing draws its sequence lengths log-uniformly in [lo, hi] from a
    seeded generator: the same 64 lengths on every run."""
    sys.path.insert(0, ROOT)
    import bench
    a, b = bench.varlen_lengths(), bench.varlen_lengths()
    cfg = bench.VARLEN
    assert a == b and len(a) == cfg["n"]
    assert all(cfg["lo"] <= n <= cfg["hi"] for n in a)
    assert len(set(a)) > cfg["n"] // 2  # a spread of lengths, not one repeated value
