"""bench.py's reference arm (the oracle on the host cores) prints one JSON
line with the contract's keys for each workload family; CPU only, one short
step each."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"}


@pytest.mark.parametrize("workload", ["tiny_decode", "indexer_tiny", "cache_write_decode", "prolog_decode"])
def test_reference_arm_prints_one_contract_line(workload):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload, "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is False
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_attention_roofline_picks_the_binding_bound():
    """bytes at the HBM peak against FLOPs at the bf16 peak: the slower one is reported."""
    sys.path.insert(0, ROOT)
    import bench
    hbm, tf = 6790.0, 1887.7
    # 301 MB and 73 GFLOP (the decode workload): 44.3 us of bytes > 38.7 us of FLOPs -> hbm
    r = bench.roofline_of({"roofline_bytes": 301e6, "flops": 73.0e9}, 163.3, hbm, tf, "measured", None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["frac"] == pytest.approx(301e6 / 163.3e-6 / 1e9 / hbm, rel=1e-3)
    # 189 MB and 73 GFLOP (INT8): 27.8 us of bytes < 38.7 us of FLOPs -> tensor
    r = bench.roofline_of({"roofline_bytes": 189e6, "flops": 73.0e9}, 178.7, hbm, tf, "measured", 1.0)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["traffic"] == 1.0
    assert r["frac"] == pytest.approx(73.0e9 / 178.7e-6 / 1e12 / tf, rel=1e-3)
    assert r["peak"] == tf and "fallback" not in r["peak_source"]
    assert "fallback" in bench.roofline_of({"roofline_bytes": 1.0, "flops": 1.0}, 1.0, hbm, tf, "fallback",
                                           None)["peak_source"]
