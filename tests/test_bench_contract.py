"""bench.py's JSON line: the keys and value types the measurement contract
fixes, for the reference arm (the oracle on the host cores, CPU) and for
the GPU arm on a short two-layer run (GPU)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
COMMON = {"metric": str, "value": float, "unit": str, "n_gpus": int, "steps": int, "warmup": int,
          "ms_per_step": float, "higher_is_better": bool, "scaling": str, "dtype": str, "data": str,
          "config": dict}


def _last_json(args, timeout):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                       timeout=timeout, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def _check_common(d, steps, warmup):
    for k, t in COMMON.items():
        assert isinstance(d[k], t) or (t is float and isinstance(d[k], int)), (k, d[k])
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert "workload" in d["config"]


def test_reference_arm_line():
    d = _last_json(["--impl", "reference", "--steps", "1", "--warmup", "3", "--cpu-budget", "0.1"], 300)
    _check_common(d, 1, 3)
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


@pytest.mark.gpu
def test_gpu_arm_line():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = _last_json(["--layers", "2", "--steps", "3", "--warmup", "3", "--skip-cpu", "--skip-prefill",
                    "--skip-long-prefill", "--skip-int4", "--admission", "2"], 900)
    _check_common(d, 3, 3)
    assert "impl" not in d
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0 and r["achieved"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-2)
    assert r["traffic"] is None or r["traffic"] > 0
    c = d["clocks"]
    assert c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list)
    e = d["e2e"]
    assert e["unit"] == d["unit"] and e["value"] > 0
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
