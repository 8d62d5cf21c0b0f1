"""bench.py's JSON line on a GPU: every key of the contract is present and self-consistent
(a short run: 20 timed steps, 3 warm-up, 3 end-to-end steps, no CPU baseline)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_has_the_contract_keys():
    p = subprocess.run([sys.executable, "bench.py", "--steps", "20", "--warmup", "3", "--no-cpu-baseline",
                        "--e2e-steps", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 3 and d["scaling"] == "weak"
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    cfg = d["config"]
    assert cfg["bytes_per_step"] == 1_151_068_224 and "workload" in cfg
    # value = bytes per step / time per step
    assert d["value"] == pytest.approx(cfg["bytes_per_step"] / (d["ms_per_step"] * 1e-3) / 1e9, rel=1e-3)
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 1.2
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-3)
    e = d["e2e"]
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in e, k
    assert e["h2d_bytes_per_step"] == 2 * 8 * 15_554_976 and e["d2h_bytes_per_step"] == 4
    assert 0 < e["value"] < d["value"]
    assert d["gpu_launches"] == 2 * 20
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
