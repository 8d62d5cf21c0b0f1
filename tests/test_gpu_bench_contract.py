"""bench.py's JSON line on a GPU: every key of the contract is present and self-consistent
(a short run: 20 timed steps, 3 warm-up, 3 end-to-end steps, no CPU baseline). The headline is the
Llama-3-8B rank-0 shard step (1,003,782,656 elements, 8 bf16 ranks) + the unshard of the 8 shards
into the 8,030,261,248-element flat unit; the per-kernel times must add up to the step time."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

N_SHARD = 1_003_782_656
P_UNIT = 8_030_261_248


def test_bench_line_has_the_contract_keys():
    p = subprocess.run([sys.executable, "bench.py", "--steps", "20", "--warmup", "3", "--no-cpu-baseline",
                        "--e2e-steps", "3"], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks", "kernels"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 3 and d["scaling"] == "weak"
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    cfg = d["config"]
    assert cfg["shard_elems"] == N_SHARD and cfg["unit_params"] == P_UNIT and "workload" in cfg
    assert cfg["bytes_per_step"] == N_SHARD * (2 * 8 + 26) + 4 * P_UNIT
    # value = bytes per step / time per step
    assert d["value"] == pytest.approx(cfg["bytes_per_step"] / (d["ms_per_step"] * 1e-3) / 1e9, rel=1e-3)
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 1.2
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-3)
    # the roofline is recomputable from the line: algorithmic bytes / average launch time / peak
    assert r["achieved"] == pytest.approx(r["algorithmic_bytes"] / (r["avg_launch_ms"] * 1e-3) / 1e9, rel=1e-3)
    # per-kernel times add up to the step's own time
    chk = d["kernels"]["sum_check"]
    assert chk["within_5pct"] and abs(chk["ratio"] - 1) <= 0.05
    assert d["roofline_unshard"]["frac"] > 0.5
    e = d["e2e"]
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in e, k
    assert e["h2d_bytes_per_step"] == 2 * 8 * N_SHARD and e["d2h_bytes_per_step"] == 4
    assert 0 < e["value"] < d["value"]
    assert d["gpu_launches"] == 2 * 20
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    sec = d["secondary"]
    for key in ("gpt2_small_rank0_shard_N8", "llama70b_layer_N64_fp16_all_shards"):
        b = sec[key]
        assert b["GB/s"] > 0 and b["kernels"]["sum_check"]["ratio"] > 0
