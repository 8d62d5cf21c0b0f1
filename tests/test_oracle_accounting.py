"""Pins of the oracle's byte accounting against the pages' worked numbers (no GPU)."""
import json
import os

import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load():
    with open(os.path.join(GOLDEN, "page_accounting.json")) as f:
        return json.load(f)


def test_page_worked_numbers():
    for c in load()["cases"]:
        b = oracle.state_bytes(int(c["P"]), c["N"], c["M"])
        for k, gb in c.get("expect_GB", {}).items():
            assert b[k] / 1e9 == pytest.approx(gb, rel=1e-12), (c["source"], k)
        for k, gb in c.get("expect_shard_GB", {}).items():
            assert b[k] / c["N"] / 1e9 == pytest.approx(gb, rel=1e-12), (c["source"], k)
        for k, (gb, rel) in c.get("expect_GB_approx", {}).items():
            assert b[k] / 1e9 == pytest.approx(gb, rel=rel), (c["source"], k)


def test_strategy_savings_per_param():
    s = load()["savings_per_P"]
    b = oracle.state_bytes(1_000_000, s["N"], 1)
    assert b["shard_grad_op_saving"] / 1e6 == pytest.approx(s["shard_grad_op_saving"][0], rel=s["shard_grad_op_saving"][1])
    assert b["full_shard_saving"] / 1e6 == pytest.approx(s["full_shard_saving"][0], rel=s["full_shard_saving"][1])


def test_mixed_precision_bill():
    mp = load()["mixed_precision_bytes_per_param"]
    b = oracle.state_bytes(1, 1, 1)
    for k in ("mp_params16", "mp_grads16", "mp_master32", "mp_adam32", "mp_total"):
        assert b[k] == mp[k]
    # the mixed bill equals the fp32 bill (16P either way)
    assert b["mp_total"] == b["fp32_total"] == 16


def test_sharding_divides_by_N():
    for N in (1, 2, 8, 64):
        b = oracle.state_bytes(10**9, N, 4)
        assert b["full_shard_per_gpu"] * N == pytest.approx(b["no_shard_per_gpu"], rel=1e-15)
        assert b["full_shard_peak"] == pytest.approx(b["full_shard_per_gpu"] + 4e9 / 4, rel=1e-15)
        assert b["shard_grad_op_per_gpu"] >= b["full_shard_per_gpu"]
