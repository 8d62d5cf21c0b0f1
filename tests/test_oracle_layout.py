"""Pins of the oracle's flat layout and shard rule (no GPU).

Page: "FSDP: Fully Sharded Data Parallel Training at Scale" -- a unit's tensors
are flattened into one vector of length P and GPU k holds elements
floor(kP/N) .. floor((k+1)P/N) - 1.
Pinned against brute force (the largest j with j*N <= k*P, found by
counting, not by division), the invariants of an exact tiling, and the
rule's worked instances in tests/golden/page_shard_rule.json.
"""
import json
import os

import numpy as np
import pytest

import oracle
from synth import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_bounds(P: int, N: int) -> np.ndarray:
    # bounds[k] = #{ j in 1..P : j*N <= k*P }  (the largest j with j*N <= k*P), by counting
    j = np.arange(1, P + 1, dtype=np.int64)
    k = np.arange(N + 1, dtype=np.int64)
    return (j[None, :] * N <= (k * P)[:, None]).sum(axis=1).astype(np.int64)


def test_bounds_brute_force_small():
    for P in range(0, 301):
        for N in range(1, 71):
            _, b = oracle.flatten_layout([P], N)
            assert np.array_equal(b, brute_bounds(P, N)), (P, N)


def test_tiling_invariants():
    rng = np.random.default_rng(1)
    for _ in range(400):
        T = int(rng.integers(0, 12))
        numels = rng.integers(0, 50, size=T)
        N = int(rng.integers(1, 40))
        offs, b = oracle.flatten_layout(numels, N)
        P = int(numels.sum())
        assert offs[0] == 0 and offs[-1] == P
        assert np.array_equal(np.diff(offs), numels)
        assert b[0] == 0 and b[-1] == P
        lens = np.diff(b)
        assert (lens >= 0).all()
        # lengths are floor(P/N) or ceil(P/N): equal shares to within one element
        assert set(np.unique(lens)).issubset({P // N, -(-P // N)})
        # every element is owned by exactly the shard the rule names
        for i in range(P):
            k = oracle.shard_of(P, N, i)
            assert b[k] <= i < b[k + 1]
        # segments of all shards cover every tensor element exactly once
        cover = np.zeros(P, dtype=np.int64)
        for k in range(N):
            segs = oracle.shard_segments(offs, b, k)
            assert sum(s[3] for s in segs) == b[k + 1] - b[k]
            for t, toff, soff, ln in segs:
                assert ln > 0 and 0 <= toff and toff + ln <= numels[t]
                lo = offs[t] + toff
                assert lo == b[k] + soff
                cover[lo:lo + ln] += 1
        assert (cover == 1).all()


def test_page_rule_instances():
    with open(os.path.join(GOLDEN, "page_shard_rule.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        _, b = oracle.flatten_layout([c["P"]], c["N"])
        assert b.tolist() == c["bounds"]


def test_first_shards_match_page_wording():
    # GPU 0 holds 0 .. floor(P/N)-1 ; GPU 1 holds floor(P/N) .. floor(2P/N)-1
    for P, N in [(1000, 7), (164224, 4), (123457, 64)]:
        _, b = oracle.flatten_layout([P], N)
        assert b[0] == 0 and b[1] == P // N and b[2] == (2 * P) // N


def test_workload_unit_sizes():
    assert sum(workloads.tiny_mlp_numels()) == 164_224
    assert sum(workloads.gpt2_small_numels()) == 124_439_808
    assert len(workloads.gpt2_small_numels()) == 148
    assert sum(workloads.llama3_8b_numels()) == 8_030_261_248
    assert sum(workloads.llama70b_layer_numels()) == 855_654_400
    _, b = oracle.flatten_layout(workloads.llama70b_layer_numels(), 64)
    assert (np.diff(b) == 13_369_600).all()


def test_large_P_needs_64bit_products():
    # k*P exceeds 2^32 for the Llama-3-8B unit; the rule must still hold exactly
    numels = workloads.llama3_8b_numels()
    offs, b = oracle.flatten_layout(numels, 8)
    P = int(offs[-1])
    assert [int(x) for x in b] == [k * P // 8 for k in range(9)]
    # and for a P near 2^62 with many ranks (k*P needs more than 64 bits)
    P = (1 << 62) + 12345
    _, b = oracle.flatten_layout([P], 1000)
    assert [int(x) for x in b] == [k * P // 1000 for k in range(1001)]


def test_segments_straddle_tensors():
    numels = workloads.llama70b_layer_numels()
    offs, b = oracle.flatten_layout(numels, 64)
    counts = [len(oracle.shard_segments(offs, b, k)) for k in range(64)]
    assert min(counts) == 1 and max(counts) == 3


def test_invalid_arguments():
    with pytest.raises(ValueError):
        oracle.flatten_layout([3, -1], 2)
    with pytest.raises(ValueError):
        oracle.flatten_layout([3], 0)
    assert oracle.shard_of(10, 3, 10) == -1 and oracle.shard_of(10, 3, -1) == -1
