"""Pins of the oracle's unshard/reshard copies, clip norm and overflow check (no GPU).

Unshard ("FSDP: Fully Sharded Data Parallel Training at Scale", the FSDP unit
communication cycle): the all-gather leaves every GPU with the concatenation
of the N shards in rank order -- pinned against numpy's concatenate and the
round trip. Clipping (same page, gradient clipping section): the norm is the
norm of the whole gradient across all shards -- pinned against
torch.nn.utils.clip_grad_norm_, the routine the page names.
"""
import math

import numpy as np
import pytest
import torch

import oracle


@pytest.mark.parametrize("P,N", [(0, 3), (1, 4), (2, 5), (1000, 7), (4099, 64), (123457, 8)])
@pytest.mark.parametrize("dt", [np.uint16, np.float32])
def test_unshard_is_concatenation(P, N, dt):
    rng = np.random.default_rng(P + N)
    _, b = oracle.flatten_layout([P], N)
    shards = [rng.integers(0, 1 << 16, size=int(b[k + 1] - b[k])).astype(dt) for k in range(N)]
    flat = oracle.unshard(shards, b)
    assert np.array_equal(flat, np.concatenate(shards) if P else np.zeros(0, dt))
    back = oracle.reshard(flat, b)
    assert all(np.array_equal(x, y) for x, y in zip(back, shards))


def test_reshard_then_unshard_identity():
    rng = np.random.default_rng(1)
    flat = rng.integers(0, 1 << 16, size=100003).astype(np.uint16)
    for N in (1, 3, 64):
        _, b = oracle.flatten_layout([flat.size], N)
        assert np.array_equal(oracle.unshard(oracle.reshard(flat, b), b), flat)


def test_sumsq_closed_forms():
    assert oracle.sumsq(np.full(1000, 0.5, np.float32)) == 250.0
    assert oracle.sumsq(np.zeros(10, np.float32)) == 0.0
    rng = np.random.default_rng(2)
    g = (rng.standard_normal(100000) * 1e-3).astype(np.float32)
    exact = math.fsum((g.astype(np.float64)) ** 2)          # every square is exact in double
    assert oracle.sumsq(g) == pytest.approx(exact, rel=1e-13)
    # sharded: the sum of shard contributions is the whole norm
    _, b = oracle.flatten_layout([g.size], 8)
    parts = sum(oracle.sumsq(g[b[k]:b[k + 1]]) for k in range(8))
    assert parts == pytest.approx(exact, rel=1e-13)


@pytest.mark.parametrize("max_norm", [1e-3, 0.05, 1.0, 1e6])
def test_clip_coef_matches_clip_grad_norm(max_norm):
    rng = np.random.default_rng(3)
    gs = [(rng.standard_normal(s) * 1e-3).astype(np.float32) for s in (1000, 337, 4096)]
    params = []
    for g in gs:
        p = torch.zeros(g.size, requires_grad=True)
        p.grad = torch.from_numpy(g.copy())
        params.append(p)
    total = torch.nn.utils.clip_grad_norm_(params, max_norm)
    tot_sq = sum(oracle.sumsq(g) for g in gs)
    assert math.sqrt(tot_sq) == pytest.approx(float(total), rel=1e-6)
    c = oracle.clip_coef(tot_sq, max_norm)
    ref_c = min(1.0, max_norm / (float(total) + 1e-6))
    assert c == pytest.approx(ref_c, rel=1e-6)
    for g, p in zip(gs, params):
        np.testing.assert_allclose(g * np.float32(c), p.grad.numpy(), rtol=2e-6, atol=0)


def test_all_finite():
    g = np.zeros(100, np.float32)
    assert oracle.all_finite(g)
    for bad in (np.inf, -np.inf, np.nan):
        h = g.copy()
        h[57] = bad
        assert not oracle.all_finite(h)
    assert oracle.all_finite(np.float32([3.4e38, -3.4e38, 1e-45]))
