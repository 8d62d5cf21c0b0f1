"""Pins of the oracle's virtual-rank gradient reduce (no GPU).

Pages: "FSDP: Fully Sharded Data Parallel Training at Scale" -- the backward
reduce-scatter sums the ranks' gradients and gives each GPU its shard's part;
the mixed-precision section fixes the accumulation type to fp32. Reading: the
sum is taken in rank order 0..N-1 starting from rank 0's value.

Pins: rank-order probes whose result differs under any other order, exact
sums (all partial sums representable), N*c for equal inputs, the classic
recursive-summation error bound against an exactly rounded reference
(math.fsum), signed zero and non-finite propagation.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def bf16_bits(x) -> np.ndarray:
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def fp16_bits(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def test_rank_order_probes():
    big = 2.0 ** 27
    # order 0,1,2: (2^27 + 1) rounds to 2^27, minus 2^27 -> 0 ; order 0,2,1 would give 1
    r = oracle.grad_reduce([bf16_bits([big]), bf16_bits([1.0]), bf16_bits([-big])], oracle.BF16)
    assert r[0] == 0.0
    # order 0,1,2 on (1, 2^27, -2^27) gives 0 ; the reverse order 2,1,0 would give 1
    r = oracle.grad_reduce([bf16_bits([1.0]), bf16_bits([big]), bf16_bits([-big])], oracle.BF16)
    assert r[0] == 0.0
    r = oracle.grad_reduce([bf16_bits([big]), bf16_bits([-big]), bf16_bits([1.0])], oracle.BF16)
    assert r[0] == 1.0


@pytest.mark.parametrize("N", [1, 2, 4, 8, 64])
def test_equal_inputs_power_of_two(N):
    rng = np.random.default_rng(N)
    c = rng.standard_normal(1000).astype(np.float32)
    bits = bf16_bits(c)
    vals = oracle.widen16(bits, oracle.BF16)
    r = oracle.grad_reduce([bits] * N, oracle.BF16)
    assert np.array_equal(r, vals * np.float32(N))


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_exact_integer_sums(dtype):
    rng = np.random.default_rng(3)
    N, n = 64, 5000
    ints = rng.integers(-256, 257, size=(N, n))
    conv = bf16_bits if dtype == oracle.BF16 else fp16_bits
    r = oracle.grad_reduce([conv(ints[k]) for k in range(N)], dtype)
    assert np.array_equal(r, ints.sum(axis=0).astype(np.float32))


def test_fp16_subnormal_sums_exact():
    # multiples of 2^-24 (fp16 subnormals) sum exactly in fp32
    rng = np.random.default_rng(4)
    N, n = 64, 4000
    k = rng.integers(-1023, 1024, size=(N, n))
    bits = [np.where(k[r] < 0, 0x8000 | (-k[r]), k[r]).astype(np.uint16) for r in range(N)]
    r = oracle.grad_reduce(bits, oracle.FP16)
    assert np.array_equal(r, (k.sum(axis=0) * 2.0 ** -24).astype(np.float32))


@pytest.mark.parametrize("N", [2, 8, 64])
def test_error_bound_vs_exact(N):
    rng = np.random.default_rng(10 + N)
    n = 3000
    x = (rng.standard_normal((N, n)) * 10.0 ** rng.integers(-4, 3, size=(N, 1))).astype(np.float32)
    bits = [bf16_bits(x[r]) for r in range(N)]
    vals = np.stack([oracle.widen16(b, oracle.BF16).astype(np.float64) for b in bits])
    r = oracle.grad_reduce(bits, oracle.BF16).astype(np.float64)
    u = 2.0 ** -24
    for i in range(n):
        exact = math.fsum(vals[:, i])
        bound = (N - 1) * u * math.fsum(np.abs(vals[:, i])) * (1 + 2 * N * u)
        assert abs(r[i] - exact) <= bound + 1e-45


def test_post_scale_and_accumulate():
    rng = np.random.default_rng(7)
    ints = rng.integers(-100, 101, size=(8, 1000))
    bits = [bf16_bits(ints[k]) for k in range(8)]
    s = ints.sum(axis=0)
    r = oracle.grad_reduce(bits, oracle.BF16, post_scale=0.125)          # power of two: exact
    assert np.array_equal(r, (s * 0.125).astype(np.float32))
    r3 = oracle.grad_reduce(bits, oracle.BF16, post_scale=1.0 / 3.0)     # one fp32 rounding of sum * fl(1/3)
    assert np.array_equal(r3, (s.astype(np.float32) * np.float32(1.0 / 3.0)).astype(np.float32))
    base = rng.integers(-1000, 1001, size=1000).astype(np.float32)
    acc = base.copy()
    oracle.grad_reduce(bits, oracle.BF16, accumulate_into=acc)
    assert np.array_equal(acc, (base + s).astype(np.float32))


def test_signed_zero_and_nonfinite():
    nz = bf16_bits([-0.0])
    pz = bf16_bits([0.0])
    r = oracle.grad_reduce([nz, nz, nz], oracle.BF16)
    assert r[0] == 0 and np.signbit(r[0])
    r = oracle.grad_reduce([nz, pz], oracle.BF16)
    assert r[0] == 0 and not np.signbit(r[0])
    inf, ninf, nan = bf16_bits([np.inf]), bf16_bits([-np.inf]), bf16_bits([np.nan])
    assert np.isnan(oracle.grad_reduce([inf, ninf], oracle.BF16)[0])
    assert np.isinf(oracle.grad_reduce([inf, pz], oracle.BF16)[0])
    assert np.isnan(oracle.grad_reduce([pz, nan, pz], oracle.BF16)[0])
    # bf16 max + bf16 max overflows fp32? no: 2 * 3.39e38 > fp32 max -> inf
    big = bf16_bits([3.3895314e38])
    assert np.isinf(oracle.grad_reduce([big, big], oracle.BF16)[0])


def test_single_rank_is_widening():
    rng = np.random.default_rng(9)
    b = rng.integers(0, 1 << 16, size=5000).astype(np.uint16)
    r = oracle.grad_reduce([b], oracle.FP16)
    w = oracle.widen16(b, oracle.FP16)
    assert np.array_equal(np.isnan(r), np.isnan(w))
    assert np.array_equal(r[~np.isnan(r)], w[~np.isnan(w)])
