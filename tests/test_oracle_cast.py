"""Pins of the oracle's 16-bit formats (no GPU).

Page: "FSDP: Fully Sharded Data Parallel Training at Scale", mixed-precision
section: bf16 has fp32's 8-bit exponent and 7 mantissa bits; fp16 has a
5-bit exponent (largest finite 65504) and 10 mantissa bits. The working
parameters are the master weights rounded to 16 bits; the rounding mode is
not printed, so round-to-nearest-even (the IEEE default) is the reading.

Pins: every one of the 2^32 fp32 bit patterns against the library
conversions (torch CPU casts, round-to-nearest-even; numpy agrees on a sample),
and a structured subset against an independent nearest-value search over all
finite 16-bit values. Widening is checked on all 2^16 patterns.
"""
import numpy as np
import pytest
import torch

import oracle

CHUNK = 1 << 24


def _all_f32_chunks():
    buf = np.arange(CHUNK, dtype=np.uint32)
    step = np.uint32(CHUNK)
    for c in range((1 << 32) // CHUNK):
        yield buf.view(np.float32)
        buf += step


def _canon(bits: np.ndarray, dtype) -> np.ndarray:
    """Bit patterns with every NaN replaced by one canonical pattern (NaN payloads may differ)."""
    exp, man = (0x7F80, 0x007F) if dtype == oracle.BF16 else (0x7C00, 0x03FF)
    nan = ((bits & exp) == exp) & ((bits & man) != 0)
    return np.where(nan, np.uint16(0x7FFF), bits)


def _same(a_bits: np.ndarray, b_bits: np.ndarray, dtype) -> bool:
    if np.array_equal(a_bits, b_bits):
        return True
    return bool(np.array_equal(_canon(a_bits, dtype), _canon(b_bits, dtype)))


@pytest.mark.slow
def test_bf16_rounding_exhaustive_vs_torch():
    for x in _all_f32_chunks():
        ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        got = oracle.round16(x, oracle.BF16)
        assert _same(got, ref, oracle.BF16)


@pytest.mark.slow
def test_fp16_rounding_exhaustive_vs_torch():
    with np.errstate(over="ignore", invalid="ignore"):
        for x in _all_f32_chunks():
            ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
            got = oracle.round16(x, oracle.FP16)
            assert _same(got, ref, oracle.FP16)


def _all_finite16(dtype):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.widen16(bits, dtype).astype(np.float64)
    keep = np.isfinite(vals) & ~((vals == 0) & (bits >= 0x8000))   # one zero, no NaN/inf
    order = np.argsort(vals[keep], kind="stable")
    return vals[keep][order], bits[keep][order]


def _nearest_search(x: np.ndarray, dtype) -> np.ndarray:
    """Independent rounding: nearest finite 16-bit value by search, ties to the even pattern."""
    vals, bits = _all_finite16(dtype)
    top, top_bits = vals[-1], bits[-1]
    ulp_top = top - vals[-2]
    xd = x.astype(np.float64)
    j = np.clip(np.searchsorted(vals, xd, side="left"), 1, len(vals) - 1)
    lo, hi = vals[j - 1], vals[j]
    lob, hib = bits[j - 1], bits[j]
    exact_hi = xd == hi
    dlo, dhi = xd - lo, hi - xd
    pick_hi = exact_hi | (dhi < dlo) | ((dhi == dlo) & ((hib & 1) == 0))
    out = np.where(pick_hi, hib, lob).astype(np.uint16)
    inf_bits = np.uint16(0x7F80 if dtype == oracle.BF16 else 0x7C00)
    over = np.abs(xd) >= top + ulp_top / 2           # beyond the last rounding boundary
    out = np.where(over, np.where(xd > 0, inf_bits, inf_bits | np.uint16(0x8000)), out)
    # signed zero: negative inputs that round to zero keep their sign
    negz = (out == 0) & (np.signbit(x))
    out = np.where(negz, np.uint16(0x8000), out)
    return out.astype(np.uint16)


def _structured_f32():
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xC000, 0xFFFF], dtype=np.uint32)
    rng = np.random.default_rng(5)
    parts = [(hi[:, None] | lows[None, :]).ravel(), rng.integers(0, 1 << 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)]
    x = np.concatenate(parts).view(np.float32)
    return x[np.isfinite(x)]


def _midpoints(dtype):
    vals, _ = _all_finite16(dtype)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)         # exact in fp32 for these formats
    near = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf))])
    return np.concatenate([near, -near])


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_rounding_vs_independent_search(dtype):
    x = np.concatenate([_structured_f32(), _midpoints(dtype)])
    if dtype == oracle.FP16:
        x = np.concatenate([x, np.float32([65504, 65519.99, 65520, 65536, 1e-8, 2.0**-25, 2.0**-24 * 1.5])])
    got = oracle.round16(x, dtype)
    ref = _nearest_search(x, dtype)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_widen_exhaustive():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f16 = oracle.widen16(bits, oracle.FP16)
    ref16 = bits.view(np.float16).astype(np.float32)
    assert np.array_equal(np.isnan(f16), np.isnan(ref16))
    ok = ~np.isnan(ref16)
    assert np.array_equal(f16[ok].view(np.uint32), ref16[ok].view(np.uint32))
    bf = oracle.widen16(bits, oracle.BF16)
    refb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(bf.view(np.uint32)[~np.isnan(bf)], refb.view(np.uint32)[~np.isnan(refb)])


def test_rounding_special_cases():
    x = np.float32([0.0, -0.0, np.inf, -np.inf, np.nan, 65504, 65520, -65520, 3.4028235e38, 1.0 + 2**-8])
    b16 = oracle.round16(x, oracle.BF16)
    h16 = oracle.round16(x, oracle.FP16)
    assert b16[0] == 0 and b16[1] == 0x8000 and b16[2] == 0x7F80 and b16[3] == 0xFF80
    assert (b16[4] & 0x7F80) == 0x7F80 and (b16[4] & 0x7F)
    assert h16[5] == 0x7BFF and h16[6] == 0x7C00 and h16[7] == 0xFC00
    assert b16[8] == 0x7F80           # fp32 max rounds past the largest bf16 to infinity
    assert b16[9] == 0x3F80           # 1 + 2^-8 is a tie: rounds to even (1.0)


def test_fp16_library_routines_agree_on_sample():
    # numpy's float16 cast is a second library implementation of the same rounding
    rng = np.random.default_rng(11)
    x = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32).view(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert _same(oracle.round16(x, oracle.FP16), ref, oracle.FP16)
