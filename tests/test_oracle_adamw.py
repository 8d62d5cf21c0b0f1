"""Pins of the oracle's AdamW step (no GPU).

Pages: "FSDP: Fully Sharded Data Parallel Training at Scale" -- Adam keeps an
exponential moving average of the gradient and of its square in fp32 next to
an fp32 master copy; each GPU steps its own shard. The update equation is not
printed; the reading is Adam with bias correction and decoupled weight decay
(AdamW), eps added after the square root of the corrected second moment.

Pins (consequences of that reading, not a retyping of the recurrence):
  * first step from zero moments: update = lr * g / (|g| + eps) plus decay;
  * zero gradients: m = v = 0 and p_t = p_0 (1 - lr wd)^t;
  * a constant gradient c: m_t = (1 - b1^t) c, v_t = (1 - b2^t) c^2 and every
    step moves p by lr c / (|c| + eps) (bias correction is exact);
  * scaling every gradient by 2^k with eps = 0 leaves the trajectory unchanged;
  * Kingma & Ba's bound |step| <= lr (1 - b1) / sqrt(1 - b2);
  * the two-step expansion of the moments;
  * grad_scale multiplies g once; the 16-bit output is the rounded master.
"""
import math

import numpy as np
import pytest

import oracle

F = np.float32
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def f32(x):
    return float(np.float32(x))


def run(hp, steps, gs, p0, m0=None, v0=None, t0=1, grad_scale=1.0):
    p = np.array(p0, dtype=F)
    m = np.zeros_like(p) if m0 is None else np.array(m0, dtype=F)
    v = np.zeros_like(p) if v0 is None else np.array(v0, dtype=F)
    for s in range(steps):
        oracle.adamw(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], t0 + s,
                     np.ascontiguousarray(gs[s], dtype=F), p, m, v, grad_scale=grad_scale)
    return p, m, v


def ulps(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    sp = np.spacing(np.abs(b).astype(F)).astype(np.float64)
    return np.abs(a - b) / np.maximum(sp, 1e-45)


def test_first_step_sign_like():
    rng = np.random.default_rng(0)
    n = 20000
    g = (rng.standard_normal(n) * 10.0 ** rng.integers(-9, 1, size=n)).astype(F)
    p0 = (rng.standard_normal(n) * 0.02).astype(F)
    p, m, v = run(HP, 1, [g], p0)
    lr, wd, eps = f32(HP["lr"]), f32(HP["weight_decay"]), f32(HP["eps"])
    gd = g.astype(np.float64)
    expect_p = p0.astype(np.float64) * (1 - lr * wd) - lr * gd / (np.abs(gd) + eps)
    assert ulps(p, expect_p).max() <= 1.0
    b1, b2 = f32(HP["beta1"]), f32(HP["beta2"])
    assert ulps(m, (1 - b1) * gd).max() <= 1.0
    assert ulps(v, (1 - b2) * gd * gd).max() <= 1.0


def test_zero_gradient_pure_decay():
    rng = np.random.default_rng(1)
    p0 = (rng.standard_normal(5000) * 0.02).astype(F)
    T = 20
    p, m, v = run(HP, T, [np.zeros(5000, F)] * T, p0)
    assert (m == 0).all() and (v == 0).all()
    d = 1 - f32(HP["lr"]) * f32(HP["weight_decay"])
    expect = p0.astype(np.float64) * d ** T
    assert ulps(p, expect).max() <= T
    assert (np.abs(p) <= np.abs(p0)).all()          # decay shrinks, never grows


@pytest.mark.parametrize("c", [3e-3, -2.5e-5, 1.0, -7.0])
def test_constant_gradient_closed_form(c):
    rng = np.random.default_rng(2)
    n, T = 2000, 12
    p0 = (rng.standard_normal(n) * 0.02).astype(F)
    cf = f32(c)
    g = np.full(n, cf, dtype=F)
    p, m, v = run(HP, T, [g] * T, p0)
    b1, b2, lr, wd, eps = (f32(HP[k]) for k in ("beta1", "beta2", "lr", "weight_decay", "eps"))
    assert ulps(m, (1 - b1 ** T) * cf).max() <= T
    assert ulps(v, (1 - b2 ** T) * cf * cf).max() <= 2 * T
    d = 1 - lr * wd
    u = lr * cf / (abs(cf) + eps)
    expect = p0.astype(np.float64) * d ** T - u * (1 - d ** T) / (1 - d)
    err = np.abs(p.astype(np.float64) - expect)
    # rounding errors are made while |p| is as large as max(|p0|, |p_T|); allow a few per step
    scale = np.maximum(np.abs(p0).astype(np.float64), np.abs(expect))
    assert (err <= 4 * T * np.spacing(scale.astype(F)).astype(np.float64)).all()


def test_gradient_scale_invariance_eps0():
    rng = np.random.default_rng(3)
    n, T = 4000, 6
    hp = dict(HP, eps=0.0)
    gs = [(rng.standard_normal(n) * 1e-3).astype(F) for _ in range(T)]
    p0 = (rng.standard_normal(n) * 0.02).astype(F)
    pa, _, _ = run(hp, T, gs, p0)
    pb, mb, vb = run(hp, T, [g * F(2.0 ** 10) for g in gs], p0)
    pc, _, _ = run(hp, T, [g * F(2.0 ** -12) for g in gs], p0)
    assert np.array_equal(pa, pb) and np.array_equal(pa, pc)


def test_step_size_bound():
    rng = np.random.default_rng(4)
    n, T = 5000, 30
    hp = dict(HP, weight_decay=0.0)
    p = (rng.standard_normal(n) * 0.02).astype(F)
    m = np.zeros(n, F)
    v = np.zeros(n, F)
    lr = f32(hp["lr"])
    bound = lr * (1 - f32(hp["beta1"])) / math.sqrt(1 - f32(hp["beta2"]))
    for t in range(1, T + 1):
        g = (rng.standard_normal(n) * 10.0 ** rng.integers(-6, 1, size=n)).astype(F)
        before = p.astype(np.float64)
        oracle.adamw(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], 0.0, t, g, p, m, v)
        assert (np.abs(p - before) <= bound * (1 + 1e-6) + 1e-12).all()
        assert (v >= 0).all()


def test_two_step_expansion():
    rng = np.random.default_rng(5)
    n = 3000
    g1 = (rng.standard_normal(n) * 1e-3).astype(F)
    g2 = (rng.standard_normal(n) * 1e-3).astype(F)
    p0 = (rng.standard_normal(n) * 0.02).astype(F)
    p, m, v = run(HP, 2, [g1, g2], p0)
    b1, b2 = f32(HP["beta1"]), f32(HP["beta2"])
    G1, G2 = g1.astype(np.float64), g2.astype(np.float64)
    m2 = b1 * (1 - b1) * G1 + (1 - b1) * G2
    v2 = b2 * (1 - b2) * G1 ** 2 + (1 - b2) * G2 ** 2
    # m may cancel: measure in ulps of the larger term (v has no cancellation)
    mscale = np.maximum(np.abs(b1 * (1 - b1) * G1), np.abs((1 - b1) * G2))
    assert (np.abs(m - m2) <= 2 * np.spacing(mscale.astype(F)).astype(np.float64)).all()
    assert ulps(v, v2).max() <= 2


def test_bias_correction_vanishes_late():
    rng = np.random.default_rng(6)
    n = 3000
    g = (rng.standard_normal(n) * 1e-3).astype(F)
    m0 = (rng.standard_normal(n) * 1e-4).astype(F)
    v0 = np.abs(rng.standard_normal(n) * 1e-8).astype(F)
    p0 = (rng.standard_normal(n) * 0.02).astype(F)
    hp = dict(HP, lr=3e-4, weight_decay=0.1)
    p, m, v = run(hp, 1, [g], p0, m0, v0, t0=100000)
    lr, wd, eps, b1, b2 = (f32(hp[k]) for k in ("lr", "weight_decay", "eps", "beta1", "beta2"))
    M = b1 * m0.astype(np.float64) + (1 - b1) * g.astype(np.float64)
    V = b2 * v0.astype(np.float64) + (1 - b2) * g.astype(np.float64) ** 2
    expect = p0.astype(np.float64) * (1 - lr * wd) - lr * M / (np.sqrt(V) + eps)   # (1 - b^t) == 1 here
    assert ulps(p, expect).max() <= 1.0


def test_grad_scale_and_p16():
    rng = np.random.default_rng(7)
    n = 4000
    g = (rng.standard_normal(n) * 1e-3).astype(F)
    p0 = (rng.standard_normal(n) * 0.02).astype(F)
    pa, ma, va = run(HP, 1, [g * F(0.25)], p0)
    pb, mb, vb = run(HP, 1, [g], p0, grad_scale=0.25)
    assert np.array_equal(pa, pb) and np.array_equal(ma, mb) and np.array_equal(va, vb)
    p = p0.copy()
    m = np.zeros(n, F)
    v = np.zeros(n, F)
    for dt in (oracle.BF16, oracle.FP16):
        p16 = oracle.adamw(HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["weight_decay"], 1, g, p, m, v,
                           p16_dtype=dt)
        assert np.array_equal(p16, oracle.round16(p, dt))


def test_invalid_step():
    z = np.zeros(4, F)
    with pytest.raises(ValueError):
        oracle.adamw(1e-3, 0.9, 0.999, 1e-8, 0.0, 0, z, z.copy(), z.copy(), z.copy())
