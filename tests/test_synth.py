"""The seeded input generator: determinism, views, distributions and formats (no GPU)."""
import numpy as np

import synth
from synth import workloads


def f32(bits):
    return bits.view(np.float32)


def bf(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_deterministic_and_range_gather_agree():
    s = synth.normal(1e-3, synth.BF16, synth.GRAD, rank=5, step=3)
    a = synth.host_range(s, 1000, 50000)
    b = synth.host_range(s, 1000, 50000)
    assert np.array_equal(a, b)
    idx = np.array([1000, 1001, 25000, 50999])
    assert np.array_equal(synth.host_gather(s, idx), a[idx - 1000])


def test_streams_differ_and_are_uncorrelated():
    a = bf(synth.host_range(synth.normal(1e-3, synth.BF16, synth.GRAD, 0, 1), 0, 200000)).astype(np.float64)
    b = bf(synth.host_range(synth.normal(1e-3, synth.BF16, synth.GRAD, 1, 1), 0, 200000)).astype(np.float64)
    c = bf(synth.host_range(synth.normal(1e-3, synth.BF16, synth.GRAD, 0, 2), 0, 200000)).astype(np.float64)
    assert abs(np.corrcoef(a, b)[0, 1]) < 0.01 and abs(np.corrcoef(a, c)[0, 1]) < 0.01


def test_normal_moments():
    x = f32(synth.host_range(synth.normal(0.02, synth.FP32, synth.MASTER), 0, 1 << 20)).astype(np.float64)
    assert abs(x.mean()) < 0.02 * 0.01
    assert abs(x.std() / 0.02 - 1) < 0.01
    assert np.abs(x).max() <= 6 * 0.02                 # Irwin-Hall support
    kurt = ((x - x.mean()) ** 4).mean() / x.var() ** 2
    assert abs(kurt - 2.9) < 0.05                      # sum of 12 uniforms: kurtosis 3 - 1.2/12


def test_irwin_hall_integer_exact():
    # the centred integer has the stated range and parity
    vals = [synth.irwin_hall_at(0, 77, i) for i in range(2000)]
    m21 = (1 << 21) - 1
    assert all(abs(v) <= 12 * m21 and v % 2 == 0 for v in vals)


def test_abs_normal_and_uniform():
    v = f32(synth.host_range(synth.normal(1e-8, synth.FP32, synth.MOM2, absolute=True), 0, 100000))
    assert (v >= 0).all() and abs(v.mean() / (1e-8 * np.sqrt(2 / np.pi)) - 1) < 0.02
    u = synth.host_range(synth.uniform(6e-5, synth.FP16, synth.GRAD, 3, 1), 0, 1 << 20)
    uf = u.view(np.float16).astype(np.float64)
    assert ((u & 0x7C00) == 0).all()                  # every value is an fp16 subnormal (or zero)
    assert np.abs(uf).max() < 6e-5 and abs(uf.std() / (6e-5 / np.sqrt(3)) - 1) < 0.01


def test_outliers_fraction():
    s = synth.normal(1e-4, synth.BF16, synth.GRAD, 2, 1, outlier_every=100, outlier_mult=100.0)
    x = np.abs(bf(synth.host_range(s, 0, 1 << 20)))
    frac = (x > 6.01e-4).mean()                          # only outliers exceed 6 sigma
    assert 0.0085 < frac < 0.0105                        # ~1% drawn at 100x, ~95% of those beyond 6 sigma


def test_values_sit_on_target_grid():
    b = synth.host_range(synth.normal(1e-3, synth.BF16, synth.GRAD), 0, 10000)
    x = bf(b)
    # bf16 value widened and re-truncated is unchanged; fp32 -> bf16 truncation toward zero never grows |x|
    assert np.array_equal((x.view(np.uint32) >> 16).astype(np.uint16), b)
    xs = f32(synth.host_range(synth.normal(1e-3, synth.FP32, synth.GRAD), 0, 10000))
    assert (np.abs(bf((xs.view(np.uint32) >> 16).astype(np.uint16))) <= np.abs(xs)).all()


def test_workload_recipes():
    w = workloads.gpt2_small()
    assert w.n_ranks == 8 and w.P == 124_439_808 and w.warmup_steps == 5 and w.steps == 10
    w = workloads.sweep(4099, 64)
    _, = [w.P // w.n_ranks]
    assert w.P == 4099 * 64 and w.first_step == 1000
