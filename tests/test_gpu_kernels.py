"""GPU edge cases of each kernel through the C ABI, against the oracle.

Reduce: bit-exact for any rank count (1..1024), ragged lengths, both 16-bit
formats, misaligned views (element-wise kernel), post_scale, accumulation and
the non-finite flag; a rank-order probe. AdamW: misaligned views and odd
lengths, the fp32-gradient entry, the optional outputs and device-side
controls (g_out, non-finite flag, gradient scale, skip flag). Unshard/reshard:
bit-exact for empty shards, P < N, odd offsets (shifted-source path), fp32,
and N = 1024.
"""
import numpy as np
import pytest

import oracle
import synth

from parity import assert_p16_within_ulp, assert_state_close

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=3)


@pytest.fixture(scope="module")
def ss():
    import fsdp_sharded_mixed_ss_gb300 as m
    return m


def tdt(fmt):
    import torch
    return {synth.BF16: torch.bfloat16, synth.FP16: torch.float16}[fmt]


def dev_bits(spec, n, offset=0, pad=0):
    """Device buffer of n generated elements, viewed `offset` elements into a larger allocation."""
    import torch
    dt = torch.float32 if spec.fmt == synth.FP32 else tdt(spec.fmt)
    base = torch.zeros(n + offset + pad, dtype=dt, device="cuda")
    view = base[offset:offset + n]
    if n:
        synth.device_fill(spec, view.view(torch.int32 if spec.fmt == synth.FP32 else torch.int16))
    return view


def host_bits(spec, n):
    return synth.host_range(spec, 0, n)


def bits_of(t):
    import torch
    if t.dtype == torch.float32:
        return t.cpu().numpy()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


# ----------------------------------------------------------------------------- reduce

@pytest.mark.parametrize("N", [1, 2, 3, 4, 8, 64, 65, 1024])
@pytest.mark.parametrize("fmt", [synth.BF16, synth.FP16])
def test_reduce_bit_exact(ss, N, fmt):
    import torch
    n = 4099 if N < 1000 else 1000
    specs = [synth.normal(1e-3, fmt, synth.GRAD, r, 1) if fmt == synth.BF16 else synth.uniform(6e-5, fmt, synth.GRAD, r, 1)
             for r in range(N)]
    G = [dev_bits(s, n) for s in specs]
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    ss.ss_grad_reduce(G, n, out)
    ref = oracle.grad_reduce([host_bits(s, n) for s in specs], fmt)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("offsets", [(0, 0), (1, 0), (0, 1), (3, 5), (7, 7)])
def test_reduce_views_scale_accumulate_flag(ss, offsets):
    import torch
    go, oo = offsets
    N, n = 8, 100_003
    specs = [synth.normal(1e-3, synth.BF16, synth.GRAD, r, 2) for r in range(N)]
    G = [dev_bits(s, n, offset=go) for s in specs]
    base = torch.zeros(n + oo, dtype=torch.float32, device="cuda")
    out = base[oo:]
    init = dev_bits(synth.normal(1e-2, synth.FP32, synth.MOM1), n)
    out.copy_(init)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ss.ss_grad_reduce(G, n, out, post_scale=0.125, accumulate=True, nonfinite_flag=flag)
    acc = bits_of(init).copy()
    oracle.grad_reduce([host_bits(s, n) for s in specs], synth.BF16, post_scale=0.125, accumulate_into=acc)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), acc.view(np.uint32))
    assert flag.item() == 0
    G[5][n // 2] = float("inf")
    ss.ss_grad_reduce(G, n, out, nonfinite_flag=flag)
    assert flag.item() == 1


@pytest.mark.parametrize("N,n", [(1, 27), (1, 300_007), (2, 1001), (2, 300_007), (3, 300_007), (4, 1001),
                                 (4, 300_007), (5, 300_007), (7, 300_007), (8, 27), (8, 300_007), (9, 1001),
                                 (9, 300_007), (64, 1001), (64, 300_007), (1024, 27), (1024, 1001)])
@pytest.mark.parametrize("accumulate", [True, False])
def test_reduce_shifted_loads(ss, N, n, accumulate):
    """Every rank's view 3 elements into its buffer, the output aligned: the warp-cooperative
    shifted reduce (runs of 31 groups; 1-4 ranks several runs a warp at a time, 7-8 ranks
    double-buffered, the others in batches of rank chunks), with a post scale, accumulating or
    not (separate kernel instances), from a 1-group body (n = 27) up; bit-exact against the
    oracle, both rank tables."""
    import torch
    specs = [synth.normal(1e-3, synth.BF16, synth.GRAD, r, 6) for r in range(N)]
    G = [dev_bits(s, n, offset=3) for s in specs]
    init = dev_bits(synth.normal(1e-2, synth.FP32, synth.MOM1), n)
    out = init.clone()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ss.ss_grad_reduce(G, n, out, post_scale=0.5, accumulate=accumulate, nonfinite_flag=flag)
    acc = bits_of(init).copy() if accumulate else None
    ref = oracle.grad_reduce([host_bits(s, n) for s in specs], synth.BF16, post_scale=0.5, accumulate_into=acc)
    ref = acc if accumulate else ref
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert flag.item() == 0


@pytest.mark.parametrize("N", [2, 3, 8, 9, 65])
def test_reduce_mixed_phases_some_aligned(ss, N):
    """Rank r's view r % 8 elements into its buffer: rank 0 (and 8, 16, ...) at the output's phase,
    the others each at its own -- the warp-cooperative mixed-phase reduce with some ranks needing no
    shift; bit-exact against the oracle, accumulating with a post scale."""
    import torch
    n = 200_003
    specs = [synth.normal(1e-3, synth.BF16, synth.GRAD, r, 9) for r in range(N)]
    G = [dev_bits(s, n, offset=r % 8) for r, s in enumerate(specs)]
    init = dev_bits(synth.normal(1e-2, synth.FP32, synth.MOM1), n)
    out = init.clone()
    ss.ss_grad_reduce(G, n, out, post_scale=0.5, accumulate=True)
    acc = bits_of(init).copy()
    oracle.grad_reduce([host_bits(s, n) for s in specs], synth.BF16, post_scale=0.5, accumulate_into=acc)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), acc.view(np.uint32))


@pytest.mark.parametrize("N", [2, 3, 4, 5, 7, 8, 9, 16, 64, 65])
@pytest.mark.parametrize("n", [1001, 300_007])
@pytest.mark.parametrize("accumulate", [True, False])
def test_reduce_mixed_phases(ss, N, n, accumulate):
    """Rank r's view (r % 7) + 1 elements into its buffer (every rank at its own phase), the
    output aligned: each rank's packed chunk moved into place by its own phase before the
    rank-ordered fp32 add, in every form (several runs at a time for 2-4 ranks, double-buffered
    for 7-8, batches of rank chunks otherwise; 65 ranks the large rank table); fp16, bit-exact
    against the oracle, with the non-finite flag raised by one rank's infinity."""
    import torch
    specs = [synth.uniform(6e-5, synth.FP16, synth.GRAD, r, 8) for r in range(N)]
    G = [dev_bits(s, n, offset=(r % 7) + 1) for r, s in enumerate(specs)]
    init = dev_bits(synth.normal(1e-2, synth.FP32, synth.MOM1), n)
    out = init.clone()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ss.ss_grad_reduce(G, n, out, post_scale=0.25, accumulate=accumulate, nonfinite_flag=flag)
    acc = bits_of(init).copy() if accumulate else None
    ref = oracle.grad_reduce([host_bits(s, n) for s in specs], synth.FP16, post_scale=0.25, accumulate_into=acc)
    ref = acc if accumulate else ref
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert flag.item() == 0
    G[N - 1][n // 3] = float("inf")
    ss.ss_grad_reduce(G, n, out, nonfinite_flag=flag)
    assert flag.item() == 1


@pytest.mark.parametrize("N,accumulate,runs_per_sm", [(8, False, 16), (5, False, 32), (4, False, 64), (3, True, 32),
                                                      (2, True, 64), (1, False, 128), (1, True, 64)])
@pytest.mark.parametrize("k,d", [(1, -1), (1, 0), (1, 1), (2, 5)])
def test_reduce_shifted_run_boundaries(ss, N, accumulate, runs_per_sm, k, d):
    """The shifted reduce's grid passes over SMs x 16 warps x 1 run (7-8 ranks, double-buffered),
    SMs x 32 warps x U runs (1-4 ranks, U runs a warp at a time: U = 4 for one rank, else 2;
    accumulating 2 up to 2 ranks, else 1) or SMs x 32 warps x 1 run (other rank counts), runs of 31
    groups; bodies of just a whole number of passes, or one run more or less: bit-exact, so every
    run is taken once."""
    import torch
    runs = k * _sms() * runs_per_sm + d
    n = (runs * 31 + 2) * 8 + 5
    specs = [synth.normal(1e-3, synth.FP16, synth.GRAD, r, 7) for r in range(N)]
    G = [dev_bits(s, n, offset=5) for s in specs]
    init = dev_bits(synth.normal(1e-2, synth.FP32, synth.MOM1), n)
    out = init.clone()
    ss.ss_grad_reduce(G, n, out, accumulate=accumulate)
    acc = bits_of(init).copy() if accumulate else None
    ref = oracle.grad_reduce([host_bits(s, n) for s in specs], synth.FP16, accumulate_into=acc)
    ref = acc if accumulate else ref
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_reduce_rank_order_probe(ss):
    import torch
    vals = torch.tensor([2.0 ** 27, 1.0, -2.0 ** 27], dtype=torch.bfloat16, device="cuda")
    n = 40
    G = [torch.full((n,), float(v), dtype=torch.bfloat16, device="cuda") for v in vals.float().tolist()]
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    ss.ss_grad_reduce(G, n, out)
    assert (out == 0).all()
    ss.ss_grad_reduce([G[0], G[2], G[1]], n, out)
    assert (out == 1).all()


# ----------------------------------------------------------------------------- AdamW step

def _state(n, off=0):
    return (dev_bits(synth.normal(0.02, synth.FP32, synth.MASTER), n, off),
            dev_bits(synth.normal(1e-4, synth.FP32, synth.MOM1), n, off),
            dev_bits(synth.normal(1e-8, synth.FP32, synth.MOM2, absolute=True), n, off))


def _oracle_step(n, N, fmt, hp, grad_scale=1.0, post_scale=1.0):
    specs = [synth.normal(1e-3, fmt, synth.GRAD, r, 9) for r in range(N)]
    master = host_bits(synth.normal(0.02, synth.FP32, synth.MASTER), n).view(np.float32).copy()
    m = host_bits(synth.normal(1e-4, synth.FP32, synth.MOM1), n).view(np.float32).copy()
    v = host_bits(synth.normal(1e-8, synth.FP32, synth.MOM2, absolute=True), n).view(np.float32).copy()
    g = oracle.grad_reduce([host_bits(s, n) for s in specs], fmt, post_scale=post_scale)
    p16 = oracle.adamw(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], hp["step"], g, master, m, v,
                       p16_dtype=fmt, grad_scale=grad_scale)
    return specs, g, master, m, v, p16


def _check(master, m, v, p16, ref, fmt):
    _, _, rm, rmm, rv, rp = ref
    assert_state_close(bits_of(master), rm, "master")
    assert_state_close(bits_of(m), rmm, "m")
    assert_state_close(bits_of(v), rv, "v")
    assert_p16_within_ulp(bits_of(p16), rp, fmt, "p16")


@pytest.mark.parametrize("n", [1, 7, 8, 9, 4099, 100_003])
@pytest.mark.parametrize("goff,soff,poff", [(0, 0, 0), (1, 1, 1), (2, 0, 0), (0, 3, 0), (5, 2, 4), (0, 0, 3)])
def test_step_odd_lengths_and_views(ss, n, goff, soff, poff):
    import torch
    N, fmt = 4, synth.BF16
    ref = _oracle_step(n, N, fmt, HP)
    G = [dev_bits(s, n, goff) for s in ref[0]]
    master, m, v = _state(n, soff)
    p16 = torch.zeros(n + poff, dtype=tdt(fmt), device="cuda")[poff:]
    ss.ss_adam_step(HP, n, master, m, v, rank_grads=G, param16=p16)
    _check(master, m, v, p16, ref, fmt)


@pytest.mark.parametrize("N,goff", [(1, 0), (2, 0), (9, 0), (64, 0), (130, 0), (1024, 0), (1024, 3), (65, 1)])
@pytest.mark.parametrize("fmt", [synth.BF16, synth.FP16])
def test_step_rank_counts(ss, N, goff, fmt):
    """Rank counts across the kernel forms and both pointer-table sizes, up to the maximum 1024
    (aligned, and all views off the state's phase: the per-thread shifted kernel)."""
    import torch
    n = 20_011
    ref = _oracle_step(n, N, fmt, HP)
    G = [dev_bits(s, n, offset=goff) for s in ref[0]]
    master, m, v = _state(n)
    p16 = torch.zeros(n, dtype=tdt(fmt), device="cuda")
    ss.ss_adam_step(HP, n, master, m, v, rank_grads=G, param16=p16)
    _check(master, m, v, p16, ref, fmt)


@pytest.mark.parametrize("gfmt,pfmt", [(synth.BF16, synth.FP16), (synth.FP16, synth.BF16), (synth.BF16, synth.BF16),
                                       (synth.FP16, synth.FP16), (synth.FP32, synth.FP16), (synth.FP32, synth.BF16)])
@pytest.mark.parametrize("N,goff", [(3, 0), (9, 0), (20, 0), (3, 5)])
def test_step_gradient_and_param_formats(ss, gfmt, pfmt, N, goff):
    """Every pairing of gradient format (bf16, fp16, or an fp32 gradient) with parameter format,
    through the double-buffered (N = 3), warp-cooperative (N = 9, aligned), single-buffered
    (N = 20) and shifted-load (views 5 elements off) kernels, against the oracle."""
    import torch
    n = 30_011
    hp = dict(HP, step=7)
    master0 = host_bits(synth.normal(0.02, synth.FP32, synth.MASTER), n).view(np.float32).copy()
    m0 = host_bits(synth.normal(1e-4, synth.FP32, synth.MOM1), n).view(np.float32).copy()
    v0 = host_bits(synth.normal(1e-8, synth.FP32, synth.MOM2, absolute=True), n).view(np.float32).copy()
    master, m, v = _state(n)
    p16 = torch.zeros(n, dtype=tdt(pfmt), device="cuda")
    if gfmt == synth.FP32:
        spec = synth.normal(1e-3, synth.FP32, synth.GRAD, 0, 7)
        g = host_bits(spec, n).view(np.float32).copy()
        g32 = dev_bits(spec, n, offset=goff)   # off by 5: no common phase with the state, element-wise
        ss.ss_adam_step(hp, n, master, m, v, g32=g32, param16=p16)
    else:
        specs = [synth.normal(1e-3, gfmt, synth.GRAD, r, 7) for r in range(N)]
        g = oracle.grad_reduce([host_bits(s_, n) for s_ in specs], gfmt)
        G = [dev_bits(s_, n, offset=goff) for s_ in specs]
        ss.ss_adam_step(hp, n, master, m, v, rank_grads=G, param16=p16)
    rp = oracle.adamw(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], hp["step"], g, master0, m0,
                      v0, p16_dtype=pfmt)
    _check(master, m, v, p16, (None, g, master0, m0, v0, rp), pfmt)


def _sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("N,from_g32", [(1, False), (2, True), (6, False), (8, False), (24, False)])
@pytest.mark.parametrize("k,d", [(1, -1), (1, 0), (1, 1), (2, -2049), (2, 255), (3, 4103)])
def test_step_chunk_boundaries(ss, N, from_g32, k, d):
    """Shard lengths around whole passes of the grid over its chunks (a pass: 16 chunks of 32
    8-element groups per block, one block per SM), so the last pass is just full, just short or
    just over, through each way the step kernels own chunks: adjacent per block (1 rank, an fp32
    gradient), round robin (6 and 24 ranks: single-buffered kernel; 8 ranks: double-buffered).
    Every element is stepped exactly once: all of the state against the oracle."""
    import torch
    n = k * _sms() * 16 * 32 * 8 + d
    ref = _oracle_step(n, N, synth.BF16, HP)
    master, m, v = _state(n)
    p16 = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    if from_g32:
        g32 = torch.from_numpy(np.ascontiguousarray(ref[1], dtype=np.float32)).cuda()
        ss.ss_adam_step(HP, n, master, m, v, g32=g32, param16=p16)
    else:
        G = [dev_bits(s, n) for s in ref[0]]
        ss.ss_adam_step(HP, n, master, m, v, rank_grads=G, param16=p16)
    _check(master, m, v, p16, ref, synth.BF16)


@pytest.mark.parametrize("N,accumulate", [(1, True), (1, False), (2, True), (2, False), (3, True), (4, True),
                                          (8, True), (9, True)])
@pytest.mark.parametrize("k,d", [(1, -1), (1, 0), (2, 257), (3, -4096)])
def test_reduce_chunk_boundaries(ss, N, accumulate, k, d):
    """The aligned reduce around whole passes of its grid (one 1024-thread block per SM whose 32
    warps take chunks of 256 elements -- 8 elements a lane, 4 + 4 at lane stride, or 8 a lane stored
    through shared memory, by rank count and accumulation; 9 ranks grid-stride), accumulating into
    the output or not: bit-exact, so no element is added twice or missed."""
    import torch
    n = k * _sms() * 32 * 32 * 8 + d
    specs = [synth.normal(1e-3, synth.BF16, synth.GRAD, r, 4) for r in range(N)]
    G = [dev_bits(s, n) for s in specs]
    init = dev_bits(synth.normal(1e-2, synth.FP32, synth.MOM1), n)
    out = init.clone()
    ss.ss_grad_reduce(G, n, out, accumulate=accumulate)
    acc = bits_of(init).copy() if accumulate else None
    ref = oracle.grad_reduce([host_bits(s, n) for s in specs], synth.BF16, accumulate_into=acc)
    ref = acc if accumulate else ref
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_step_from_fp32_grad_matches_fused(ss):
    import torch
    n, N = 50_001, 8
    ref = _oracle_step(n, N, synth.BF16, HP)
    G = [dev_bits(s, n) for s in ref[0]]
    g32 = torch.empty(n, dtype=torch.float32, device="cuda")
    ss.ss_grad_reduce(G, n, g32)
    master, m, v = _state(n)
    p16 = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    ss.ss_adam_step(HP, n, master, m, v, g32=g32, param16=p16)
    _check(master, m, v, p16, ref, synth.BF16)
    # the two-kernel path and the fused path write identical bits
    master2, m2, v2 = _state(n)
    p2 = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    ss.ss_adam_step(HP, n, master2, m2, v2, rank_grads=G, param16=p2)
    for a, b in ((master, master2), (m, m2), (v, v2)):
        assert torch.equal(a, b)
    assert torch.equal(p16.view(torch.int16), p2.view(torch.int16))


@pytest.mark.parametrize("N,offsets", [
    (4, lambda r: 0),            # aligned: the double-buffered kernel
    (12, lambda r: 0),           # aligned: the single-buffered kernel
    (2, lambda r: 1),            # one phase off: warp-cooperative double-buffered, 512-thread blocks
    (8, lambda r: 3),            # one phase off: warp-cooperative double-buffered, 384-thread blocks
    (4, lambda r: (r % 7) + 1),  # mixed phases: warp-cooperative double-buffered, a shift per rank
    (12, lambda r: 5),           # one phase off: warp-cooperative double-buffered, 256-thread blocks
    (20, lambda r: 5),           # one phase off: warp-cooperative single-buffered
    (12, lambda r: (r % 7) + 1), # mixed phases, 256-thread blocks, a shift per rank
    (13, lambda r: (r % 7) + 1), # mixed phases, more ranks: the per-thread kernel
])
def test_step_options(ss, N, offsets):
    """post_scale, g_out, the non-finite flag, the device gradient scale and the skip flag through
    every form of the fused step kernel, against the oracle (g_out bit-exact)."""
    import torch
    n = 30_001
    coef = np.float32(0.37)
    ref = _oracle_step(n, N, synth.BF16, HP, grad_scale=float(coef), post_scale=0.25)
    G = [dev_bits(s, n, offset=offsets(r)) for r, s in enumerate(ref[0])]
    master, m, v = _state(n)
    p16 = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    g_out = torch.empty(n, dtype=torch.float32, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = torch.tensor([coef], dtype=torch.float32, device="cuda")
    skip = torch.zeros(1, dtype=torch.int32, device="cuda")
    ss.ss_adam_step(HP, n, master, m, v, rank_grads=G, post_scale=0.25, param16=p16, g_out=g_out,
                    nonfinite_flag=flag, dev_grad_scale=scale, dev_skip_flag=skip)
    _check(master, m, v, p16, ref, synth.BF16)
    assert np.array_equal(g_out.cpu().numpy().view(np.uint32), ref[1].view(np.uint32))
    assert flag.item() == 0
    # skip flag set: nothing is written
    before = [t.clone() for t in (master, m, v, p16)]
    skip.fill_(1)
    G[1][77] = float("nan")
    ss.ss_adam_step(HP, n, master, m, v, rank_grads=G, param16=p16, nonfinite_flag=flag, dev_skip_flag=skip)
    for a, b in zip(before, (master, m, v, p16)):
        assert torch.equal(a.view(torch.int16) if a.dtype != torch.float32 else a,
                           b.view(torch.int16) if b.dtype != torch.float32 else b)
    assert flag.item() == 0
    skip.fill_(0)
    ss.ss_adam_step(HP, n, master, m, v, rank_grads=G, param16=p16, nonfinite_flag=flag, dev_skip_flag=skip)
    assert flag.item() == 1


def test_step_writes_into_flat_buffer(ss):
    """param16 may point into the flat unit buffer at the shard's offset (fused unshard)."""
    import torch
    P, N = 100_000, 7
    _, bounds = ss.ss_flatten_layout([P], N)
    flat = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    for k in range(N):
        lo, hi = int(bounds[k]), int(bounds[k + 1])
        n = hi - lo
        ref = _oracle_step(n, 2, synth.BF16, HP)
        G = [dev_bits(s, n) for s in ref[0]]
        master, m, v = _state(n)
        ss.ss_adam_step(HP, n, master, m, v, rank_grads=G, param16=flat[lo:hi])
        _check(master, m, v, flat[lo:hi], ref, synth.BF16)


# ----------------------------------------------------------------------------- unshard / reshard

@pytest.mark.parametrize("P,N", [(0, 3), (2, 5), (100, 3), (4099, 64), (1_000_003, 8), (123_457, 1024)])
@pytest.mark.parametrize("fmt", [synth.BF16, synth.FP32])
def test_unshard_reshard_exact(ss, P, N, fmt):
    import torch
    _, b = ss.ss_flatten_layout([P], N)
    dt = torch.float32 if fmt == synth.FP32 else torch.bfloat16
    shards = []
    for k in range(N):
        n = int(b[k + 1] - b[k])
        shards.append(dev_bits(synth.normal(1.0, fmt, synth.PARAM16, k), n, offset=k % 3))
    flat = torch.full((P,), -1.0, dtype=dt, device="cuda")
    ss.ss_unshard(shards, b, flat)
    host = [bits_of(s) for s in shards]
    expect = oracle.unshard(host, b) if P else np.zeros(0)
    got = bits_of(flat)
    assert np.array_equal(got.view(np.uint8), expect.view(np.uint8))
    back = [torch.full((int(b[k + 1] - b[k]) + 3,), 7.0, dtype=dt, device="cuda")[(k * 5) % 4:][:int(b[k + 1] - b[k])]
            for k in range(N)]
    ss.ss_reshard(flat, b, back)
    for x, y in zip(back, host):
        assert np.array_equal(bits_of(x).view(np.uint8), y.view(np.uint8))


def test_unshard_into_offset_flat(ss):
    """The flat buffer itself at odd element offsets: every shard lands on a shifted boundary."""
    import torch
    P, N = 65_537, 8
    _, b = ss.ss_flatten_layout([P], N)
    for off in range(8):
        shards = [dev_bits(synth.normal(1.0, synth.FP16, synth.PARAM16, k, off), int(b[k + 1] - b[k])) for k in range(N)]
        base = torch.zeros(P + 8, dtype=torch.float16, device="cuda")
        flat = base[off:off + P]
        ss.ss_unshard(shards, b, flat)
        assert torch.equal(flat.view(torch.int16), torch.cat([s.view(torch.int16) for s in shards]))
        assert (base[:off] == 0).all() and (base[off + P:] == 0).all()


@pytest.mark.parametrize("N,off,dtname", [(8, 1, "bfloat16"), (64, 3, "bfloat16"), (7, 1, "float32"),
                                           (1, 5, "float16")])
def test_unshard_reshard_large_off_phase(ss, N, off, dtname):
    """2^26 + 13 elements with the flat buffer `off` elements past a 16-byte boundary: every
    segment takes the warp-cooperative shifted reads over many warp iterations; the round trip is
    bit-exact and nothing outside the flat view is written."""
    import torch
    dt = getattr(torch, dtname)
    P = (1 << 26) + 13
    _, b = ss.ss_flatten_layout([P], N)
    src = torch.arange(P, device="cuda", dtype=torch.int32)
    iv = torch.int32 if dt == torch.float32 else torch.int16
    shards = [src[int(b[k]):int(b[k + 1])].to(iv).view(dt).clone() for k in range(N)]
    base = torch.zeros(P + 16, dtype=dt, device="cuda")
    flat = base[off:off + P]
    ss.ss_unshard(shards, b, flat)
    assert torch.equal(flat.view(iv), torch.cat([t.view(iv) for t in shards]))
    assert (base.view(iv)[:off] == 0).all() and (base.view(iv)[off + P:] == 0).all()
    back = [torch.zeros(int(b[k + 1] - b[k]), dtype=dt, device="cuda") for k in range(N)]
    ss.ss_reshard(flat, b, back)
    for x, y in zip(back, shards):
        assert torch.equal(x.view(iv), y.view(iv))


def test_step_split_calls_agree(ss):
    """A shard stepped in two calls (a short one and a long one) gets the same bits as in one call."""
    import torch
    n, N, cut = 200_003, 8, 1000
    specs = [synth.normal(1e-3, synth.BF16, synth.GRAD, r, 4) for r in range(N)]
    G = [dev_bits(s, n) for s in specs]
    a = _state(n)
    b = _state(n)
    pa = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    pb = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    ss.ss_adam_step(HP, n, *a, rank_grads=G, param16=pa)
    ss.ss_adam_step(HP, cut, *(t[:cut] for t in b), rank_grads=[g[:cut] for g in G], param16=pb[:cut])
    ss.ss_adam_step(HP, n - cut, *(t[cut:] for t in b), rank_grads=[g[cut:] for g in G], param16=pb[cut:])
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert torch.equal(pa.view(torch.int16), pb.view(torch.int16))


@pytest.mark.parametrize("N", [1, 2, 3, 5, 6, 7, 8, 9, 11, 12, 13])
@pytest.mark.parametrize("n", [27, 40, 1000, 300_007])
@pytest.mark.parametrize("fmt", [synth.BF16, synth.FP16])
@pytest.mark.parametrize("same", [True, False])
def test_step_shifted_loads_each_rank_count(ss, N, n, fmt, same):
    """Rank views off the aligned state's phase: all at one offset (1..7) or rank r at (r % 7) + 1
    (mixed phases), from a 1-group body (n = 27) to many runs per warp: the warp-cooperative
    double-buffered kernel (one sum shifted once, up to 16 ranks, or each rank's packed chunk
    shifted by its own phase, up to 12), for 13 ranks at mixed phases the per-thread one; equal
    to the aligned kernel bit for bit and to the oracle."""
    import torch
    hp = dict(HP, step=5)
    ref = _oracle_step(n, N, fmt, hp)
    G_al = [dev_bits(s, n) for s in ref[0]]
    offs = [(n % 7) + 1] * N if same else [(r % 7) + 1 for r in range(N)]
    G_off = [dev_bits(s, n, offset=o) for s, o in zip(ref[0], offs)]
    a, b = _state(n), _state(n)
    pa = torch.zeros(n, dtype=tdt(fmt), device="cuda")
    pb = torch.zeros(n + 2, dtype=tdt(fmt), device="cuda")[(n % 3):(n % 3) + n]
    ss.ss_adam_step(hp, n, *a, rank_grads=G_al, param16=pa)
    ss.ss_adam_step(hp, n, *b, rank_grads=G_off, param16=pb)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert torch.equal(pa.view(torch.int16), pb.view(torch.int16))
    _check(*b, pb, ref, fmt)


@pytest.mark.parametrize("N", [3, 8, 12, 16, 65, 1024])
def test_step_mixed_phases(ss, N):
    """Rank r's gradient view r % 8 elements into its buffer (so some ranks sit on the state's
    16-byte phase and the others at every other phase): up to 12 ranks the warp-cooperative
    double-buffered kernel shifts each rank by its own phase before adding it in rank order, more
    ranks take the per-thread kernel (both rank-table sizes); bit-equal to the aligned kernel and
    within the tolerance of the oracle."""
    import torch
    n = 40_009
    ref = _oracle_step(n, N, synth.BF16, HP)
    G_al = [dev_bits(s, n) for s in ref[0]]
    G_mx = [dev_bits(s, n, offset=r % 8) for r, s in enumerate(ref[0])]
    a, b = _state(n), _state(n)
    pa = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    pb = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    ss.ss_adam_step(HP, n, *a, rank_grads=G_al, param16=pa)
    ss.ss_adam_step(HP, n, *b, rank_grads=G_mx, param16=pb)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert torch.equal(pa.view(torch.int16), pb.view(torch.int16))
    _check(*b, pb, ref, synth.BF16)


@pytest.mark.parametrize("N", [2, 8, 16, 32])
@pytest.mark.parametrize("warps_per_sm", [8, 12, 16])
@pytest.mark.parametrize("k,d", [(1, -1), (1, 0), (1, 1), (2, 7), (3, -5)])
def test_step_shifted_run_boundaries(ss, N, warps_per_sm, k, d):
    """The warp-cooperative shifted-load kernels take runs of 31 groups from a per-block counter;
    their grid passes over k x (SMs x resident warps) runs (16, 12 or 8 warps per SM, by block
    shape), so shard lengths whose body is just a whole number of passes, or one run more or less,
    check that every run is taken exactly once (2, 8 and 16 ranks: double-buffered in 512-, 384-
    and 256-thread blocks; 32: single-buffered), with the gradient views one element off the
    state's phase: all of the state against the oracle, and bit-equal to the aligned kernel."""
    import torch
    runs = k * _sms() * warps_per_sm + d
    n = (runs * 31 + 2) * 8 + 3          # body groups 1 .. nvec - 2, plus a 3-element tail
    ref = _oracle_step(n, N, synth.BF16, HP)
    G_al = [dev_bits(s, n) for s in ref[0]]
    G_off = [dev_bits(s, n, offset=1) for s in ref[0]]
    a, b = _state(n), _state(n)
    pa = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    pb = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    ss.ss_adam_step(HP, n, *a, rank_grads=G_al, param16=pa)
    ss.ss_adam_step(HP, n, *b, rank_grads=G_off, param16=pb)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert torch.equal(pa.view(torch.int16), pb.view(torch.int16))
    _check(*b, pb, ref, synth.BF16)


@pytest.mark.parametrize("goffs,poff", [((1,) * 8, 0), ((0, 1, 2, 3, 4, 5, 6, 7), 3), ((3,) * 8, 1)])
def test_step_views_off_phase_match_aligned(ss, goffs, poff):
    """Rank views (and param16) off the state's 16-byte phase take the shifted-load kernel;
    it must write exactly the bits the aligned kernel writes, and match the oracle."""
    import torch
    n, N = (1 << 22) + 3, 8
    ref = _oracle_step(n, N, synth.BF16, HP)
    G_al = [dev_bits(s, n) for s in ref[0]]
    G_off = [dev_bits(s, n, offset=o) for s, o in zip(ref[0], goffs)]
    a, b = _state(n), _state(n)
    pa = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    pb = torch.zeros(n + poff, dtype=torch.bfloat16, device="cuda")[poff:]
    ss.ss_adam_step(HP, n, *a, rank_grads=G_al, param16=pa)
    ss.ss_adam_step(HP, n, *b, rank_grads=G_off, param16=pb)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert torch.equal(pa.view(torch.int16), pb.view(torch.int16))
    _check(*b, pb, ref, synth.BF16)


def test_long_run_does_not_drift(ss):
    """1000 AdamW steps on one 65,539-element shard (4 bf16 ranks, fresh gradients every step,
    lr 1e-3, wd 0.1): the stored fp32 master/m/v stay within the per-step tolerance of the oracle
    after all 1000 steps, i.e. the GPU's rounding does not accumulate."""
    import torch
    n, N, T = 65_539, 4, 1000
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
    master, m, v = _state(n)
    om = host_bits(synth.normal(0.02, synth.FP32, synth.MASTER), n).view(np.float32).copy()
    omm = host_bits(synth.normal(1e-4, synth.FP32, synth.MOM1), n).view(np.float32).copy()
    ov = host_bits(synth.normal(1e-8, synth.FP32, synth.MOM2, absolute=True), n).view(np.float32).copy()
    G = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    p16 = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    for t in range(1, T + 1):
        specs = [synth.normal(1e-3, synth.BF16, synth.GRAD, r, t) for r in range(N)]
        for r in range(N):
            synth.device_fill(specs[r], G[r].view(torch.int16))
        ss.ss_adam_step(dict(hp, step=t), n, master, m, v, rank_grads=G, param16=p16)
        g = oracle.grad_reduce([host_bits(s_, n) for s_ in specs], synth.BF16)
        rp = oracle.adamw(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], t, g, om, omm, ov,
                          p16_dtype=synth.BF16)
    _check(master, m, v, p16, (None, None, om, omm, ov, rp), synth.BF16)
