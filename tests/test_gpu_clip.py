"""GPU parity of the global gradient-norm clipping path through the C ABI.

Page: "FSDP: Fully Sharded Data Parallel Training at Scale", gradient clipping --
the norm is taken over the whole gradient, each shard contributing its sum of
squares. The GPU sum of squares adds each group of 8 squares in fp32 and the
rest in double: within 8 * 2^-24 (< 5e-7) relative of the exact sum, so the
tests hold it, and the clip coefficient, to 1e-6 relative of the oracle's
double sum. The clipped steps then meet the usual state tolerance.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads

from parity import assert_p16_within_ulp, assert_state_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    import fsdp_sharded_mixed_ss_gb300 as m
    return m


def tdt(fmt):
    import torch
    return {synth.BF16: torch.bfloat16, synth.FP16: torch.float16}[fmt]


def dev_bits(spec, n, offset=0):
    import torch
    dt = torch.float32 if spec.fmt == synth.FP32 else tdt(spec.fmt)
    base = torch.zeros(n + offset, dtype=dt, device="cuda")
    view = base[offset:]
    if n:
        synth.device_fill(spec, view.view(torch.int32 if spec.fmt == synth.FP32 else torch.int16))
    return view


def workspace(ss, n):
    import torch
    return torch.empty(max(ss.ss_grad_sumsq_workspace(n) // 8, 1), dtype=torch.float64, device="cuda")


@pytest.mark.parametrize("N", [1, 2, 8, 64])
@pytest.mark.parametrize("n", [1, 7, 4099, 100_003, (1 << 20) + 7])
@pytest.mark.parametrize("fmt", [synth.BF16, synth.FP16])
def test_sumsq_matches_oracle(ss, N, n, fmt):
    import torch
    specs = [synth.normal(1e-3, fmt, synth.GRAD, r, 5) for r in range(N)]
    G = [dev_bits(s, n, offset=(r % 2) * (n % 3)) for r, s in enumerate(specs)]
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    g_out = torch.empty(n, dtype=torch.float32, device="cuda")
    ss.ss_grad_sumsq(n, out, workspace(ss, n), rank_grads=G, post_scale=0.5, g_out=g_out)
    g = oracle.grad_reduce([synth.host_range(s, 0, n) for s in specs], fmt, post_scale=0.5)
    assert np.array_equal(g_out.cpu().numpy().view(np.uint32), g.view(np.uint32))
    ref = oracle.sumsq(g)
    assert abs(out.item() - ref) <= 1e-6 * ref


@pytest.mark.parametrize("N", [1, 2, 3, 4, 8])
def test_sumsq_several_tiles_per_block(ss, N):
    """2^24 + 5 elements: more tiles than blocks, so each block runs its pipelined loads across
    several tiles (and the last ones read past their tiles' ends), with a ragged 5-element tail."""
    import torch
    n = (1 << 24) + 5
    specs = [synth.normal(1e-3, synth.BF16, synth.GRAD, r, 9) for r in range(N)]
    G = [dev_bits(s, n) for s in specs]
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    g_out = torch.empty(n, dtype=torch.float32, device="cuda")
    ws = workspace(ss, n)
    ss.ss_grad_sumsq(n, out, ws, rank_grads=G, post_scale=0.25, g_out=g_out)
    g = oracle.grad_reduce([synth.host_range(s, 0, n) for s in specs], oracle.BF16, post_scale=0.25)
    assert np.array_equal(g_out.cpu().numpy().view(np.uint32), g.view(np.uint32))
    ref = oracle.sumsq(g)
    assert abs(out.item() - ref) <= 1e-6 * ref
    again = torch.zeros(1, dtype=torch.float64, device="cuda")
    ss.ss_grad_sumsq(n, again, ws, rank_grads=G, post_scale=0.25)
    assert again.item() == out.item()


@pytest.mark.parametrize("N", [2, 8, 64])
@pytest.mark.parametrize("n", [1001, (1 << 20) + 7])
@pytest.mark.parametrize("off", [1, 2, 3])
def test_sumsq_gout_off_the_inputs_phase(ss, N, n, off):
    """The rank gradients aligned and g_out `off` floats off their 16-byte phase: the groups follow
    the gradients (16-byte loads) and g_out is written as aligned vectors realigned by shuffles
    between neighbouring lanes (with the warps' edge elements one by one), for the per-rank-count
    tiles (2, 8 ranks) and the general ones (64). g_out bit-exact and nothing written outside it,
    the sum within the header's 5e-7 of the oracle's and the same bits on a second call."""
    import torch
    specs = [synth.normal(1e-3, synth.BF16, synth.GRAD, r, 8) for r in range(N)]
    G = [dev_bits(s, n) for s in specs]
    base = torch.zeros(n + off + 4, dtype=torch.float32, device="cuda")
    g_out = base[off:off + n]
    out = torch.zeros(2, dtype=torch.float64, device="cuda")
    ws = workspace(ss, n)
    ss.ss_grad_sumsq(n, out[0:1], ws, rank_grads=G, post_scale=0.5, g_out=g_out)
    ss.ss_grad_sumsq(n, out[1:2], ws, rank_grads=G, post_scale=0.5, g_out=g_out)
    g = oracle.grad_reduce([synth.host_range(s, 0, n) for s in specs], oracle.BF16, post_scale=0.5)
    assert np.array_equal(g_out.cpu().numpy().view(np.uint32), g.view(np.uint32))
    assert (base[:off] == 0).all() and (base[off + n:] == 0).all()
    o = out.cpu().numpy()
    ref = oracle.sumsq(g)
    assert o[0] == o[1] and abs(o[0] - ref) <= 5e-7 * ref


def test_sumsq_from_fp32_and_reproducible(ss):
    import torch
    n = 3_000_017
    g = dev_bits(synth.normal(1e-2, synth.FP32, synth.GRAD, 0, 1), n, offset=1)   # misaligned: element path
    ws = workspace(ss, n)
    outs = torch.zeros(3, dtype=torch.float64, device="cuda")
    for i in range(3):
        ss.ss_grad_sumsq(n, outs[i:i + 1], ws, g32=g)
    ref = oracle.sumsq(synth.host_range(synth.normal(1e-2, synth.FP32, synth.GRAD, 0, 1), 0, n).view(np.float32))
    o = outs.cpu().numpy()
    assert o[0] == o[1] == o[2]
    assert abs(o[0] - ref) <= 1e-6 * ref
    g2 = dev_bits(synth.normal(1e-2, synth.FP32, synth.GRAD, 0, 1), n)             # aligned: vector path
    ss.ss_grad_sumsq(n, outs[0:1], ws, g32=g2)
    assert abs(outs[0].item() - ref) <= 1e-6 * ref


def test_sumsq_nonfinite_flag_and_skip(ss):
    """fp16 loss-scale unscaling with overflow skip: a non-finite reduced gradient sets the flag
    in the sum-of-squares pass, and the step reading that flag writes nothing."""
    import torch
    n, N, S = 50_000, 4, 1024.0
    specs = [synth.normal(1e-3, synth.FP16, synth.GRAD, r, 2) for r in range(N)]
    G = [dev_bits(s, n) for s in specs]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    ws = workspace(ss, n)
    ss.ss_grad_sumsq(n, out, ws, rank_grads=G, post_scale=1.0 / S, nonfinite_flag=flag)
    assert flag.item() == 0
    G[2][12345] = float("inf")
    ss.ss_grad_sumsq(n, out, ws, rank_grads=G, post_scale=1.0 / S, nonfinite_flag=flag)
    assert flag.item() == 1
    master = dev_bits(synth.normal(0.02, synth.FP32, synth.MASTER), n)
    m = torch.zeros(n, device="cuda")
    v = torch.zeros(n, device="cuda")
    before = master.clone()
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1)
    ss.ss_adam_step(hp, n, master, m, v, rank_grads=G, post_scale=1.0 / S, dev_skip_flag=flag)
    assert torch.equal(master, before) and (m == 0).all() and (v == 0).all()


@pytest.mark.parametrize("max_norm", [0.3, 1e9])
def test_clipped_steps_tiny_mlp(ss, max_norm):
    """Tiny MLP, 4 shards, 3 steps, each step clipped to the global norm across the 4 shards."""
    import torch
    w = workloads.tiny_mlp()
    N, P = w.n_ranks, w.P
    _, bounds = ss.ss_flatten_layout(w.numels, N)
    G = [torch.empty(P, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    master = torch.empty(P, dtype=torch.float32, device="cuda")
    synth.device_fill(w.master, master.view(torch.int32))
    m = torch.zeros(P, device="cuda")
    v = torch.zeros(P, device="cuda")
    p16 = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
    sums = torch.zeros(N, dtype=torch.float64, device="cuda")
    coef = torch.zeros(1, dtype=torch.float32, device="cuda")
    ws = workspace(ss, P)
    om = synth.host_range(w.master, 0, P).view(np.float32).copy()
    omm = np.zeros(P, np.float32)
    ov = np.zeros(P, np.float32)
    op16 = None
    for t in range(1, w.steps + 1):
        for r in range(N):
            synth.device_fill(w.grad(r, t), G[r].view(torch.int16))
        sl = [slice(int(bounds[k]), int(bounds[k + 1])) for k in range(N)]
        for k in range(N):
            ss.ss_grad_sumsq(sl[k].stop - sl[k].start, sums[k:k + 1], ws, rank_grads=[g[sl[k]] for g in G])
        ss.ss_clip_coef(sums, N, max_norm, coef)
        for k in range(N):
            ss.ss_adam_step(w.hp(t), sl[k].stop - sl[k].start, master[sl[k]], m[sl[k]], v[sl[k]],
                            rank_grads=[g[sl[k]] for g in G], param16=p16[sl[k]], dev_grad_scale=coef)
        # oracle: the same three stages from the same seeded inputs
        g = oracle.grad_reduce([synth.host_range(w.grad(r, t), 0, P) for r in range(N)], oracle.BF16)
        total = 0.0
        for k in range(N):
            total += oracle.sumsq(g[sl[k]])
        oc = oracle.clip_coef(total, max_norm)
        assert abs(coef.item() - oc) <= 1e-6 * oc
        if max_norm > 1e6:
            assert coef.item() == 1.0
        hp = w.hp(t)
        op16 = oracle.adamw(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], t, g, om, omm, ov,
                            p16_dtype=oracle.BF16, grad_scale=oc)
    assert_state_close(master.cpu().numpy(), om, "master")
    assert_state_close(m.cpu().numpy(), omm, "m")
    assert_state_close(v.cpu().numpy(), ov, "v")
    assert_p16_within_ulp(p16.view(torch.int16).cpu().numpy().view(np.uint16), op16, oracle.BF16, "p16")


def test_sumsq_gpt2_shard_full_size(ss):
    """The GPT-2 rank-0 shard (15,554,976 elements, 8 bf16 ranks) at full size."""
    import torch
    w = workloads.gpt2_small()
    _, bounds = ss.ss_flatten_layout(w.numels, w.n_ranks)
    n = int(bounds[1])
    G = [dev_bits(w.grad(r, 1), n) for r in range(w.n_ranks)]
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    ss.ss_grad_sumsq(n, out, workspace(ss, n), rank_grads=G)
    g = oracle.grad_reduce([synth.host_range(w.grad(r, 1), 0, n) for r in range(w.n_ranks)], oracle.BF16)
    ref = oracle.sumsq(g)
    assert abs(out.item() - ref) <= 1e-6 * ref
