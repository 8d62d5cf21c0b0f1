"""Optimizer-state offload: master, m and v kept in pinned host memory.

Pages: "AI Model Sharding: FSDP, DeepSpeed ZeRO, and Tensor Parallelism" and
"Distributed Deep Learning & Model Sharding" describe moving optimizer state to
CPU memory (ZeRO-Offload, FSDP CPU offload) when GPU memory runs out. On
GB300 the GPU reads and writes pinned Grace memory directly over NVLink-C2C,
so the same fused kernel runs with host-resident state and no copy step. The
host-resident result is checked against the oracle (rank-ordered reduce +
AdamW on the host-regenerated inputs) at sampled elements, within the stated
tolerances, and must also be bit-identical to the device-resident run.
"""
import numpy as np
import pytest

import oracle
import synth

from parity import assert_p16_within_ulp, assert_state_close, sample_indices

pytestmark = pytest.mark.gpu

SPECS = (synth.normal(0.02, synth.FP32, synth.MASTER), synth.normal(1e-4, synth.FP32, synth.MOM1),
         synth.normal(1e-8, synth.FP32, synth.MOM2, absolute=True))


def _hp(step):
    return dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=step)


def test_host_resident_state_matches_oracle_and_device_run():
    import torch

    import fsdp_sharded_mixed_ss_gb300 as ss

    n, N = 3_000_001, 8
    gspec = [synth.normal(1e-3, synth.BF16, synth.GRAD, r, 1) for r in range(N)]
    G = []
    for r in range(N):
        t = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        synth.device_fill(gspec[r], t.view(torch.int16))
        G.append(t)
    dev = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(3)]
    for t, spec in zip(dev, SPECS):
        synth.device_fill(spec, t.view(torch.int32))
    host = [t.cpu().pin_memory() for t in dev]
    p_dev = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    p_host = torch.zeros(n, dtype=torch.bfloat16).pin_memory()
    for step in (1, 2):
        ss.ss_adam_step(_hp(step), n, *dev, rank_grads=G, param16=p_dev)
        ss.ss_adam_step(_hp(step), n, host[0].data_ptr(), host[1].data_ptr(), host[2].data_ptr(), rank_grads=G,
                        param16=p_host.data_ptr(), pdtype=ss.SS_BF16)
    torch.cuda.synchronize()

    # the oracle on the same seeded inputs, regenerated on the host at sampled elements
    idx = sample_indices(0, n, 200_000, 11)
    g = oracle.grad_reduce([synth.host_gather(s, idx) for s in gspec], oracle.BF16)
    st = [synth.host_gather(s, idx).view(np.float32).copy() for s in SPECS]
    for step in (1, 2):
        h = _hp(step)
        p16 = oracle.adamw(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], step, g, *st,
                           p16_dtype=oracle.BF16)
    for name, got, ref in zip(("master", "m", "v"), host, st):
        assert_state_close(got.numpy()[idx], ref, f"host-resident {name}")
    assert_p16_within_ulp(p_host.view(torch.int16).numpy().view(np.uint16)[idx], p16, oracle.BF16,
                          "host-resident param16")

    # and the host-resident run is the device-resident run, bit for bit
    for a, b in zip(dev, host):
        assert np.array_equal(a.cpu().numpy().view(np.uint32), b.numpy().view(np.uint32))
    assert torch.equal(p_dev.cpu().view(torch.int16), p_host.view(torch.int16))
