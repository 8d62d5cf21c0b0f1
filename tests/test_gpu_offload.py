"""Optimizer-state offload: master, m and v kept in pinned host memory.

Pages: "AI Model Sharding: FSDP, DeepSpeed ZeRO, and Tensor Parallelism" and
"Distributed Deep Learning & Model Sharding" describe moving optimizer state to
CPU memory (ZeRO-Offload, FSDP CPU offload) when GPU memory runs out. On
GB300 the GPU reads and writes pinned Grace memory directly over NVLink-C2C,
so the same fused kernel runs with host-resident state and no copy step; the
results must be bit-identical to the device-resident run.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def test_host_resident_state_bit_identical():
    import torch

    import fsdp_sharded_mixed_ss_gb300 as ss

    n, N = 3_000_001, 8
    G = []
    for r in range(N):
        t = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        synth.device_fill(synth.normal(1e-3, synth.BF16, synth.GRAD, r, 1), t.view(torch.int16))
        G.append(t)
    dev = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(3)]
    for t, spec in zip(dev, (synth.normal(0.02, synth.FP32, synth.MASTER), synth.normal(1e-4, synth.FP32, synth.MOM1),
                             synth.normal(1e-8, synth.FP32, synth.MOM2, absolute=True))):
        synth.device_fill(spec, t.view(torch.int32))
    host = [t.cpu().pin_memory() for t in dev]
    p_dev = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    p_host = torch.zeros(n, dtype=torch.bfloat16).pin_memory()
    for step in (1, 2):
        hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=step)
        ss.ss_adam_step(hp, n, *dev, rank_grads=G, param16=p_dev)
        ss.ss_adam_step(hp, n, host[0].data_ptr(), host[1].data_ptr(), host[2].data_ptr(), rank_grads=G,
                        param16=p_host.data_ptr(), pdtype=ss.SS_BF16)
    torch.cuda.synchronize()
    for a, b in zip(dev, host):
        assert np.array_equal(a.cpu().numpy().view(np.uint32), b.numpy().view(np.uint32))
    assert torch.equal(p_dev.cpu().view(torch.int16), p_host.view(torch.int16))
