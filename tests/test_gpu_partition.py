"""partition.shard_step on a GPU, in a one-rank NCCL group: the exchanges degenerate to local copies
through NCCL, so the call chain (all-to-all into rows, fused step on the rows, padded all-gather,
unshard of the gathered rows) must give exactly what ss_adam_step + ss_unshard give on the same
inputs, and the oracle's values. (More ranks need more GPUs; the exchanges across ranks are covered
by the gloo test on CPU.)"""
import socket

import numpy as np
import pytest

import oracle
import synth

from parity import assert_p16_within_ulp, assert_state_close

pytestmark = pytest.mark.gpu

NUMELS = [4099, 1001, 37, 20_000]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shard_step_one_rank_nccl_matches_direct_calls():
    import torch
    import torch.distributed as dist

    import fsdp_sharded_mixed_ss_gb300 as ss
    from fsdp_sharded_mixed_ss_gb300.partition import Partition, shard_step

    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1)
    dist.init_process_group("nccl", rank=0, world_size=1, init_method=f"tcp://127.0.0.1:{_free_port()}",
                            device_id=torch.device("cuda", 0))
    try:
        part = Partition(NUMELS, 1, 0)
        P = part.P
        gspec = synth.normal(1e-3, synth.BF16, synth.GRAD, 0, 1)
        mspec = synth.normal(0.02, synth.FP32, synth.MASTER)
        grad = torch.empty(P, dtype=torch.bfloat16, device="cuda")
        synth.device_fill(gspec, grad.view(torch.int16))
        st = [torch.zeros(P, dtype=torch.float32, device="cuda") for _ in range(3)]
        synth.device_fill(mspec, st[0].view(torch.int32))
        ref_st = [t.clone() for t in st]
        pad = torch.zeros(part.max_len, dtype=torch.bfloat16, device="cuda")
        flat = torch.empty(P, dtype=torch.bfloat16, device="cuda")
        shard_step(hp, part, grad, *st, pad, flat)
        ref_p = torch.empty(P, dtype=torch.bfloat16, device="cuda")
        ss.ss_adam_step(hp, P, *ref_st, rank_grads=[grad], param16=ref_p)
        ref_flat = torch.empty(P, dtype=torch.bfloat16, device="cuda")
        ss.ss_unshard([ref_p], part.bounds, ref_flat)
        torch.cuda.synchronize()
        for a, b in zip(st, ref_st):
            assert torch.equal(a, b)
        assert torch.equal(flat.view(torch.int16), ref_flat.view(torch.int16))
        # and the oracle on the host-regenerated inputs
        g = oracle.grad_reduce([synth.host_range(gspec, 0, P)], oracle.BF16)
        om = synth.host_range(mspec, 0, P).view(np.float32).copy()
        z1, z2 = np.zeros(P, np.float32), np.zeros(P, np.float32)
        p16 = oracle.adamw(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], 1, g, om, z1, z2,
                           p16_dtype=oracle.BF16)
        assert_state_close(st[0].cpu().numpy(), om, "master")
        assert_p16_within_ulp(flat.view(torch.int16).cpu().numpy().view(np.uint16), p16, oracle.BF16, "flat")
    finally:
        dist.destroy_process_group()
