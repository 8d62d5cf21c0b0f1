"""One shard per rank across real processes, on CPU (gloo): the partition and the two exchanges.

Page: "FSDP: Fully Sharded Data Parallel Training at Scale" (how FSDP shards a layer; the FSDP
unit communication cycle). Each process builds the floor(kP/N) partition from the library's
host calls, holds its own full 16-bit gradient of the unit (a seeded stream of its rank),
exchanges gradients with the all-to-all of `partition.exchange_grads`, steps its shard, and
all-gathers the 16-bit shards with `partition.gather_params`. The arithmetic of the step is the
oracle's here (the library's kernels need a GPU); the exchanges are the product code. Checked bit
for bit: every received row is the sending rank's slice; each rank's rank-ordered fp32 sum of the
rows equals the virtual-rank sum of the same slice; and the flat unit assembled from the
gathered rows equals the single-process run of all virtual ranks (oracle reduce + AdamW + cast
on every shard, then the oracle's unshard).
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

# a unit whose P is not a multiple of the rank counts: shards of unequal length, odd offsets
NUMELS = [1001, 37, 4099, 64 * 33, 6]   # P = 7255: odd, and not a multiple of 3, 4 or 7
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _grad_spec(r):
    import synth
    return synth.normal(1e-3, synth.BF16, synth.GRAD, r, 1)


def _master_spec():
    import synth
    return synth.normal(0.02, synth.FP32, synth.MASTER)


def _worker(rank, world, port, out):
    import sys

    import torch
    import torch.distributed as dist

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import oracle
    import synth
    from fsdp_sharded_mixed_ss_gb300.partition import Partition, exchange_grads, gather_params, gathered_rows

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        part = Partition(NUMELS, world, rank)
        P = part.P
        full = torch.from_numpy(synth.host_range(_grad_spec(rank), 0, P).view(np.int16)).view(torch.bfloat16)
        rows = exchange_grads(full, part)
        got_rows = [rows[r].view(torch.int16).numpy().view(np.uint16).copy() for r in range(world)]
        g = oracle.grad_reduce(got_rows, oracle.BF16)
        master = synth.host_range(_master_spec(), part.lo, part.n).view(np.float32).copy()
        m = np.zeros(part.n, np.float32)
        v = np.zeros(part.n, np.float32)
        p16 = oracle.adamw(HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["weight_decay"], HP["step"], g,
                           master, m, v, p16_dtype=oracle.BF16)
        pad = torch.zeros(part.max_len, dtype=torch.bfloat16)
        pad.view(torch.int16)[:part.n] = torch.from_numpy(p16.view(np.int16))
        gathered = gather_params(pad, part)
        flat = torch.cat([x.view(torch.int16) for x in gathered_rows(gathered, part)]).numpy().view(np.uint16)
        out[rank] = dict(bounds=part.bounds.tolist(), lo=part.lo, n=part.n, rows=got_rows, g=g, flat=flat.copy(),
                         segments=part.segments())
    finally:
        dist.destroy_process_group()


def _run(world):
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    return dict(out)


@pytest.mark.parametrize("world", [2, 3, 4, 7])
def test_partition_exchanges_compose_into_the_virtual_rank_unit(world):
    import oracle
    import synth

    res = _run(world)
    offsets, bounds = oracle.flatten_layout(NUMELS, world)
    P = int(bounds[-1])
    lengths = np.diff(bounds)
    assert len(set(lengths.tolist())) == 2          # uneven shards, as floor(kP/N) gives for this P
    # the single-process reference: every virtual rank's gradient, every shard stepped, then unshard
    grads = [synth.host_range(_grad_spec(r), 0, P) for r in range(world)]
    shards = []
    for k in range(world):
        lo, hi = int(bounds[k]), int(bounds[k + 1])
        g = oracle.grad_reduce([x[lo:hi] for x in grads], oracle.BF16)
        master = synth.host_range(_master_spec(), lo, hi - lo).view(np.float32).copy()
        m = np.zeros(hi - lo, np.float32)
        v = np.zeros(hi - lo, np.float32)
        shards.append(oracle.adamw(HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["weight_decay"], HP["step"],
                                   g, master, m, v, p16_dtype=oracle.BF16))
        r = res[k]
        assert r["bounds"] == bounds.tolist() and r["lo"] == lo and r["n"] == hi - lo
        for s in range(world):                       # row s on rank k = rank s's slice of shard k
            assert np.array_equal(r["rows"][s], grads[s][lo:hi])
        assert np.array_equal(r["g"].view(np.uint32), g.view(np.uint32))
        # the shard's segments tile it, in tensor order
        segs = r["segments"]
        assert sum(x[3] for x in segs) == hi - lo
        assert [x[2] for x in segs] == list(np.cumsum([0] + [x[3] for x in segs[:-1]]))
        for t, toff, soff, ln in segs:
            assert offsets[t] + toff == lo + soff
    flat_ref = oracle.unshard(shards, bounds)
    for k in range(world):                           # every rank assembles the same flat unit
        assert np.array_equal(res[k]["flat"], flat_ref)
