"""GPU tests of the launch machinery around the kernels: CUDA-graph capture and replay,
concurrent calls on two streams, and back-to-back dependent calls.

Every kernel of the library is launched as a programmatic dependent of the kernel ahead of it
and waits for that kernel's grid before touching memory. These tests check that the ordering
holds wherever results depend on it -- a step reading the gradient a reduce wrote just before,
a reduce reading what a torch kernel wrote just before -- by comparing unsynchronised chains
with the same calls separated by device synchronisations, bit for bit; and that the calls can
be captured into a CUDA graph and replayed with the same results as eager execution.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    import fsdp_sharded_mixed_ss_gb300 as m
    return m


def fill(spec, t):
    import torch
    synth.device_fill(spec, t.view(torch.int32 if t.dtype == torch.float32 else torch.int16))
    return t


def mlp_state(w):
    import torch
    P = w.P
    master = fill(w.master, torch.empty(P, dtype=torch.float32, device="cuda"))
    return [master, torch.zeros(P, device="cuda"), torch.zeros(P, device="cuda")]


def mlp_step(ss, w, bounds, G, state, flat, p16, sums, coef, ws, t):
    """One clipped step of every shard of the tiny MLP, parameters written straight into `flat`,
    then the shards' 16-bit copies unsharded into `p16`'s flat image (two unshard paths)."""
    N = w.n_ranks
    sl = [slice(int(bounds[k]), int(bounds[k + 1])) for k in range(N)]
    for k in range(N):
        ss.ss_grad_sumsq(sl[k].stop - sl[k].start, sums[k:k + 1], ws, rank_grads=[g[sl[k]] for g in G])
    ss.ss_clip_coef(sums, N, 0.05, coef)
    master, m, v = state
    for k in range(N):
        ss.ss_adam_step(w.hp(t), sl[k].stop - sl[k].start, master[sl[k]], m[sl[k]], v[sl[k]],
                        rank_grads=[g[sl[k]] for g in G], param16=flat[sl[k]], dev_grad_scale=coef)
    ss.ss_reshard(flat, bounds, p16)


def test_graph_capture_replays_the_clipped_step(ss):
    """Tiny MLP (4 shards): sum of squares, clip coefficient, fused step into the flat buffer and a
    reshard, captured once into a CUDA graph and replayed 3 times, equal bit for bit to the same
    calls run eagerly 3 times (the step number is fixed at capture, so both repeat step 1)."""
    import torch
    w = workloads.tiny_mlp()
    N, P = w.n_ranks, w.P
    _, bounds = ss.ss_flatten_layout(w.numels, N)
    G = [fill(w.grad(r, 1), torch.empty(P, dtype=torch.bfloat16, device="cuda")) for r in range(N)]
    ws = torch.empty(ss.ss_grad_sumsq_workspace(P) // 8, dtype=torch.float64, device="cuda")

    def buffers():
        flat = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
        p16 = [torch.zeros(int(bounds[k + 1] - bounds[k]), dtype=torch.bfloat16, device="cuda") for k in range(N)]
        return (mlp_state(w), flat, p16, torch.zeros(N, dtype=torch.float64, device="cuda"),
                torch.zeros(1, device="cuda"))

    eager = buffers()
    for _ in range(3):
        mlp_step(ss, w, bounds, G, eager[0], eager[1], eager[2], eager[3], eager[4], ws, 1)
    torch.cuda.synchronize()

    graphed = buffers()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # one eager call first (library and allocator warm)
        mlp_step(ss, w, bounds, G, *buffers()[:5], ws, 1)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mlp_step(ss, w, bounds, G, graphed[0], graphed[1], graphed[2], graphed[3], graphed[4], ws, 1)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()

    for a, b in zip(eager[0], graphed[0]):
        assert torch.equal(a, b)
    assert torch.equal(eager[1], graphed[1])
    for a, b in zip(eager[2], graphed[2]):
        assert torch.equal(a, b)
    assert torch.equal(eager[3], graphed[3]) and torch.equal(eager[4], graphed[4])
    # and the graph did real work: the flat buffer holds the rounded master
    m16 = oracle.round16(graphed[0][0].cpu().numpy(), oracle.BF16)
    assert np.array_equal(graphed[1].view(torch.int16).cpu().numpy().view(np.uint16), m16)


def test_graph_capture_replays_the_shifted_load_steps(ss):
    """The warp-cooperative shifted-load kernel forms -- 8 ranks one element off the state's phase
    (double-buffered, 384-thread blocks), 4 ranks at mixed phases (a shift per rank), 16 ranks off
    phase (double-buffered, 256-thread blocks), 20 ranks off phase (single-buffered) -- each take
    their runs from a counter in shared memory; captured once into a CUDA graph and replayed 3
    times, equal bit for bit to the same calls run eagerly 3 times."""
    import torch
    n = 1_000_003
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=2)
    cases = [(8, lambda r: 1), (4, lambda r: (r % 7) + 1), (16, lambda r: 3), (20, lambda r: 5)]
    G = []
    for N, off in cases:
        views = []
        for r in range(N):
            base = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")
            views.append(fill(synth.normal(1e-3, synth.BF16, synth.GRAD, r, 5), base[off(r):off(r) + n]))
        G.append(views)

    def buffers():
        return [[fill(synth.normal(0.02, synth.FP32, synth.MASTER, i), torch.empty(n, device="cuda")),
                 torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda"),
                 torch.empty(n, dtype=torch.bfloat16, device="cuda")] for i in range(len(cases))]

    def step(bufs):
        for views, b in zip(G, bufs):
            ss.ss_adam_step(hp, n, *b[:3], rank_grads=views, param16=b[3])

    eager = buffers()
    for _ in range(3):
        step(eager)
    torch.cuda.synchronize()
    graphed = buffers()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):      # the eager calls above warmed up the library
        step(graphed)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, graphed):
        for x, y in zip(a, b):
            assert torch.equal(x, y)


def test_two_streams_run_independent_shards_concurrently(ss):
    """Two shards stepped in alternation on two streams (no ordering between the streams) give the
    same bits as the same steps run one after another on one stream."""
    import torch
    n, N = 3_000_011, 8
    G = [[fill(synth.normal(1e-3, synth.BF16, synth.GRAD, 8 * s + r, 2), torch.empty(n, dtype=torch.bfloat16,
                                                                                    device="cuda"))
          for r in range(N)] for s in range(2)]

    def state(s):
        return [fill(synth.normal(0.02, synth.FP32, synth.MASTER, s), torch.empty(n, device="cuda")),
                torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda"),
                torch.empty(n, dtype=torch.bfloat16, device="cuda")]

    hp = lambda t: dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=t)
    seq = [state(0), state(1)]
    for t in range(1, 6):
        for s in range(2):
            ss.ss_adam_step(hp(t), n, *seq[s][:3], rank_grads=G[s], param16=seq[s][3])
    torch.cuda.synchronize()

    par = [state(0), state(1)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    for t in range(1, 6):
        for s in range(2):
            ss.ss_adam_step(hp(t), n, *par[s][:3], rank_grads=G[s], param16=par[s][3], stream=streams[s])
    torch.cuda.synchronize()
    for a, b in zip(seq, par):
        for x, y in zip(a, b):
            assert torch.equal(x, y)


def test_dependent_calls_back_to_back_match_synchronised_calls(ss):
    """reduce -> step through an fp32 gradient buffer, five times with different gradients, no
    synchronisation between the calls; then the same sequence with a device synchronisation after
    every call. A step that read the gradient before the reduce ahead of it had finished would
    differ."""
    import torch
    n, N = 6_000_037, 4
    Gs = [[fill(synth.normal(1e-3, synth.BF16, synth.GRAD, r, i + 1), torch.empty(n, dtype=torch.bfloat16,
                                                                                 device="cuda"))
           for r in range(N)] for i in range(5)]

    def run(sync):
        master = fill(synth.normal(0.02, synth.FP32, synth.MASTER), torch.empty(n, device="cuda"))
        m, v = torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
        g32 = torch.empty(n, device="cuda")
        p16 = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        for i in range(5):
            ss.ss_grad_reduce(Gs[i], n, g32, post_scale=0.25)
            if sync:
                torch.cuda.synchronize()
            ss.ss_adam_step(dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=i + 1), n,
                            master, m, v, g32=g32, param16=p16)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return master, m, v, p16

    for a, b in zip(run(False), run(True)):
        assert torch.equal(a, b)


def test_library_call_right_after_a_torch_kernel(ss):
    """A torch kernel writes the rank gradients and the reduce is queued right behind it, eight
    times with different contents: every result equals the oracle's sum of what torch wrote."""
    import torch
    n, N = 2_000_003, 3
    srcs = [[fill(synth.normal(1e-3, synth.FP16, synth.GRAD, r, i + 1), torch.empty(n, dtype=torch.float16,
                                                                                   device="cuda"))
             for r in range(N)] for i in range(8)]
    G = [torch.empty(n, dtype=torch.float16, device="cuda") for _ in range(N)]
    outs = [torch.empty(n, device="cuda") for _ in range(8)]
    torch.cuda.synchronize()
    for i in range(8):
        for r in range(N):
            G[r].copy_(srcs[i][r])
        ss.ss_grad_reduce(G, n, outs[i])
    torch.cuda.synchronize()
    for i in range(8):
        ref = oracle.grad_reduce([synth.host_range(synth.normal(1e-3, synth.FP16, synth.GRAD, r, i + 1), 0, n)
                                  for r in range(N)], oracle.FP16)
        assert np.array_equal(outs[i].cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_library_call_right_after_a_host_copy_and_across_streams(ss):
    """Each kernel waits for whatever precedes it in its stream, not only kernels: gradients
    copied in from pinned host memory right before the reduce (same stream), and copied on a
    second stream that the reduce's stream waits for through an event, eight times each with
    different contents: every result equals the oracle's sum of the copied values."""
    import torch
    n, N = 1_500_007, 2
    specs = [[synth.normal(1e-3, synth.BF16, synth.GRAD, r, i + 1) for r in range(N)] for i in range(8)]
    host = [[torch.from_numpy(synth.host_range(s, 0, n).view(np.int16)).pin_memory() for s in row] for row in specs]
    G = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    outs = [torch.empty(n, device="cuda") for _ in range(16)]
    copy_stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    for i in range(8):                                   # same stream: copy, then reduce
        for r in range(N):
            G[r].view(torch.int16).copy_(host[i][r], non_blocking=True)
        ss.ss_grad_reduce(G, n, outs[i])
    for i in range(8):                                   # copy on another stream, event, reduce
        copy_stream.wait_stream(torch.cuda.current_stream())   # G no longer read by the last reduce
        with torch.cuda.stream(copy_stream):
            for r in range(N):
                G[r].view(torch.int16).copy_(host[i][r], non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(copy_stream)
        torch.cuda.current_stream().wait_event(ev)
        ss.ss_grad_reduce(G, n, outs[8 + i])
    torch.cuda.synchronize()
    for j in range(16):
        ref = oracle.grad_reduce([synth.host_range(s, 0, n) for s in specs[j % 8]], oracle.BF16)
        assert np.array_equal(outs[j].cpu().numpy().view(np.uint32), ref.view(np.uint32))
