"""Canary guards around every output buffer, through every kernel form.

Each output (master, m, v, param16, g_out, the reduce output, the flat unit and the shards) is a view
into a larger buffer whose elements before and after the view hold a canary bit pattern. The calls run
on ragged lengths with views at offsets that select each kernel form -- aligned double-buffered,
single-buffered, warp-cooperative shifted (one phase and mixed phases, 512-, 384- and 256-thread
blocks), per-thread shifted, element-wise, the fp32-gradient form; the reduce's vector and shifted
forms (one phase and mixed phases); the sum of squares with g_out staged through shared memory,
realigned between lanes and element by element; the copies at and off the shards' phase -- and every canary must be intact afterwards, so no
form writes outside its arrays (the head/tail and first/last-group edges included).
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

GUARD = 64
CANARY16 = 0x7BCD
CANARY32 = 0x7F8ABCDE   # a NaN pattern no kernel writes


@pytest.fixture(scope="module")
def ss():
    import fsdp_sharded_mixed_ss_gb300 as m
    return m


def guarded(n, dtype, off, fill=None):
    """(base, view): view = base[GUARD + off : GUARD + off + n], everything else the canary."""
    import torch
    base = torch.empty(n + 2 * GUARD + 8, dtype=dtype, device="cuda")
    iv = torch.int32 if dtype == torch.float32 else torch.int16
    base.view(iv).fill_(CANARY32 if dtype == torch.float32 else CANARY16)
    view = base[GUARD + off:GUARD + off + n]
    if fill is not None:
        synth.device_fill(fill, view.view(iv))
    return base, view


def intact(base, off, n):
    import torch
    iv = torch.int32 if base.dtype == torch.float32 else torch.int16
    b = base.view(iv).cpu().numpy()
    want = np.int32(CANARY32) if base.dtype == torch.float32 else np.int16(CANARY16)
    lo, hi = GUARD + off, GUARD + off + n
    return bool((b[:lo] == want).all() and (b[hi:] == want).all())


def grads(n, N, offsets, dtype=None):
    import torch
    out = []
    for r in range(N):
        base = torch.empty(n + 16, dtype=dtype or torch.bfloat16, device="cuda")
        v = base[offsets(r):offsets(r) + n]
        synth.device_fill(synth.normal(1e-3, synth.BF16, synth.GRAD, r, 2), v.view(torch.int16))
        out.append(v)
    return out


HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=2)

STEP_FORMS = [  # (N, gradient view offset of rank r, master/m/v offsets, param16 offset)
    (8, lambda r: 0, (0, 0, 0), 0),              # aligned double-buffered
    (6, lambda r: 4, (4, 4, 4), 4),              # single-buffered, every array 4 elements past a boundary
    (2, lambda r: 1, (0, 0, 0), 0),              # one phase off: warp-cooperative, 512-thread blocks
    (8, lambda r: 3, (0, 0, 0), 5),              # one phase off: 384-thread blocks, param16 off too
    (12, lambda r: 0, (0, 0, 0), 0),             # aligned 9-16 ranks: warp-cooperative, 256-thread blocks
    (12, lambda r: 7, (0, 0, 0), 2),             # one phase off, 256-thread blocks
    (4, lambda r: (r % 7) + 1, (0, 0, 0), 0),    # mixed phases: a shift per rank
    (12, lambda r: (r % 7) + 1, (0, 0, 0), 0),   # mixed phases, 256-thread blocks
    (13, lambda r: (r % 7) + 1, (0, 0, 0), 3),   # mixed phases, more ranks: per-thread, param16 off too
    (20, lambda r: 1, (0, 0, 0), 0),             # one phase off, more ranks: single-buffered warp-cooperative
    (4, lambda r: 0, (1, 2, 0), 0),              # no common fp32 phase: element-wise
]


@pytest.mark.parametrize("form", range(len(STEP_FORMS)))
@pytest.mark.parametrize("n", [37, 100_003])
def test_step_writes_only_its_arrays(ss, form, n):
    import torch
    N, goff, soffs, poff = STEP_FORMS[form]
    G = grads(n, N, goff)
    specs = (synth.normal(0.02, synth.FP32, synth.MASTER), synth.normal(1e-4, synth.FP32, synth.MOM1),
             synth.normal(1e-8, synth.FP32, synth.MOM2, absolute=True))
    st = [guarded(n, torch.float32, o, sp) for o, sp in zip(soffs, specs)]
    p16 = guarded(n, torch.bfloat16, poff)
    gout = guarded(n, torch.float32, soffs[0])
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ss.ss_adam_step(HP, n, *(v for _, v in st), rank_grads=G, param16=p16[1], g_out=gout[1], nonfinite_flag=flag)
    torch.cuda.synchronize()
    for (b, _), o in zip(st, soffs):
        assert intact(b, o, n)
    assert intact(p16[0], poff, n) and intact(gout[0], soffs[0], n)
    assert flag.item() == 0


def test_step_from_fp32_gradient_writes_only_its_arrays(ss):
    import torch
    n = 100_003
    g = guarded(n, torch.float32, 0, synth.normal(1e-3, synth.FP32, synth.GRAD, 0, 3))
    st = [guarded(n, torch.float32, 0, synth.normal(0.02, synth.FP32, synth.MASTER)) for _ in range(3)]
    p16 = guarded(n, torch.bfloat16, 3)   # param16 off phase: the per-thread form
    ss.ss_adam_step(HP, n, *(v for _, v in st), g32=g[1], param16=p16[1])
    torch.cuda.synchronize()
    assert all(intact(b, 0, n) for b, _ in st) and intact(p16[0], 3, n) and intact(g[0], 0, n)


REDUCE_FORMS = [  # (N, gradient view offset of rank r, output offset)
    (1, lambda r: 0, 0),             # vector: 4 + 4 elements a lane (accumulating: stored through shared memory)
    (2, lambda r: 0, 0),             # vector: stored through shared memory (accumulating: 4 + 4 a lane)
    (4, lambda r: 0, 0),             # vector, chunked
    (16, lambda r: 0, 0),            # vector, grid-stride
    (1, lambda r: 1, 0),             # shifted, four runs a warp at a time
    (3, lambda r: 2, 0),             # shifted, two runs at a time (one accumulating)
    (6, lambda r: 1, 0),             # shifted, batches of rank chunks
    (8, lambda r: 5, 0),             # shifted, double-buffered
    (8, lambda r: 0, 3),             # the output off the ranks' phase
    (3, lambda r: (r % 7) + 1, 0),   # mixed phases, two runs at a time (accumulating: batches of rank chunks)
    (4, lambda r: (r % 7) + 1, 0),   # mixed phases, batches of rank chunks
    (8, lambda r: (r % 7) + 1, 0),   # mixed phases, double-buffered
    (12, lambda r: (r % 7) + 1, 0),  # mixed phases, batches of rank chunks
    (4, lambda r: (r % 7) + 1, 1),   # mixed phases, the output one float past a boundary (3 head elements)
]


@pytest.mark.parametrize("form", range(len(REDUCE_FORMS)))
@pytest.mark.parametrize("n", [37, 100_003])
@pytest.mark.parametrize("accumulate", [False, True])
def test_reduce_writes_only_its_output(ss, form, n, accumulate):
    import torch
    N, goff, ooff = REDUCE_FORMS[form]
    G = grads(n, N, goff)
    out = guarded(n, torch.float32, ooff, synth.normal(1e-2, synth.FP32, synth.MOM1))
    ss.ss_grad_reduce(G, n, out[1], post_scale=0.5, accumulate=accumulate)
    torch.cuda.synchronize()
    assert intact(out[0], ooff, n)


@pytest.mark.parametrize("N,goff,ooff", [(2, 0, 0), (2, 0, 1), (8, 0, 2), (8, 0, 3), (64, 0, 1), (4, 1, 0),
                                         (4, 3, 0)])
@pytest.mark.parametrize("n", [37, 100_003])
def test_sumsq_writes_only_g_out(ss, N, goff, ooff, n):
    """g_out aligned (staged through shared memory in the per-rank-count tiles), 1-3 floats off the
    gradients' phase (realigned between lanes for the per-rank-count tiles, element by element for
    the general ones), and the gradients off g_out's phase."""
    import torch
    G = grads(n, N, lambda r: goff)
    g_out = guarded(n, torch.float32, ooff)
    ws = torch.empty(ss.ss_grad_sumsq_workspace(n) // 8, dtype=torch.float64, device="cuda")
    acc = torch.zeros(1, dtype=torch.float64, device="cuda")
    ss.ss_grad_sumsq(n, acc, ws, rank_grads=G, g_out=g_out[1])
    torch.cuda.synchronize()
    assert intact(g_out[0], ooff, n)
    assert acc.item() > 0


@pytest.mark.parametrize("P,N", [(37, 3), (100_003, 8), (4099, 64)])
@pytest.mark.parametrize("foff", [0, 1, 5])
def test_copies_write_only_their_buffers(ss, P, N, foff):
    import torch
    _, b = ss.ss_flatten_layout([P], N)
    shards = [guarded(int(b[k + 1] - b[k]), torch.bfloat16, k % 3, synth.normal(1.0, synth.BF16, synth.PARAM16, k))
              for k in range(N)]
    flat = guarded(P, torch.bfloat16, foff)
    ss.ss_unshard([v for _, v in shards], b, flat[1])
    back = [guarded(int(b[k + 1] - b[k]), torch.bfloat16, (k + 1) % 4) for k in range(N)]
    ss.ss_reshard(flat[1], b, [v for _, v in back])
    torch.cuda.synchronize()
    assert intact(flat[0], foff, P)
    for k in range(N):
        n = int(b[k + 1] - b[k])
        assert intact(back[k][0], (k + 1) % 4, n)
        assert torch.equal(back[k][1].view(torch.int16), shards[k][1].view(torch.int16))
