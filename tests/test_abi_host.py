"""The C ABI library without a GPU: it loads, exports every declared symbol, its
host-side layout and accounting agree with the oracle bit for bit, and argument
errors are reported before anything is launched."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from synth import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ss():
    import fsdp_sharded_mixed_ss_gb300 as m
    return m


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(ss_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(ss):
    names = declared_functions()
    assert {"ss_flatten_layout", "ss_grad_reduce", "ss_adam_step", "ss_unshard"} <= set(names)
    lib = ctypes.CDLL(ss.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert ss.ss_abi_version() == 2


@pytest.mark.parametrize("numels,N", [(workloads.tiny_mlp_numels(), 4), (workloads.gpt2_small_numels(), 8),
                                      (workloads.llama3_8b_numels(), 8), (workloads.llama70b_layer_numels(), 64),
                                      ([5, 0, 3], 7), ([], 3), ([1], 1024)])
def test_layout_matches_oracle(ss, numels, N):
    o1, b1 = ss.ss_flatten_layout(numels, N)
    o2, b2 = oracle.flatten_layout(numels, N)
    assert np.array_equal(o1, o2) and np.array_equal(b1, b2)
    P = int(o1[-1])
    for k in range(N):
        assert ss.ss_shard_segments(o1, b1, k) == oracle.shard_segments(o2, b2, k)
    rng = np.random.default_rng(N)
    for i in list(rng.integers(0, max(P, 1), size=200)) + [0, P - 1, P, -1]:
        assert ss.ss_shard_of(P, N, int(i)) == oracle.shard_of(P, N, int(i))


def test_layout_brute_force_small(ss):
    for P in range(0, 120):
        for N in range(1, 40):
            _, b1 = ss.ss_flatten_layout([P], N)
            _, b2 = oracle.flatten_layout([P], N)
            assert np.array_equal(b1, b2)
            for i in range(P):
                assert ss.ss_shard_of(P, N, i) == oracle.shard_of(P, N, i)


def test_state_bytes_match_oracle(ss):
    for P, N, M in [(7 * 10**9, 8, 32), (13 * 10**9, 8, 1), (175 * 10**9, 64, 1), (1, 1, 1), (0, 3, 2)]:
        assert ss.ss_state_bytes(P, N, M) == oracle.state_bytes(P, N, M)


def test_layout_errors(ss):
    with pytest.raises(ss.SSError) as e:
        ss.ss_flatten_layout([3, -1], 2)
    assert e.value.status == 1
    with pytest.raises(ss.SSError) as e:
        ss.ss_flatten_layout([2**62, 2**62], 2)
    assert e.value.status == 5
    with pytest.raises(ss.SSError):
        ss.ss_flatten_layout([3], 0)


HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1)
# fake, never dereferenced device addresses: every call below fails its host-side checks
A, B, C, D = 0x10000000, 0x20000000, 0x30000000, 0x40000000


def test_step_argument_errors_before_launch(ss):
    n = 1000
    ranks = [0x50000000, 0x60000000]
    def step(**kw):
        args = dict(rank_grads=ranks, gdtype=ss.SS_BF16, param16=D, pdtype=ss.SS_BF16, stream=0)
        args.update(kw)
        hp = args.pop("hp", HP)
        nn = args.pop("n", n)
        master, m, v = args.pop("master", A), args.pop("m", B), args.pop("v", C)
        ss.ss_adam_step(hp, nn, master, m, v, **args)

    cases = [
        (dict(n=-1), 1), (dict(hp=dict(HP, step=0)), 1), (dict(hp=dict(HP, beta1=1.0)), 1),
        (dict(hp=dict(HP, lr=float("nan"))), 1), (dict(master=0), 1),
        (dict(gdtype=ss.SS_FP32), 4), (dict(pdtype=ss.SS_FP32), 4),
        (dict(master=A + 2), 2), (dict(param16=D + 1), 2), (dict(rank_grads=[0x50000001]), 2),
        (dict(m=A + 4 * 10), 3), (dict(param16=C + 100), 3), (dict(rank_grads=[A]), 3),
        (dict(rank_grads=[]), 1), (dict(rank_grads=[0x50000000] * 1025), 1), (dict(n=2**62), 5),
    ]
    for kw, status in cases:
        with pytest.raises(ss.SSError) as e:
            step(**kw)
        assert e.value.status == status, (kw, e.value)
    step(n=0)   # nothing to do: no launch, no error


def test_reduce_and_copy_argument_errors(ss):
    with pytest.raises(ss.SSError) as e:
        ss.ss_grad_reduce([A, B], 100, C + 1, gdtype=ss.SS_BF16, stream=0)
    assert e.value.status == 2
    with pytest.raises(ss.SSError) as e:
        ss.ss_grad_reduce([A, B], 100, A + 8, gdtype=ss.SS_BF16, stream=0)
    assert e.value.status == 3
    ss.ss_grad_reduce([A, B], 0, C, gdtype=ss.SS_BF16, stream=0)
    _, b = oracle.flatten_layout([100], 4)
    with pytest.raises(ss.SSError) as e:
        ss.ss_unshard([A, B, C, D], b, A + 10, dtype=ss.SS_BF16, stream=0)
    assert e.value.status == 3
    with pytest.raises(ss.SSError) as e:
        ss.ss_unshard([A, B, C, D], b, 0x70000001, dtype=ss.SS_BF16, stream=0)
    assert e.value.status == 2
    with pytest.raises(ss.SSError) as e:
        ss.ss_unshard([A, B, C, D], np.array([0, 30, 20, 60, 100]), 0x70000000, dtype=ss.SS_BF16, stream=0)
    assert e.value.status == 1
    with pytest.raises(ss.SSError) as e:
        ss.ss_reshard(0x70000000, b, [A, B, C, D], dtype=7, stream=0)
    assert e.value.status == 4


def test_sumsq_and_clip_argument_errors(ss):
    n = 10_000
    ws = ss.ss_grad_sumsq_workspace(n)
    assert ws == 8 * ((n + 16383) // 16384 + 2) and ss.ss_grad_sumsq_workspace(-1) == -1
    W, O = 0x70000000, 0x71000000
    with pytest.raises(ss.SSError) as e:            # workspace too small
        ss.ss_grad_sumsq(n, O, W, rank_grads=[A, B], gdtype=ss.SS_BF16, workspace_bytes=ws - 8, stream=0)
    assert e.value.status == 1
    with pytest.raises(ss.SSError) as e:            # output inside the workspace
        ss.ss_grad_sumsq(n, W + 8, W, rank_grads=[A, B], gdtype=ss.SS_BF16, workspace_bytes=ws, stream=0)
    assert e.value.status == 3
    with pytest.raises(ss.SSError) as e:            # misaligned double output
        ss.ss_grad_sumsq(n, O + 4, W, rank_grads=[A, B], gdtype=ss.SS_BF16, workspace_bytes=ws, stream=0)
    assert e.value.status == 2
    with pytest.raises(ss.SSError) as e:
        ss.ss_clip_coef(O, 4, 0.0, O + 64, stream=0)
    assert e.value.status == 1
    with pytest.raises(ss.SSError) as e:
        ss.ss_clip_coef(O, 4, 1.0, O + 8, stream=0)  # coefficient overlaps the shard sums
    assert e.value.status == 3


def _header_defines():
    """The integer #defines of include/ss.h, evaluated the way the C preprocessor would for these
    simple forms (a literal, or an expression over earlier defines and an int64 cast)."""
    import re

    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ss.h")
    env = {}
    with open(path) as f:
        for line in f:
            m = re.match(r"#define\s+(SS_\w+)\s+(.+)$", line.strip())
            if not m:
                continue
            expr = m.group(2).replace("(int64_t)", "")
            try:
                env[m.group(1)] = int(eval(expr, {}, dict(env)))
            except Exception:  # not an integer expression
                pass
    return env


def test_noalloc_size_limit_rejected_on_host(ss):
    # n above the fixed scratch capacity is refused before anything touches a GPU
    with pytest.raises(ss.SSError) as e:
        ss.ss_grad_sumsq_noalloc(ss.SS_NOALLOC_SUMSQ_MAX_N + 1, 0x70000000, g32=0x71000000, stream=0)
    assert e.value.status == 5


def test_noalloc_limit_follows_the_header_and_the_workspace_rule(ss):
    """The binding's limit is the header's, and it is exactly the largest shard whose workspace
    (as the library itself sizes it) fits the fixed slot array."""
    d = _header_defines()
    slots, max_n = d["SS_NOALLOC_SUMSQ_SLOTS"], d["SS_NOALLOC_SUMSQ_MAX_N"]
    assert ss.SS_NOALLOC_SUMSQ_MAX_N == max_n
    assert ss.ss_grad_sumsq_workspace(max_n) <= 8 * slots
    assert ss.ss_grad_sumsq_workspace(max_n + 1) > 8 * slots
