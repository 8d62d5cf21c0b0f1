"""Helpers of the GPU parity tests: run a workload through the C ABI and through the oracle.

The CUDA side generates its inputs on the device with the `synth` generator;
the oracle side regenerates the same inputs on the host (same generator, same
counters) at the flat indices it checks. Nothing the oracle consumes comes from
the GPU.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth
from synth.workloads import Workload

BF16, FP16 = synth.BF16, synth.FP16


# ----------------------------------------------------------------------------- tolerances

def assert_state_close(gpu: np.ndarray, ref: np.ndarray, what: str, rel: float = 1e-6, abs_: float = 1e-9) -> dict:
    """|gpu - ref| <= max(rel * |ref|, abs_) elementwise; NaN positions must match."""
    gpu = np.asarray(gpu, dtype=np.float32)
    ref = np.asarray(ref, dtype=np.float32)
    assert gpu.shape == ref.shape
    gn, rn = np.isnan(gpu), np.isnan(ref)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ"
    g, r = gpu[~gn].astype(np.float64), ref[~rn].astype(np.float64)
    inf = np.isinf(r)
    assert np.array_equal(g[inf], r[inf]), f"{what}: infinities differ"
    g, r = g[~inf], r[~inf]
    d = np.abs(g - r)
    tol = np.maximum(rel * np.abs(r), abs_)
    bad = np.nonzero(d > tol)[0]
    assert bad.size == 0, f"{what}: {bad.size} elements out of tolerance, e.g. gpu={g[bad[0]]!r} ref={r[bad[0]]!r}"
    return {"n": int(r.size), "bit_equal": int((g == r).sum()), "max_rel": float((d / np.maximum(np.abs(r), 1e-30)).max(initial=0))}


def ordinal16(bits: np.ndarray) -> np.ndarray:
    """Order-preserving integer of a 16-bit float pattern (+0 and -0 both map to 0)."""
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def assert_p16_within_ulp(gpu_bits: np.ndarray, ref_bits: np.ndarray, dtype: int, what: str) -> dict:
    exp, man = (0x7F80, 0x007F) if dtype == BF16 else (0x7C00, 0x03FF)
    gn = ((gpu_bits & exp) == exp) & ((gpu_bits & man) != 0)
    rn = ((ref_bits & exp) == exp) & ((ref_bits & man) != 0)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ"
    d = np.abs(ordinal16(gpu_bits[~gn]) - ordinal16(ref_bits[~rn]))
    assert (d <= 1).all(), f"{what}: {(d > 1).sum()} elements more than 1 ulp apart"
    return {"n": int(d.size), "bit_equal": int((d == 0).sum())}


# ----------------------------------------------------------------------------- sampling

def sample_indices(lo: int, hi: int, k: int, seed: int) -> np.ndarray:
    """All of [lo, hi) when small, else both ends, 16-element runs and random points."""
    n = hi - lo
    if n <= k:
        return np.arange(lo, hi, dtype=np.int64)
    rng = np.random.default_rng(seed)
    ends = np.concatenate([np.arange(lo, lo + 64), np.arange(hi - 64, hi)])
    starts = rng.integers(lo, hi - 16, size=k // 64)
    runs = (starts[:, None] + np.arange(16)[None, :]).ravel()
    pts = rng.integers(lo, hi, size=k - ends.size - runs.size)
    return np.unique(np.concatenate([ends, runs, pts])).astype(np.int64)


# ----------------------------------------------------------------------------- oracle side

def oracle_shard(w: Workload, idx: np.ndarray, step_range) -> dict:
    """Oracle state at flat indices `idx` (all inside one stepped shard) after the given steps."""
    def f32(spec):
        return synth.host_gather(spec, idx).view(np.float32).copy() if spec is not None else np.zeros(idx.size, np.float32)

    master, m, v = f32(w.master), f32(w.m), f32(w.v)
    p16 = None
    for t in step_range:
        grads = [synth.host_gather(w.grad(r, t), idx) for r in range(w.n_ranks)]
        g = oracle.grad_reduce(grads, w.gdtype)
        hp = w.hp(t)
        p16 = oracle.adamw(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], t, g, master, m, v,
                           p16_dtype=w.gdtype)
    return {"master": master, "m": m, "v": v, "p16": p16}


# ----------------------------------------------------------------------------- GPU side

def torch_dtype(fmt: int):
    import torch

    return {BF16: torch.bfloat16, FP16: torch.float16}[fmt]


def gpu_run(w: Workload, device: str = "cuda:0", keep_grads: bool = False) -> dict:
    """Run the workload's steps (and unshard/reshard) through the C ABI; returns device tensors."""
    import torch

    import fsdp_sharded_mixed_ss_gb300 as ss

    N, P = w.n_ranks, w.P
    offs, bounds = ss.ss_flatten_layout(w.numels, N)
    gdt = torch_dtype(w.gdtype)
    n0 = int(bounds[1] - bounds[0])
    glen = P if w.per_rank_full else n0
    if not w.per_rank_full:
        assert w.shards == [0]
    G = [torch.empty(glen, dtype=gdt, device=device) for _ in range(N)]
    state = {}
    for k in w.shards:
        lo, hi = int(bounds[k]), int(bounds[k + 1])
        st = {}
        for name, spec in (("master", w.master), ("m", w.m), ("v", w.v)):
            t = torch.zeros(hi - lo, dtype=torch.float32, device=device)
            if spec is not None and hi > lo:
                synth.device_fill(spec, t.view(torch.int32), start=lo)
            st[name] = t
        state[k] = st
    p16 = []
    for k in range(N):
        lo, hi = int(bounds[k]), int(bounds[k + 1])
        t = torch.zeros(hi - lo, dtype=gdt, device=device)
        if k not in w.shards and w.param16 is not None and hi > lo:
            synth.device_fill(w.param16(k), t.view(torch.int16), start=lo)
        p16.append(t)
    steps = range(w.first_step, w.first_step + w.warmup_steps + w.steps)
    for t in steps:
        for r in range(N):
            synth.device_fill(w.grad(r, t), G[r].view(torch.int16), start=0)
        for k in w.shards:
            lo, hi = int(bounds[k]), int(bounds[k + 1])
            views = [g[lo:hi] for g in G] if w.per_rank_full else G
            st = state[k]
            ss.ss_adam_step(w.hp(t), hi - lo, st["master"], st["m"], st["v"], rank_grads=views, param16=p16[k])
    out = {"bounds": bounds, "offsets": offs, "state": state, "p16": p16, "steps": steps}
    if w.unshard:
        flat = torch.empty(P, dtype=gdt, device=device)
        ss.ss_unshard(p16, bounds, flat)
        out["flat"] = flat
        if w.reshard:
            back = [torch.empty_like(x) for x in p16]
            ss.ss_reshard(flat, bounds, back)
            out["back"] = back
    if keep_grads:
        out["grads"] = G
    torch.cuda.synchronize()
    return out


def to_np_bits16(t) -> np.ndarray:
    import torch

    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def gather_np(t, idx_local: np.ndarray) -> np.ndarray:
    import torch

    ii = torch.from_numpy(idx_local.astype(np.int64)).to(t.device)
    return t.index_select(0, ii).cpu().numpy()


def compare_workload(w: Workload, out: dict, per_shard_samples: int, seed: int = 0) -> dict:
    """Check every stepped shard (sampled) and the unshard/reshard copies against the oracle."""
    import torch

    bounds = out["bounds"]
    stats = {}
    for k in w.shards:
        lo, hi = int(bounds[k]), int(bounds[k + 1])
        if hi == lo:
            continue
        idx = sample_indices(lo, hi, per_shard_samples, seed + k)
        ref = oracle_shard(w, idx, out["steps"])
        st = out["state"][k]
        loc = idx - lo
        for name in ("master", "m", "v"):
            stats[(k, name)] = assert_state_close(gather_np(st[name], loc), ref[name], f"shard {k} {name}")
        got16 = gather_np(out["p16"][k].view(torch.int16), loc).view(np.uint16)
        stats[(k, "p16")] = assert_p16_within_ulp(got16, ref["p16"], w.gdtype, f"shard {k} p16")
        if "flat" in out:
            flat16 = gather_np(out["flat"].view(torch.int16), idx).view(np.uint16)
            assert np.array_equal(flat16, got16), f"shard {k}: flat buffer differs from the shard's params"
    if "flat" in out:
        # the flat buffer is the concatenation of the shards (property at any size)
        assert torch.equal(out["flat"].view(torch.int16), torch.cat([x.view(torch.int16) for x in out["p16"]]))
        for k in range(w.n_ranks):
            lo, hi = int(bounds[k]), int(bounds[k + 1])
            if k in w.shards or hi == lo or w.param16 is None:
                continue
            idx = sample_indices(lo, hi, 4096, seed + 1000 + k)
            got = gather_np(out["flat"].view(torch.int16), idx).view(np.uint16)
            assert np.array_equal(got, synth.host_gather(w.param16(k), idx)), f"unshard of shard {k}"
    if "back" in out:
        for k in range(w.n_ranks):
            assert torch.equal(out["back"][k].view(torch.int16), out["p16"][k].view(torch.int16)), f"reshard {k}"
    return stats
