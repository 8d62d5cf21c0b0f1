#!/usr/bin/env python3
"""Benchmark of the fused shard step on GB300.

Workload (one "step" = one pass of the whole hot path): the Llama-3-8B unit
(8,030,261,248 parameters in 291 tensors, module order) flattened and cut at
floor(kP/8) into N = 8 virtual-rank shards of 1,003,782,656 elements. Rank 0's
shard runs the fused kernel -- the rank-ordered fp32 sum of the 8 ranks' bf16
gradients (N(0, 1e-4) with 1% of entries x100), AdamW on fp32 master/m/v and
the bf16 cast -- then the unshard copy gathers the 8 bf16 shards into the flat
unit buffer. Inputs are synthetic (seeded generator; its "N(0, s)" is an
Irwin-Hall sum of twelve uniforms, support +-6s, truncated onto the bf16 grid)
and resident in HBM; one step moves 74.3 GB, far above the 129 MB L2, so no L2
flush is needed.

Metric: algorithmic HBM bytes of the step / step time (GB/s), with params/s
(shard elements updated per second). Each kernel is also timed alone, back to
back, and reported with its roofline fraction against the measured HBM copy
bandwidth; the two per-kernel times must add up to the step time. Secondary
blocks time the GPT-2 small rank-0 shard step + unshard and the Llama-70B layer
(64 fp16 shard steps + unshard + reshard) the same way.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With N > 1 (launched by torch.distributed.run) every rank runs its own
independent unit on its own GPU (weak scaling, no data-path collective); the
time is the max over ranks and the value the sum of all ranks' bytes.
`--impl reference` times the CPU oracle (the slow, plain C definition of the
same step) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused shard-step HBM GB/s and params/s (fraction of GB300 HBM peak), 1 GPU"
WORKLOAD = ("llama3-8b flat unit (8,030,261,248 params), N=8 virtual ranks: rank-0 shard (1,003,782,656 elements) "
            "fused reduce of 8 bf16 grads + AdamW + bf16 cast, then unshard of the 8 bf16 shards into the flat unit")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (e.g. under a profiler)")
    ap.add_argument("--no-secondary", action="store_true", help="skip the GPT-2 and Llama-70B layer blocks")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--suite", action="store_true",
                    help="instead of the benchmark line, time every kernel on the sweep and layer shapes")
    ap.add_argument("--suite-n", type=int, default=1 << 26, help="shard length of the --suite runs")
    ap.add_argument("--suite-pad", type=int, default=0, metavar="ELEMS",
                    help="allocate each rank's gradient buffer ELEMS elements longer than the shard (so the "
                         "buffers do not sit at power-of-two distances from each other)")
    ap.add_argument("--suite-only", default=None, metavar="REGEX",
                    help="time only the --suite entries whose name matches (e.g. for a small ncu capture)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers

def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def kernel_fingerprint() -> str:
    """SHA-256 of the fused step kernel's source: the per-element arithmetic header, the work
    division it takes its chunks from (the common header's section) and the double-buffered
    kernel's text in the CUDA source (from its comment block to the next kernel)."""
    import hashlib

    src = os.path.join(ROOT, "fsdp_sharded_mixed_ss_gb300", "csrc")
    with open(os.path.join(src, "ss_math.cuh"), "rb") as f:
        math = f.read()
    with open(os.path.join(src, "ss_common.cuh")) as f:
        common = f.read()
    with open(os.path.join(src, "ss_step.cu")) as f:
        text = f.read()
    c0 = common.index("// ------------------------------------------------------------------ work division")
    c1 = common.index("// Programmatic dependent launch", c0)
    start = text.index("// Register double-buffered form for small rank counts")
    end = text.index("adam_scalar_kernel(", start)
    return hashlib.sha256(math + common[c0:c1].encode() + text[start:end].encode()).hexdigest()


def profile_traffic(kernel: str, elements: int):
    """DRAM bytes per launch from the committed ncu record, while the record is for this kernel
    on a shard of this many elements and the kernel's source still matches it."""
    path = os.path.join(ROOT, "profiles", "adam_traffic.txt")
    if not os.path.exists(path):
        return None
    ent = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                ent[k.strip()] = v.strip()
    if ent.get("kernel") != kernel or ent.get("elements") != str(elements):
        return None
    if ent.get("source_sha256") != kernel_fingerprint():
        return None                     # the kernel changed since the counters were taken
    return int(ent["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) while the benchmark runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def _smi_id(self) -> str:
        # the device's UUID names the same physical GPU to nvidia-smi whatever CUDA_VISIBLE_DEVICES
        # does to ordinals; the ordinal is the fallback
        try:
            import torch

            u = getattr(torch.cuda.get_device_properties(self.index), "uuid", None)
            u = str(u) if u else ""
            u = u[4:] if u.startswith("GPU-") else u
            if len(u) == 36 and all(c in "0123456789abcdefABCDEF-" for c in u):  # a real (not masked) UUID
                return "GPU-" + u
        except Exception:  # no torch/CUDA here: fall back to the ordinal
            pass
        return str(self.index)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self._smi_id(), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        win = [s for (t, s) in self.samples if t0 <= t <= t1]
        window = "timed"
        if not win:
            win = [s for (_, s) in self.samples]
            window = "whole run"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[1]) for s in win if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4) if s[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(win[0][2]),
                "reasons": reasons, "samples": len(win), "window": window,
                "power_w_max": max((num(s[3]) or 0.0) for s in win)}


# ----------------------------------------------------------------------------- GPU arm

def unit_setup(w, device, stepped, state_whole_unit: bool = False):
    """Device buffers of one unit: the ranks' 16-bit gradients, fp32 master/m/v of the stepped
    shards, every shard's 16-bit parameters and the flat unit buffer, all from seeded streams.
    Gradients hold the full unit per rank when `w.per_rank_full`, else rank 0's shard only;
    with `state_whole_unit` master/m/v are unit-wide arrays viewed per shard."""
    import torch

    import fsdp_sharded_mixed_ss_gb300 as ss
    import synth

    N, P = w.n_ranks, w.P
    _, bounds = ss.ss_flatten_layout(w.numels, N)
    bounds = [int(x) for x in bounds]
    dt = torch.bfloat16 if w.gdtype == synth.BF16 else torch.float16
    glen = P if w.per_rank_full else bounds[1]
    grads = torch.empty((N, glen), dtype=dt, device=device)
    for r in range(N):
        synth.device_fill(w.grad(r, 1), grads[r].view(torch.int16))
    lo_all, hi_all = (0, P) if state_whole_unit else (bounds[stepped[0]], bounds[stepped[-1] + 1])
    st = []
    for i in range(3):
        t = torch.zeros(hi_all - lo_all, dtype=torch.float32, device=device)
        if i == 0:
            synth.device_fill(w.master, t.view(torch.int32), start=lo_all)
        st.append(t)
    shards = []
    for k in range(N):
        t = torch.empty(bounds[k + 1] - bounds[k], dtype=dt, device=device)
        synth.device_fill(w.param16(k) if w.param16 is not None else synth.normal(0.02, w.gdtype, synth.PARAM16, k),
                          t.view(torch.int16), start=bounds[k])
        shards.append(t)
    flat = torch.empty(P, dtype=dt, device=device)
    torch.cuda.synchronize(device)

    def shard_args(k):
        lo, hi = bounds[k], bounds[k + 1]
        views = [grads[r, lo:hi] for r in range(N)] if w.per_rank_full else [grads[r] for r in range(N)]
        return hi - lo, [x[lo - lo_all:hi - lo_all] for x in st], views

    return dict(w=w, N=N, P=P, bounds=bounds, grads=grads, state=st, shards=shards, flat=flat,
                stepped=list(stepped), shard_args=shard_args)


def step_bytes(u) -> dict:
    """Algorithmic bytes of one step: the fused kernel reads N x 2 B of gradients and 12 B of state
    and writes 12 B of state and 2 B of parameters per shard element; a copy moves 2 B in and 2 B
    out per element of the unit."""
    N, b = u["N"], u["bounds"]
    adam = sum((b[k + 1] - b[k]) * (2 * N + 26) for k in u["stepped"])
    return {"adam": adam, "copy": 4 * u["P"]}


def max_over_ranks(values, device=None):
    """Element-wise max of per-rank timings over the process group (the job is as slow as its
    slowest rank); identity without a group. Host bookkeeping only, not the data path."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_gbs(bytes_per_rank_step: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank moves its own unit's bytes each step (weak scaling)."""
    return bytes_per_rank_step * world / (ms_per_step * 1e-3) / 1e9


def timed_block(fn, reps: int, stream) -> float:
    """Mean ms of `reps` back-to-back calls of fn, between two CUDA events on `stream` (the
    stream every call launches on), synchronised on both sides."""
    import torch

    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def kernel_split(parts: dict, step_ms: float, peak: float) -> dict:
    """Per-kernel timings of a step (each kernel timed alone, back to back) with their GB/s and
    fractions of the copy peak, and the check that they add up to the step's own time."""
    out = {}
    total = 0.0
    for name, (ms, nbytes, launches) in parts.items():
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms_per_step": round(ms, 5), "launches_per_step": launches,
                     "avg_launch_ms": round(ms / launches, 5), "bytes_per_step": nbytes,
                     "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4)}
        total += ms
    out["sum_check"] = {"sum_ms": round(total, 5), "step_ms": round(step_ms, 5),
                        "ratio": round(total / step_ms, 4), "within_5pct": abs(total / step_ms - 1.0) <= 0.05}
    return out


def run_step_loop(step, steps: int, warmup: int, stream):
    """W untimed steps, then the mean ms of K steps between two events."""
    import torch

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    return timed_block(step, steps, stream)


def run_e2e(u, steps: int, device, t_counter):
    """Steps through the public API with every step's gradients copied in from pinned host memory
    and the step's result -- the fused step's non-finite-gradient flag, the found-inf value a
    mixed-precision loop reads each step -- read back to the host. Three streams: the host-to-
    device copy of step i+1 and the device-to-host copy of step i-1 overlap step i (double-
    buffered device gradients). Returns (ms per step, H2D GB/s alone, input bytes per step)."""
    import torch

    import fsdp_sharded_mixed_ss_gb300 as ss

    w, N, b = u["w"], u["N"], u["bounds"]
    n = b[1] - b[0]
    src = u["grads"][:, :n]
    host_in = torch.empty((N, n), dtype=src.dtype, pin_memory=True)
    nbytes = host_in.numel() * host_in.element_size()
    host_in.copy_(src)
    dev_in = [src.contiguous() if u["w"].per_rank_full else u["grads"],
              torch.empty((N, n), dtype=src.dtype, device=device)]
    flags = [torch.zeros(1, dtype=torch.int32, device=device) for _ in range(2)]
    host_out = [torch.full((1,), -1, dtype=torch.int32, pin_memory=True) for _ in range(2)]
    s_cmp, s_d2h = (torch.cuda.Stream(device) for _ in range(2))
    # the gradients go in as 256 MB pieces spread over four copy streams (measured on GB300:
    # back-to-back pieces on one stream moved ~105 GB/s, four streams or one 16 GB copy ~210 GB/s)
    s_h2d = [torch.cuda.Stream(device) for _ in range(4)]
    piece = 256 << 20
    src_b = host_in.view(torch.uint8).view(-1)
    dst_b = [d.view(torch.uint8).view(-1) for d in dev_in]
    done = {"h2d": {}, "cmp": {}, "d2h": {}}
    n0, st, _ = u["shard_args"](0)

    def mark(kind, i, s):
        e = torch.cuda.Event()
        e.record(s)
        done[kind][i] = e

    def copy_in(j, after=None):
        evs = []
        for q, s in enumerate(s_h2d):
            if after is not None:
                s.wait_event(after)
            with torch.cuda.stream(s):
                for o in range(q * piece, nbytes, len(s_h2d) * piece):
                    dst_b[j][o:o + piece].copy_(src_b[o:o + piece], non_blocking=True)
            e = torch.cuda.Event()
            e.record(s)
            evs.append(e)
        return evs

    def step(i):
        j = i % 2
        t = t_counter[0]
        t_counter[0] += 1
        evs = copy_in(j, done["cmp"].get(i - 2))          # dev_in[j] no longer read by step i - 2
        done["h2d"][i] = evs[-1]
        for e in evs:
            s_cmp.wait_event(e)
        if i - 2 in done["d2h"]:
            s_cmp.wait_event(done["d2h"][i - 2])          # flags[j] already copied out
        with torch.cuda.stream(s_cmp):
            flags[j].zero_()
        ss.ss_adam_step(w.hp(t), n0, *st, rank_grads=[dev_in[j][r] for r in range(N)],
                        param16=u["shards"][0], nonfinite_flag=flags[j], stream=s_cmp)
        ss.ss_unshard(u["shards"], b, u["flat"], stream=s_cmp)
        mark("cmp", i, s_cmp)
        s_d2h.wait_event(done["cmp"][i])
        with torch.cuda.stream(s_d2h):
            host_out[j].copy_(flags[j], non_blocking=True)
        mark("d2h", i, s_d2h)

    for i in range(3):
        step(i)
    torch.cuda.synchronize(device)
    for d in done.values():
        d.clear()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_h2d[0])
    for s in s_h2d[1:]:
        s.wait_event(e0)
    for i in range(steps):
        step(i)
    for s in s_h2d:
        s_d2h.wait_stream(s)
    s_d2h.wait_stream(s_cmp)
    e1.record(s_d2h)
    torch.cuda.synchronize(device)
    e2e_ms = e0.elapsed_time(e1) / steps
    if any(int(h.item()) != 0 for h in host_out):
        raise RuntimeError("e2e: a step flagged non-finite gradients on finite synthetic inputs")
    cur = torch.cuda.current_stream(device)

    def copy_alone():
        a = torch.cuda.Event()
        a.record(cur)
        for e in copy_in(1, a):
            cur.wait_event(e)

    copy_alone()
    h2d_ms = timed_block(copy_alone, 3, cur)
    del dev_in
    return e2e_ms, nbytes / (h2d_ms * 1e-3) / 1e9, nbytes


def unit_step_fn(u, stream, t_counter, copies=("unshard",)):
    """One step of the unit: the fused kernel on every stepped shard, then the copies."""
    import fsdp_sharded_mixed_ss_gb300 as ss

    w = u["w"]
    args = [(k, *u["shard_args"](k)) for k in u["stepped"]]

    def adam():
        t = t_counter[0]
        t_counter[0] += 1
        hp = w.hp(t)
        for k, n, st, views in args:
            ss.ss_adam_step(hp, n, *st, rank_grads=views, param16=u["shards"][k], stream=stream)

    def unshard():
        ss.ss_unshard(u["shards"], u["bounds"], u["flat"], stream=stream)

    def reshard():
        ss.ss_reshard(u["flat"], u["bounds"], u["shards"], stream=stream)

    fns = {"adam": adam, "unshard": unshard, "reshard": reshard}

    def step():
        adam()
        for c in copies:
            fns[c]()

    return step, fns


def time_unit(u, args, stream, peak, copies=("unshard",)):
    """Step loop, then each kernel of the step alone (back to back, as many launches)."""
    t_counter = [1]
    step, fns = unit_step_fn(u, stream, t_counter, copies)
    ms = run_step_loop(step, args.steps, args.warmup, stream)
    nb = step_bytes(u)
    parts = {"adam": (timed_block(fns["adam"], args.steps, stream), nb["adam"], len(u["stepped"]))}
    for c in copies:
        parts[c] = (timed_block(fns[c], args.steps, stream), nb["copy"], 1)
    total = nb["adam"] + nb["copy"] * len(copies)
    return ms, total, kernel_split(parts, ms, peak)


def secondary_blocks(args, device, stream, peak) -> dict:
    """The GPT-2 small rank-0 shard step + unshard, and the Llama-70B layer: all 64 fp16 shards
    stepped (one launch each) + unshard + reshard of the flat layer buffer."""
    import torch

    from synth import workloads

    out = {}
    for key, w, stepped, copies, steps in (
            ("gpt2_small_rank0_shard_N8", workloads.gpt2_small(), [0], ("unshard",), max(args.steps, 50)),
            ("llama70b_layer_N64_fp16_all_shards", workloads.llama70b_layer(), list(range(64)),
             ("unshard", "reshard"), max(min(args.steps, 10), 3))):
        u = unit_setup(w, device, stepped, state_whole_unit=len(stepped) > 1)
        a = argparse.Namespace(steps=steps, warmup=max(args.warmup, 3))
        ms, total, split = time_unit(u, a, stream, peak, copies)
        n = sum(u["bounds"][k + 1] - u["bounds"][k] for k in stepped)
        out[key] = {"workload": w.name, "unit_params": u["P"], "virtual_ranks": u["N"], "stepped_elems": n,
                    "steps": steps, "ms_per_step": round(ms, 5), "bytes_per_step": total,
                    "GB/s": round(total / (ms * 1e-3) / 1e9, 1), "frac": round(total / (ms * 1e-3) / 1e9 / peak, 4),
                    "params_per_s": round(n / (ms * 1e-3), 1), "kernels": split}
        del u
        torch.cuda.empty_cache()
    return out


def run_ours(args, rank: int, world: int, device):
    import torch
    import torch.distributed as dist

    from synth import workloads

    w = workloads.llama3_8b_shard()
    u = unit_setup(w, device, [0])
    stream = torch.cuda.current_stream(device)
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"]

    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    t_counter = [1]
    step, fns = unit_step_fn(u, stream, t_counter)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    if world > 1:
        dist.barrier()
    h0 = time.time()
    elapsed_ms = timed_block(step, args.steps, stream) * args.steps
    h1 = time.time()
    if world > 1:
        dist.barrier()
    # each kernel of the step alone, back to back, as many launches as timed steps
    adam_ms = timed_block(fns["adam"], args.steps, stream)
    copy_ms = timed_block(fns["unshard"], args.steps, stream)
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(h0, h1)

    nb = step_bytes(u)
    n = u["bounds"][1]
    elapsed_ms, adam_ms, copy_ms = max_over_ranks([elapsed_ms, adam_ms, copy_ms], device if world > 1 else None)
    ms_per_step = elapsed_ms / args.steps
    per_step = nb["adam"] + nb["copy"]
    split = kernel_split({"adam_pipe_kernel": (adam_ms, nb["adam"], 1),
                          "copy_segments_kernel": (copy_ms, nb["copy"], 1)}, ms_per_step, peak)
    chk = split["sum_check"]
    print(f"bench: per-kernel times {adam_ms:.4f} + {copy_ms:.4f} = {chk['sum_ms']:.4f} ms against the step's "
          f"{ms_per_step:.4f} ms (ratio {chk['ratio']:.4f}, {'within' if chk['within_5pct'] else 'NOT within'} 5%)",
          file=sys.stderr, flush=True)
    value = job_gbs(per_step, world, ms_per_step)
    achieved = nb["adam"] / (adam_ms * 1e-3) / 1e9
    copy_gbs = nb["copy"] / (copy_ms * 1e-3) / 1e9
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "unit_params": u["P"], "virtual_ranks": u["N"], "shard_elems": n,
                   "grad_dtype": "bf16", "param_dtype": "bf16", "state_dtype": "f32",
                   "grads": "N(0,1e-4) (Irwin-Hall approximation), 1% of entries x100; master N(0,0.02); m=v=0",
                   "bytes_per_step": per_step, "adam_bytes_per_step": nb["adam"], "unshard_bytes_per_step": nb["copy"],
                   "l2": f"inputs larger than L2 ({per_step / 1e9:.1f} GB moved per step vs 129 MB L2); no flush"},
        "params_per_s": round(n * world / (ms_per_step * 1e-3), 1),
        "unit_params_per_s": round(u["P"] * world / (ms_per_step * 1e-3), 1),
        "roofline": {"kernel": "adam_pipe_kernel (fused reduce of 8 bf16 ranks + AdamW + bf16 cast)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profile_traffic("adam_pipe_kernel", n),
                     "algorithmic_bytes": nb["adam"], "avg_launch_ms": round(adam_ms, 5),
                     "timing": f"{args.steps} back-to-back launches between CUDA events on the launching stream",
                     "peak_source": peaks["source"]},
        "roofline_unshard": {"kernel": "copy_segments_kernel (unshard of 8 bf16 shards into the flat unit)",
                             "bound": "hbm", "achieved": round(copy_gbs, 1), "peak": peak, "unit": "GB/s",
                             "frac": round(copy_gbs / peak, 4), "algorithmic_bytes": nb["copy"],
                             "avg_launch_ms": round(copy_ms, 5)},
        "kernels": split,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    if not args.no_e2e:
        # end to end through the public API with host buffers: the step's gradients in from
        # pinned host memory, the step's result (its non-finite flag) out, every step
        e2e_ms, h2d_gbs, in_bytes = run_e2e(u, args.e2e_steps, device, t_counter)
        e2e_ms = max_over_ranks([e2e_ms], device if world > 1 else None)[0]
        result["e2e"] = {"value": round(per_step * world / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                         "ms_per_step": round(e2e_ms, 4), "steps": args.e2e_steps, "h2d_bytes_per_step": in_bytes,
                         "d2h_bytes_per_step": 4, "h2d_gbs": round(h2d_gbs, 1),
                         "result": "the step's non-finite-gradient flag (int32), read back every step",
                         "pipeline": "h2d of step i+1 (256 MB pieces over 4 copy streams) and d2h of step i-1 "
                                     "overlap step i (double-buffered device gradients)"}
    del u, fns, step
    torch.cuda.empty_cache()
    if not args.no_secondary:
        result["secondary"] = secondary_blocks(args, device, stream, peak)
    return result


# ----------------------------------------------------------------------------- kernel suite

def run_suite(args, device) -> dict:
    """Mean CUDA-event time and algorithmic GB/s of each kernel on synthetic shards."""
    import torch

    import fsdp_sharded_mixed_ss_gb300 as ss
    import synth

    def timed(fn, reps=30):
        # back-to-back launches between two events: the host stays ahead of the GPU, so
        # the time is the kernels' own, not the host's launch latency
        for _ in range(3):
            fn()
        torch.cuda.synchronize(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize(device)
        return a.elapsed_time(b) / reps

    def entry(ms, nbytes):
        return {"ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}

    def want(*names):
        return args.suite_only is None or any(re.search(args.suite_only, k) for k in names)

    out = {"peak_hbm_gbs": measured_peaks()["hbm_gbs"], "n": args.suite_n, "pad": args.suite_pad}
    n = args.suite_n
    hp = dict(lr=3e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, step=1000)
    st = []
    for spec in (synth.normal(0.02, synth.FP32, synth.MASTER), synth.normal(1e-4, synth.FP32, synth.MOM1),
                 synth.normal(1e-8, synth.FP32, synth.MOM2, absolute=True)):
        t = torch.empty(n, dtype=torch.float32, device=device)
        synth.device_fill(spec, t.view(torch.int32))
        st.append(t)
    p16 = torch.empty(n, dtype=torch.bfloat16, device=device)
    g32 = torch.empty(n, dtype=torch.float32, device=device)
    synth.device_fill(synth.normal(1e-3, synth.FP32, synth.GRAD, 0, 1), g32.view(torch.int32))
    if want("adam_step_fp32_grad"):
        out["adam_step_fp32_grad"] = entry(timed(lambda: ss.ss_adam_step(hp, n, *st, g32=g32, param16=p16)), 30 * n)
    ws = torch.empty(max(ss.ss_grad_sumsq_workspace(n) // 8, 1), dtype=torch.float64, device=device)
    acc = torch.empty(1, dtype=torch.float64, device=device)
    if want("grad_sumsq_fp32_grad"):
        # the clip pass over an fp32 gradient (accumulated micro-batches), before a step from g32
        out["grad_sumsq_fp32_grad"] = entry(timed(lambda: ss.ss_grad_sumsq(n, acc, ws, g32=g32)), 4 * n)
    extra8 = ("adam_step_N8_grads_off_by_one", "grad_reduce_accumulate_N8", "adam_step_N8_fp16_unscale_flag_skip",
              "adam_step_N8_param16_into_flat")
    for N in (2, 8, 64):
        off = f"adam_step_N{N}_grads_off_by_one"
        mixed = f"adam_step_N{N}_grads_mixed_phase"
        if not want(f"adam_step_N{N}", f"grad_reduce_N{N}", f"grad_sumsq_N{N}", off, mixed,
                    f"grad_reduce_N{N}_grads_off_by_one", f"grad_sumsq_gout_N{N}_grads_off_by_one",
                    *(extra8 if N == 8 else ())):
            continue
        G = []
        for r in range(N):
            t = torch.empty(n + args.suite_pad, dtype=torch.bfloat16, device=device)[:n]
            synth.device_fill(synth.normal(1e-3, synth.BF16, synth.GRAD, r, 1), t.view(torch.int16))
            G.append(t)
        if want(f"adam_step_N{N}"):
            out[f"adam_step_N{N}"] = entry(timed(lambda: ss.ss_adam_step(hp, n, *st, rank_grads=G, param16=p16)),
                                           (2 * N + 26) * n)
        if want(f"grad_reduce_N{N}"):
            out[f"grad_reduce_N{N}"] = entry(timed(lambda: ss.ss_grad_reduce(G, n, g32)), (2 * N + 4) * n)
        if want(f"grad_sumsq_N{N}"):
            out[f"grad_sumsq_N{N}"] = entry(timed(lambda: ss.ss_grad_sumsq(n, acc, ws, rank_grads=G)), 2 * N * n)
        if want(f"grad_reduce_N{N}_grads_off_by_one", f"grad_sumsq_gout_N{N}_grads_off_by_one"):
            # the gradient views one element off the fp32 output's 16-byte phase
            Gm = [g[1:] for g in G]
            m1 = n - 1
            if want(f"grad_reduce_N{N}_grads_off_by_one"):
                out[f"grad_reduce_N{N}_grads_off_by_one"] = entry(
                    timed(lambda: ss.ss_grad_reduce(Gm, m1, g32[:m1])), (2 * N + 4) * m1)
            if want(f"grad_sumsq_gout_N{N}_grads_off_by_one"):
                out[f"grad_sumsq_gout_N{N}_grads_off_by_one"] = entry(
                    timed(lambda: ss.ss_grad_sumsq(m1, acc, ws, rank_grads=Gm, g_out=g32[:m1])), (2 * N + 4) * m1)
        if want(off):
            # gradient views one element off the state's 16-byte phase: the shifted-load kernels
            Gm = [g[1:] for g in G]
            m1 = n - 1
            out[off] = entry(
                timed(lambda: ss.ss_adam_step(hp, m1, *(t[:m1] for t in st), rank_grads=Gm, param16=p16[:m1])),
                (2 * N + 26) * m1)
        if want(mixed):
            # rank r's gradient view (r % 7) + 1 elements off the state's phase: every rank shifted by its own
            # phase (views into one stacked buffer whose row length is not a multiple of 8 look like this)
            m7 = n - 7
            Gx = [g[(r % 7) + 1:(r % 7) + 1 + m7] for r, g in enumerate(G)]
            out[mixed] = entry(
                timed(lambda: ss.ss_adam_step(hp, m7, *(t[:m7] for t in st), rank_grads=Gx, param16=p16[:m7])),
                (2 * N + 26) * m7)
        if N == 8 and want(extra8[1]):
            # next rows: gradient accumulation (read-modify-write of the fp32 gradient) ...
            out[extra8[1]] = entry(timed(lambda: ss.ss_grad_reduce(G, n, g32, accumulate=True)), (2 * N + 8) * n)
        if N == 8 and want(extra8[2]):
            # ... fp16 loss-scale unscaling with the overflow flag and the skip flag read ...
            G16 = [g.view(torch.float16) for g in G]   # the same bits read as fp16: finite, small
            flag = torch.zeros(2, dtype=torch.int32, device=device)   # [0]: this step's flag, [1]: skip
            out[extra8[2]] = entry(
                timed(lambda: ss.ss_adam_step(hp, n, *st, rank_grads=G16, post_scale=1.0 / 1024, param16=p16,
                                              nonfinite_flag=flag[0:1], dev_skip_flag=flag[1:2])), (2 * N + 26) * n)
            assert int(flag[0].item()) == 0
            del flag
        if N == 8 and want(extra8[3]):
            # ... and the 16-bit parameters written straight into a flat unit buffer at the shard's offset
            flat = torch.empty(n + 1024, dtype=torch.bfloat16, device=device)
            out[extra8[3]] = entry(
                timed(lambda: ss.ss_adam_step(hp, n, *st, rank_grads=G, param16=flat[1024:])), (2 * N + 26) * n)
            del flat
        del G
        torch.cuda.empty_cache()
    # the fused step with every rank's gradient view one element off the state's phase, across
    # rank counts (the shifted-load kernel forms)
    # (and with rank r's view (r % 7) + 1 elements off: every rank at its own phase)
    for key, offset in (("adam_step_off_by_one_by_ranks", lambda r: 1),
                        ("adam_step_mixed_phase_by_ranks", lambda r: (r % 7) + 1)):
        if not want(key):
            continue
        m7 = n - 7
        G = []
        for r in range(64):
            t = torch.empty(n + 8 + args.suite_pad, dtype=torch.bfloat16, device=device)
            synth.device_fill(synth.normal(1e-3, synth.BF16, synth.GRAD, r, 1), t.view(torch.int16))
            G.append(t[offset(r):offset(r) + m7])
        by_ranks = {}
        for N in (1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 16, 32, 64):
            Gn = G[:N]
            by_ranks[str(N)] = entry(timed(lambda: ss.ss_adam_step(hp, m7, *(t[:m7] for t in st), rank_grads=Gn,
                                                                  param16=p16[:m7])), (2 * N + 26) * m7)
        out[key] = by_ranks
        del G
    # the reduce across rank counts: aligned, and with every rank's view one element off the output's
    # phase (also accumulating into the output, and with rank r's view (r % 7) + 1 elements off)
    for key, offset, accum, ranks in (
            ("grad_reduce_by_ranks", lambda r: 0, False, (1, 2, 3, 4, 6, 8, 16)),
            ("grad_reduce_accumulate_by_ranks", lambda r: 0, True, (1, 2, 3, 4, 8)),
            ("grad_reduce_off_by_one_by_ranks", lambda r: 1, False, (1, 2, 3, 4, 5, 6, 7, 8, 9, 16, 64)),
            ("grad_reduce_accumulate_off_by_one_by_ranks", lambda r: 1, True, (1, 2, 3, 4, 6, 8, 16)),
            ("grad_reduce_mixed_phase_by_ranks", lambda r: (r % 7) + 1, False, (2, 3, 4, 6, 8, 12, 16, 64))):
        if not want(key):
            continue
        m7 = n - 7
        G = []
        for r in range(max(ranks)):
            t = torch.empty(n + 8, dtype=torch.bfloat16, device=device)
            synth.device_fill(synth.normal(1e-3, synth.BF16, synth.GRAD, r, 1), t.view(torch.int16))
            G.append(t[offset(r):offset(r) + m7])
        by_ranks = {}
        for N in ranks:
            Gn = G[:N]
            by_ranks[str(N)] = entry(timed(lambda: ss.ss_grad_reduce(Gn, m7, g32[:m7], accumulate=accum)),
                                     (2 * N + 4 + 4 * accum) * m7)
        out[key] = by_ranks
        del G
    # the sum of squares across rank counts: read-only, writing g_out, and writing g_out with every
    # rank's view one element off g_out's phase
    for key, off, gout in (("grad_sumsq_by_ranks", 0, False), ("grad_sumsq_gout_by_ranks", 0, True),
                           ("grad_sumsq_gout_off_by_one_by_ranks", 1, True)):
        if not want(key):
            continue
        m7 = n - 7
        G = []
        for r in range(64):
            t = torch.empty(n + 8, dtype=torch.bfloat16, device=device)
            synth.device_fill(synth.normal(1e-3, synth.BF16, synth.GRAD, r, 1), t.view(torch.int16))
            G.append(t[off:off + m7])
        by_ranks = {}
        for N in (1, 2, 3, 4, 5, 6, 7, 8, 9, 16, 64):
            Gn = G[:N]
            go = g32[:m7] if gout else None
            by_ranks[str(N)] = entry(timed(lambda: ss.ss_grad_sumsq(m7, acc, ws, rank_grads=Gn, g_out=go)),
                                     (2 * N + 4 * gout) * m7)
        out[key] = by_ranks
        del G
    # the fused step across the rank counts between (kernel forms and prefetch thresholds)
    if want("adam_step_by_ranks"):
        G = []
        for r in range(32):
            t = torch.empty(n + args.suite_pad, dtype=torch.bfloat16, device=device)[:n]
            synth.device_fill(synth.normal(1e-3, synth.BF16, synth.GRAD, r, 1), t.view(torch.int16))
            G.append(t)
        by_ranks = {}
        for N in (1, 3, 4, 5, 6, 7, 9, 10, 12, 13, 16, 24, 32):
            Gn = G[:N]
            by_ranks[str(N)] = entry(timed(lambda: ss.ss_adam_step(hp, n, *st, rank_grads=Gn, param16=p16)),
                                     (2 * N + 26) * n)
        out["adam_step_by_ranks"] = by_ranks
        del G
    del st, p16, g32, ws
    torch.cuda.empty_cache()
    out.update(run_config_steps(ss, device, timed, entry, want))
    for name, numels, N, dt in (("unshard_gpt2_small_N8", [124_439_808], 8, torch.bfloat16),
                                ("unshard_llama70b_layer_N64", [855_654_400], 64, torch.float16)):
        reshard = name.replace("unshard", "reshard")
        off_names = (name + "_flat_off_phase", reshard + "_flat_off_phase") if N == 8 else ()
        if not want(name, reshard, *off_names):
            continue
        _, b = ss.ss_flatten_layout(numels, N)
        P = int(b[-1])
        shards = [torch.zeros(int(b[k + 1] - b[k]), dtype=dt, device=device) for k in range(N)]
        flat = torch.empty(P, dtype=dt, device=device)
        if want(name):
            out[name] = entry(timed(lambda: ss.ss_unshard(shards, b, flat)), 4 * P)
        if want(reshard):
            out[reshard] = entry(timed(lambda: ss.ss_reshard(flat, b, shards)), 4 * P)
        if off_names and want(*off_names):
            # flat buffer one element off the shards' 16-byte phase: the SIMT copy with shifted loads
            base = torch.empty(P + 8, dtype=dt, device=device)
            off = base[1:P + 1]
            if want(off_names[0]):
                out[off_names[0]] = entry(timed(lambda: ss.ss_unshard(shards, b, off)), 4 * P)
            if want(off_names[1]):
                out[off_names[1]] = entry(timed(lambda: ss.ss_reshard(off, b, shards)), 4 * P)
            del base, off
        del shards, flat
        torch.cuda.empty_cache()
    return out


def run_config_steps(ss, device, timed, entry, want=lambda *names: True) -> dict:
    """The two large configurations at full size: the Llama-3-8B rank-0 shard (1,003,782,656
    elements, 8 bf16 ranks with outliers) and the Llama-70B layer stepped as one unit (855,654,400
    elements, 64 fp16 ranks, every shard at once, parameters written straight into the flat
    layer buffer: the whole unit's step without a separate unshard)."""
    import torch

    import synth
    from synth import workloads

    out = {}
    for w, whole_unit in ((workloads.llama3_8b_shard(), False), (workloads.llama70b_layer(), True)):
        key = f"{w.name}_{'unit_step_into_flat' if whole_unit else 'shard_step'}"
        if not want(key):
            continue
        _, b = ss.ss_flatten_layout(w.numels, w.n_ranks)
        n = int(b[-1]) if whole_unit else int(b[1])
        dt = torch.bfloat16 if w.gdtype == synth.BF16 else torch.float16
        G = []
        for r in range(w.n_ranks):
            t = torch.empty(n, dtype=dt, device=device)
            synth.device_fill(w.grad(r, 1), t.view(torch.int16))
            G.append(t)
        st = [torch.empty(n, dtype=torch.float32, device=device)]
        synth.device_fill(w.master, st[0].view(torch.int32))
        st += [torch.zeros(n, dtype=torch.float32, device=device) for _ in range(2)]
        p16 = torch.empty(n, dtype=dt, device=device)
        hp = w.hp(1)
        out[key] = entry(timed(lambda: ss.ss_adam_step(hp, n, *st, rank_grads=G, param16=p16), 5),
                         (2 * w.n_ranks + 26) * n)
        out[key]["elements"] = n
        del G, st, p16
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample_step(sample: int, reps: int):
    """Time the oracle's step on the headline workload's inputs: the rank-ordered reduce of the 8
    ranks' bf16 gradients + AdamW + bf16 cast on the first `sample` elements of rank 0's shard,
    then the unshard copy of the matching `sample`-element slice of each of the 8 shards."""
    import numpy as np

    import oracle
    import synth
    from synth import workloads

    w = workloads.llama3_8b_shard()
    N = w.n_ranks
    _, bounds = oracle.flatten_layout(w.numels, N)
    grads = [synth.host_range(w.grad(r, 1), 0, sample) for r in range(N)]
    master = synth.host_range(w.master, 0, sample).view(np.float32).copy()
    m = np.zeros(sample, np.float32)
    v = np.zeros(sample, np.float32)
    shards = [synth.host_range(w.param16(k), int(bounds[k]), sample) for k in range(N)]
    sb = np.arange(N + 1, dtype=np.int64) * sample
    times = []
    for t in range(1, reps + 1):
        t0 = time.perf_counter()
        g = oracle.grad_reduce(grads, oracle.BF16)
        hp = w.hp(t)
        shards[0] = oracle.adamw(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], t, g, master, m, v,
                                 p16_dtype=oracle.BF16)
        oracle.unshard(shards, sb)
        times.append(time.perf_counter() - t0)
    bytes_ = sample * (2 * N + 26) + 4 * sample * N
    return bytes_, times, oracle.max_threads()


def cpu_baseline(target_s: float = 12.0) -> dict:
    sample = 1 << 21
    b, times, cores = oracle_sample_step(sample, 2)
    per = max(times[-1], 1e-6)
    reps = max(3, min(5000, int(target_s / per)))
    b, times, cores = oracle_sample_step(sample, reps)
    gbs = b * len(times) / sum(times) / 1e9
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{sample} elements of the Llama-3-8B rank-0 shard (8 ranks' bf16 grads with outliers) + the "
                      f"matching {sample}-element slice of each of the 8 shards for the unshard copy; "
                      f"{len(times)} steps, {sum(times):.1f} s of CPU time"}


def run_reference(args):
    sample = 1 << 20
    b, times, cores = oracle_sample_step(sample, args.warmup + args.steps)
    timed = times[args.warmup:]
    ms = 1e3 * sum(timed) / len(timed)
    gbs = b / (ms * 1e-3) / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "unit_params": 8_030_261_248, "virtual_ranks": 8,
                   "shard_elems": 1_003_782_656, "sample_elems": sample},
        "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample} elements of the Llama-3-8B rank-0 shard + the matching slices of the "
                                   f"8 shards for the unshard, per step"},
        "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    import torch
    import torch.distributed as dist

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.suite:
        print(json.dumps({"suite": run_suite(args, device)}), flush=True)
        return
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    result = run_ours(args, rank, world, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
