"""Python binding of the GB300 shard-step library (libss.so).

Thin ctypes marshalling over the C ABI in ``include/ss.h``: the functions have
the C names, take torch tensors (or raw device addresses as ints) and enqueue
the library's CUDA kernels on torch's current stream. Every step of the path
runs in the library's kernels; this module only converts arguments. There is
no fallback: if ``libss.so`` is missing or fails to load, importing this
package raises.

The method is the per-shard training-state update of fully sharded data
parallel training ("FSDP: Fully Sharded Data Parallel Training at Scale"):
flatten and cut at floor(kP/N), sum the N virtual ranks' 16-bit gradients in
fp32, AdamW on the fp32 master/m/v, cast to 16-bit, unshard copy.
"""
from __future__ import annotations

import array
import ctypes
import os
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# SS_LIBRARY may name another build of the same library (e.g. one compiled with other tuning constants)
LIB_PATH = os.environ.get("SS_LIBRARY") or os.path.join(_HERE, "libss.so")

SS_BF16, SS_FP16, SS_FP32 = 0, 1, 2
SS_MAX_RANKS = 1024

STATUS = {0: "SS_OK", 1: "SS_ERR_INVALID_ARG", 2: "SS_ERR_ALIGN", 3: "SS_ERR_OVERLAP", 4: "SS_ERR_DTYPE",
          5: "SS_ERR_OVERFLOW", 6: "SS_ERR_CUDA"}


class SSError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)} ({_lib.ss_status_string(status).decode()})"
        if status == 6:
            msg += f": {_lib.ss_last_cuda_error().decode()}"
        super().__init__(msg)


class _Segment(ctypes.Structure):
    _fields_ = [("tensor", ctypes.c_int32), ("pad_", ctypes.c_int32), ("tensor_offset", ctypes.c_int64),
                ("shard_offset", ctypes.c_int64), ("length", ctypes.c_int64)]


BYTES_FIELDS = ["fp32_params", "fp32_grads", "fp32_adam", "fp32_total", "mp_params16", "mp_grads16",
                "mp_master32", "mp_adam32", "mp_total", "optimizer_state", "zero1_optimizer_per_gpu",
                "full_shard_per_gpu", "shard_grad_op_per_gpu", "no_shard_per_gpu", "unit_gather",
                "full_shard_peak", "full_shard_saving", "shard_grad_op_saving", "mp_full_shard_per_gpu",
                "mp_unit_gather16"]


class _Bytes(ctypes.Structure):
    _fields_ = [(f, ctypes.c_double) for f in BYTES_FIELDS]


class _HParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("pad_", ctypes.c_int32),
                ("step", ctypes.c_int64)]


class _Options(ctypes.Structure):
    _fields_ = [("g_out", ctypes.c_void_p), ("nonfinite_flag", ctypes.c_void_p),
                ("dev_grad_scale", ctypes.c_void_p), ("dev_skip_flag", ctypes.c_void_p)]


_NO_OPTIONS = _Options(None, None, None, None)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python fsdp_sharded_mixed_ss_gb300/_build.py` "
                          "(or __graft_entry__.build()) first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.ss_flatten_layout.argtypes = [vp, i32, i32, vp, vp]
    lib.ss_shard_segments.argtypes = [vp, i32, vp, i32, i32, vp, i32, ctypes.POINTER(i32)]
    lib.ss_shard_of.argtypes = [i64, i32, i64]
    lib.ss_shard_of.restype = i32
    lib.ss_state_bytes.argtypes = [i64, i32, i32, ctypes.POINTER(_Bytes)]
    lib.ss_grad_reduce.argtypes = [vp, i32, i32, i64, f32, i32, vp, vp, vp]
    lib.ss_adam_step.argtypes = [ctypes.POINTER(_HParams), i64, vp, vp, i32, i32, f32, vp, vp, vp, vp, i32,
                                 ctypes.POINTER(_Options), vp]
    lib.ss_unshard.argtypes = [vp, vp, i32, i32, vp, vp]
    lib.ss_reshard.argtypes = [vp, vp, i32, i32, vp, vp]
    lib.ss_status_string.argtypes = [i32]
    lib.ss_status_string.restype = ctypes.c_char_p
    lib.ss_last_cuda_error.restype = ctypes.c_char_p
    lib.ss_abi_version.restype = i32
    lib.ss_grad_sumsq_workspace.argtypes = [i64]
    lib.ss_grad_sumsq_workspace.restype = i64
    lib.ss_grad_sumsq.argtypes = [i64, vp, vp, i32, i32, f32, vp, vp, i64, vp, vp, vp]
    lib.ss_clip_coef.argtypes = [vp, i32, f32, vp, vp, vp]
    lib.ss_grad_sumsq_noalloc.argtypes = [i64, vp, vp, i32, i32, f32, vp, vp, vp, vp]
    return lib


_lib = _load()


def lib():
    """The loaded ctypes library (for callers that marshal their own arguments)."""
    return _lib


# ----------------------------------------------------------------------------- marshalling

_torch = None
_DTYPES = None
_RAW_STREAM = None
_GET_DEVICE = None


def _t():
    global _torch, _DTYPES, _RAW_STREAM, _GET_DEVICE
    if _torch is None:
        import torch

        _torch = torch
        _DTYPES = {torch.bfloat16: SS_BF16, torch.float16: SS_FP16, torch.float32: SS_FP32}
        # torch's own C entry points for the current device and the current stream's handle
        # (public equivalents are used when a torch build lacks them)
        _RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _GET_DEVICE = getattr(torch._C, "_cuda_getDevice", None)
        if _RAW_STREAM is None or _GET_DEVICE is None:
            _RAW_STREAM = _GET_DEVICE = None
    return _torch


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _dtype_of(t) -> int | None:
    if isinstance(t, int) or t is None:
        return None
    _t()
    return _DTYPES.get(t.dtype)


def _stream(stream, like=None) -> int | None:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    torch = _t()
    dev = like.device if (like is not None and not isinstance(like, int) and like.is_cuda) else None
    if _RAW_STREAM is not None:
        # the current stream's handle without building a torch Stream object (a few microseconds
        # per call, which small shards feel)
        return _RAW_STREAM(dev.index if dev is not None and dev.index is not None else _GET_DEVICE())
    return torch.cuda.current_stream(dev).cuda_stream


class _DeviceGuard:
    """Makes the tensors' device current for the call (the library sizes grids from it); a no-op
    when it already is."""

    __slots__ = ("dev", "ctx")

    def __init__(self, t):
        self.dev = None
        self.ctx = None
        if t is not None and not isinstance(t, int) and t.is_cuda:
            idx = t.device.index
            if idx is not None and idx != (_GET_DEVICE() if _GET_DEVICE is not None else _t().cuda.current_device()):
                self.dev = idx

    def __enter__(self):
        if self.dev is not None:
            self.ctx = _torch.cuda.device(self.dev)
            self.ctx.__enter__()

    def __exit__(self, *exc):
        if self.ctx is not None:
            self.ctx.__exit__(*exc)


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise SSError(rc, where)


def _ptr_array(xs) -> array.array:
    """The addresses of xs as a C array of 64-bit pointers (keep it alive across the call)."""
    if xs and not isinstance(xs[0], int):
        try:
            return array.array("Q", [x.data_ptr() for x in xs])
        except AttributeError:
            pass
    return array.array("Q", [x if isinstance(x, int) else x.data_ptr() for x in xs])


def _addr(a: array.array | None) -> int | None:
    return a.buffer_info()[0] if a is not None and len(a) else None


# ----------------------------------------------------------------------------- layout (host)

def ss_abi_version() -> int:
    return int(_lib.ss_abi_version())


def ss_flatten_layout(numels: Sequence[int], n_ranks: int):
    """(tensor_offsets[T+1], shard_bounds[N+1]) as int64 numpy arrays."""
    num = np.ascontiguousarray(np.asarray(numels, dtype=np.int64))
    offs = np.zeros(num.size + 1, dtype=np.int64)
    bounds = np.zeros(n_ranks + 1, dtype=np.int64)
    _check(_lib.ss_flatten_layout(num.ctypes.data if num.size else None, num.size, n_ranks, offs.ctypes.data,
                                  bounds.ctypes.data), "ss_flatten_layout")
    return offs, bounds


def ss_shard_segments(tensor_offsets: np.ndarray, shard_bounds: np.ndarray, shard: int):
    """[(tensor, tensor_offset, shard_offset, length), ...] of one shard."""
    offs = np.ascontiguousarray(tensor_offsets, dtype=np.int64)
    b = np.ascontiguousarray(shard_bounds, dtype=np.int64)
    cnt = ctypes.c_int32(0)
    _check(_lib.ss_shard_segments(offs.ctypes.data, offs.size - 1, b.ctypes.data, b.size - 1, shard, None, 0,
                                  ctypes.byref(cnt)), "ss_shard_segments")
    segs = (_Segment * max(cnt.value, 1))()
    _check(_lib.ss_shard_segments(offs.ctypes.data, offs.size - 1, b.ctypes.data, b.size - 1, shard,
                                  ctypes.cast(segs, ctypes.c_void_p), cnt.value, ctypes.byref(cnt)),
           "ss_shard_segments")
    return [(s.tensor, s.tensor_offset, s.shard_offset, s.length) for s in segs[:cnt.value]]


def ss_shard_of(P: int, n_ranks: int, i: int) -> int:
    return int(_lib.ss_shard_of(P, n_ranks, i))


def ss_state_bytes(P: int, n_ranks: int, n_units: int) -> dict:
    b = _Bytes()
    _check(_lib.ss_state_bytes(P, n_ranks, n_units, ctypes.byref(b)), "ss_state_bytes")
    return {f: getattr(b, f) for f in BYTES_FIELDS}


# ----------------------------------------------------------------------------- device calls

def ss_grad_reduce(rank_grads, n: int, g_out, *, gdtype: int | None = None, post_scale: float = 1.0,
                   accumulate: bool = False, nonfinite_flag=None, stream=None) -> None:
    """g_out[:n] (+)= post_scale * sum over ranks (rank order, fp32) of rank_grads[r][:n]."""
    gdtype = gdtype if gdtype is not None else _dtype_of(rank_grads[0])
    ptrs = _ptr_array(rank_grads)
    with _DeviceGuard(g_out):
        _check(_lib.ss_grad_reduce(_addr(ptrs), len(ptrs), -1 if gdtype is None else gdtype,
                                   n, float(post_scale), int(bool(accumulate)), _ptr(g_out), _ptr(nonfinite_flag),
                                   _stream(stream, g_out)), "ss_grad_reduce")


def ss_adam_step(hp: dict, n: int, master, m, v, *, g32=None, rank_grads=None, gdtype: int | None = None,
                 post_scale: float = 1.0, param16=None, pdtype: int | None = None, g_out=None,
                 nonfinite_flag=None, dev_grad_scale=None, dev_skip_flag=None, stream=None) -> None:
    """Fused (reduce +) AdamW + 16-bit cast over one shard of n elements, in place on master/m/v.

    hp: dict with lr, beta1, beta2, eps, weight_decay, step (1-based).
    """
    h = _HParams(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], 0, int(hp["step"]))
    ranks = rank_grads or []
    if g32 is None and gdtype is None and ranks:
        gdtype = _dtype_of(ranks[0])
    if param16 is not None and pdtype is None:
        pdtype = _dtype_of(param16)
    ptrs = _ptr_array(ranks) if ranks else None
    if g_out is None and nonfinite_flag is None and dev_grad_scale is None and dev_skip_flag is None:
        opts = _NO_OPTIONS  # read-only for the library
    else:
        opts = _Options(_ptr(g_out), _ptr(nonfinite_flag), _ptr(dev_grad_scale), _ptr(dev_skip_flag))
    with _DeviceGuard(master):
        _check(_lib.ss_adam_step(ctypes.byref(h), n, _ptr(g32), _addr(ptrs),
                                 len(ranks), -1 if gdtype is None else gdtype, float(post_scale), _ptr(master), _ptr(m),
                                 _ptr(v), _ptr(param16), -1 if pdtype is None else pdtype, ctypes.byref(opts),
                                 _stream(stream, master)), "ss_adam_step")


def ss_grad_sumsq_workspace(n: int) -> int:
    """Bytes of device workspace ss_grad_sumsq needs for a shard of n elements."""
    return int(_lib.ss_grad_sumsq_workspace(n))


def ss_grad_sumsq(n: int, sumsq_out, workspace, *, g32=None, rank_grads=None, gdtype: int | None = None,
                  post_scale: float = 1.0, g_out=None, nonfinite_flag=None, workspace_bytes: int | None = None,
                  stream=None) -> None:
    """sumsq_out[0] (float64) = sum of squares of the shard's reduced gradient (workspace: device scratch)."""
    ranks = rank_grads or []
    if g32 is None and gdtype is None and ranks:
        gdtype = _dtype_of(ranks[0])
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    ptrs = _ptr_array(ranks) if ranks else None
    with _DeviceGuard(sumsq_out):
        _check(_lib.ss_grad_sumsq(n, _ptr(g32), _addr(ptrs), len(ranks),
                                  -1 if gdtype is None else gdtype, float(post_scale), _ptr(sumsq_out),
                                  _ptr(workspace), int(workspace_bytes), _ptr(g_out), _ptr(nonfinite_flag),
                                  _stream(stream, sumsq_out)), "ss_grad_sumsq")


# the fixed scratch of ss_grad_sumsq_noalloc (include/ss.h): one fp64 slot per 16,384-element tile, plus two
SS_NOALLOC_SUMSQ_SLOTS = 65536
SS_NOALLOC_SUMSQ_MAX_N = (SS_NOALLOC_SUMSQ_SLOTS - 2) * 16384


def ss_grad_sumsq_noalloc(n: int, sumsq_out, *, g32=None, rank_grads=None, gdtype: int | None = None,
                          post_scale: float = 1.0, g_out=None, nonfinite_flag=None, stream=None) -> None:
    """ss_grad_sumsq without a workspace argument: for callers that cannot allocate device memory.

    The scratch lives in a fixed 512 KiB array inside the library, so n is limited to
    SS_NOALLOC_SUMSQ_MAX_N and calls that may run concurrently on the GPU must not be issued.
    """
    ranks = rank_grads or []
    if g32 is None and gdtype is None and ranks:
        gdtype = _dtype_of(ranks[0])
    ptrs = _ptr_array(ranks) if ranks else None
    with _DeviceGuard(sumsq_out):
        _check(_lib.ss_grad_sumsq_noalloc(n, _ptr(g32), _addr(ptrs),
                                          len(ranks), -1 if gdtype is None else gdtype, float(post_scale),
                                          _ptr(sumsq_out), _ptr(g_out), _ptr(nonfinite_flag),
                                          _stream(stream, sumsq_out)), "ss_grad_sumsq_noalloc")


def ss_clip_coef(shard_sumsq, n_shards: int, max_norm: float, coef_out, *, norm_out=None, stream=None) -> None:
    """coef_out[0] = min(1, max_norm / (sqrt(sum of shard_sumsq[:n_shards]) + 1e-6))."""
    with _DeviceGuard(coef_out):
        _check(_lib.ss_clip_coef(_ptr(shard_sumsq), n_shards, float(max_norm), _ptr(coef_out), _ptr(norm_out),
                                 _stream(stream, coef_out)), "ss_clip_coef")


def ss_unshard(shards, shard_bounds: np.ndarray, flat, *, dtype: int | None = None, stream=None) -> None:
    """flat[b_k : b_{k+1}] = shards[k] for every k, one launch."""
    b = np.ascontiguousarray(shard_bounds, dtype=np.int64)
    dtype = dtype if dtype is not None else _dtype_of(flat)
    ptrs = _ptr_array(shards)
    with _DeviceGuard(flat):
        _check(_lib.ss_unshard(_addr(ptrs), b.ctypes.data, len(ptrs),
                               -1 if dtype is None else dtype, _ptr(flat), _stream(stream, flat)), "ss_unshard")


def ss_reshard(flat, shard_bounds: np.ndarray, shards, *, dtype: int | None = None, stream=None) -> None:
    """shards[k] = flat[b_k : b_{k+1}] for every k, one launch."""
    b = np.ascontiguousarray(shard_bounds, dtype=np.int64)
    dtype = dtype if dtype is not None else _dtype_of(flat)
    ptrs = _ptr_array(shards)
    with _DeviceGuard(flat):
        _check(_lib.ss_reshard(_ptr(flat), b.ctypes.data, len(ptrs), -1 if dtype is None else dtype,
                               _addr(ptrs), _stream(stream, flat)), "ss_reshard")
