"""Seeded, counter-based synthetic inputs shared by the oracle side and the GPU side.

This module makes input data only; it holds none of the shard step's arithmetic.
The generator is defined once in ``synth_core.h`` and compiled twice: into
``libsynth_host.so`` (gcc, fills numpy arrays) and ``libsynth_dev.so`` (nvcc,
fills device buffers). Both produce identical bits for the same
(seed, stream, element index); a GPU test checks that on sampled ranges.

A stream is one logical tensor instance: (kind, virtual rank, step). The
element index is the element's position in the flat parameter vector of the
unit, so a shard is a view of the same numbers whatever the shard boundaries.
"""
from __future__ import annotations

import ctypes
import math
import os
import shutil
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libsynth_host.so")
_DEV_SO = os.path.join(_HERE, "libsynth_dev.so")

NORMAL, ABS_NORMAL, UNIFORM = 0, 1, 2
BF16, FP16, FP32 = 0, 1, 2

# stream kinds
GRAD, MASTER, MOM1, MOM2, SELECT, PARAM16, FLAT16 = 1, 2, 3, 4, 5, 6, 7


class _Spec(ctypes.Structure):
    _fields_ = [
        ("seed", ctypes.c_uint64),
        ("stream", ctypes.c_uint64),
        ("outlier_stream", ctypes.c_uint64),
        ("scale", ctypes.c_double),
        ("outlier_scale", ctypes.c_double),
        ("outlier_mod", ctypes.c_uint32),
        ("dist", ctypes.c_int32),
        ("fmt", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
    ]


def stream_id(kind: int, rank: int = 0, step: int = 0) -> int:
    """Pack (kind, rank, step) into one 64-bit stream id."""
    assert 0 <= kind < 256 and 0 <= rank < (1 << 24) and 0 <= step < (1 << 32)
    return (kind << 56) | (rank << 32) | step


@dataclass(frozen=True)
class Spec:
    """One synthetic tensor: distribution, scale, format and stream."""

    dist: int
    fmt: int
    scale: float
    seed: int = 0
    stream: int = 0
    outlier_mod: int = 0
    outlier_scale: float = 0.0
    outlier_stream: int = 0

    def c(self) -> _Spec:
        return _Spec(self.seed, self.stream, self.outlier_stream, self.scale, self.outlier_scale,
                     self.outlier_mod, self.dist, self.fmt, 0)

    @property
    def itemsize(self) -> int:
        return 4 if self.fmt == FP32 else 2


def normal(sigma: float, fmt: int, kind: int, rank: int = 0, step: int = 0, seed: int = 0,
           outlier_every: int = 0, outlier_mult: float = 1.0, absolute: bool = False) -> Spec:
    """N(0, sigma) (Irwin-Hall approximation) truncated onto `fmt`'s grid.

    With `outlier_every` = k > 0, about one element in k (chosen by an
    independent stream) is drawn with sigma * outlier_mult instead.
    """
    return Spec(ABS_NORMAL if absolute else NORMAL, fmt, math.ldexp(sigma, -22), seed,
                stream_id(kind, rank, step), outlier_every,
                math.ldexp(sigma * outlier_mult, -22) if outlier_every else 0.0,
                stream_id(SELECT, rank, step) if outlier_every else 0)


def uniform(a: float, fmt: int, kind: int, rank: int = 0, step: int = 0, seed: int = 0) -> Spec:
    """U(-a, a) truncated onto `fmt`'s grid."""
    return Spec(UNIFORM, fmt, math.ldexp(a, -53), seed, stream_id(kind, rank, step))


# ----------------------------------------------------------------------------- build

def build(verbose: bool = False) -> None:
    """Compile the host (gcc) and device (nvcc) generator libraries in place."""
    host_cmd = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fopenmp", "-std=c11",
                os.path.join(_HERE, "synth_host.c"), "-o", _HOST_SO]
    dev_cmd = [shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc", "-O3", "-shared",
               "-Xcompiler", "-fPIC", "-gencode", "arch=compute_103a,code=sm_103a", "-cudart", "shared",
               "-fmad=false", os.path.join(_HERE, "synth_dev.cu"), "-o", _DEV_SO]
    procs = [subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
             for c in (host_cmd, dev_cmd)]
    for cmd, p in zip((host_cmd, dev_cmd), procs):
        out, _ = p.communicate()
        if verbose and out:
            print(out)
        if p.returncode != 0:
            raise RuntimeError(f"synth build failed: {' '.join(cmd)}\n{out}")


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        if not os.path.exists(_HOST_SO):
            build()
        lib = ctypes.CDLL(_HOST_SO)
        lib.synth_fill_range.argtypes = [ctypes.POINTER(_Spec), ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p]
        lib.synth_fill_gather.argtypes = [ctypes.POINTER(_Spec), ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]
        lib.synth_irwin_hall_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_irwin_hall_at.restype = ctypes.c_int64
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(_DEV_SO):
            build()
        lib = ctypes.CDLL(_DEV_SO)
        lib.synth_fill_range_dev.argtypes = [ctypes.POINTER(_Spec), ctypes.c_uint64, ctypes.c_uint64,
                                             ctypes.c_void_p, ctypes.c_void_p]
        _dev = lib
    return _dev


def _np_dtype(spec: Spec):
    return np.uint32 if spec.fmt == FP32 else np.uint16


def host_range(spec: Spec, start: int, count: int) -> np.ndarray:
    """Bit patterns of elements [start, start+count) (uint16 for 16-bit formats, uint32 for fp32)."""
    out = np.empty(count, dtype=_np_dtype(spec))
    c = spec.c()
    if _host_lib().synth_fill_range(ctypes.byref(c), start, count, out.ctypes.data) != 0:
        raise RuntimeError("synth_fill_range failed")
    return out


def host_gather(spec: Spec, idx) -> np.ndarray:
    """Bit patterns of the elements at the given flat indices."""
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.uint64))
    out = np.empty(idx.size, dtype=_np_dtype(spec))
    c = spec.c()
    if _host_lib().synth_fill_gather(ctypes.byref(c), idx.ctypes.data, idx.size, out.ctypes.data) != 0:
        raise RuntimeError("synth_fill_gather failed")
    return out


def irwin_hall_at(seed: int, stream: int, i: int) -> int:
    return int(_host_lib().synth_irwin_hall_at(seed, stream, i))


def device_fill(spec: Spec, tensor, start: int = 0) -> None:
    """Fill a contiguous CUDA tensor with elements [start, start+numel) on torch's current stream."""
    import torch

    assert tensor.is_cuda and tensor.is_contiguous() and tensor.element_size() == spec.itemsize
    c = spec.c()
    stream = torch.cuda.current_stream(tensor.device).cuda_stream
    with torch.cuda.device(tensor.device):
        rc = _dev_lib().synth_fill_range_dev(ctypes.byref(c), start, tensor.numel(), tensor.data_ptr(), stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_range_dev failed ({rc})")


def as_float32(bits: np.ndarray) -> np.ndarray:
    """View fp32 bit patterns as float32 values."""
    return bits.view(np.float32)
