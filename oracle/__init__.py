"""CPU oracle of the shard step -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct C (``oracle.c``) loaded through ctypes. Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package; the product library never links, loads or calls it, and
the two share no code. ``build()`` compiles ``liboracle.so`` with gcc.

Every function follows the pages on fully sharded data parallel training
("FSDP: Fully Sharded Data Parallel Training at Scale" and companions); the
citations are in ``oracle.c``. Every function is pinned by a ``-m "not gpu"``
test against something other than itself (brute force, the pages' worked
numbers, closed forms, library conversions).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.environ.get("ORACLE_SO") or os.path.join(_HERE, "liboracle.so")   # override: mutation tests

BF16, FP16, FP32 = 0, 1, 2


class _Segment(ctypes.Structure):
    _fields_ = [("tensor", ctypes.c_int32), ("pad_", ctypes.c_int32), ("tensor_offset", ctypes.c_int64),
                ("shard_offset", ctypes.c_int64), ("length", ctypes.c_int64)]


_BYTES_FIELDS = ["fp32_params", "fp32_grads", "fp32_adam", "fp32_total", "mp_params16", "mp_grads16",
                 "mp_master32", "mp_adam32", "mp_total", "optimizer_state", "zero1_optimizer_per_gpu",
                 "full_shard_per_gpu", "shard_grad_op_per_gpu", "no_shard_per_gpu", "unit_gather",
                 "full_shard_peak", "full_shard_saving", "shard_grad_op_saving", "mp_full_shard_per_gpu",
                 "mp_unit_gather16"]


class _Bytes(ctypes.Structure):
    _fields_ = [(f, ctypes.c_double) for f in _BYTES_FIELDS]


class _HP(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("pad_", ctypes.c_int32),
                ("step", ctypes.c_int64)]


def build(verbose: bool = False) -> None:
    """Compile liboracle.so (gcc; OpenMP when available, else single-threaded)."""
    base = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11", "-Wall",
            os.path.join(_HERE, "oracle.c"), "-o", _SO, "-lm"]
    for extra in (["-fopenmp"], []):
        p = subprocess.run(base[:1] + extra + base[1:], capture_output=True, text=True)
        if verbose and (p.stdout or p.stderr):
            print(p.stdout, p.stderr)
        if p.returncode == 0:
            return
    raise RuntimeError(f"oracle build failed:\n{p.stderr}")


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_SO):
            build()
        L = ctypes.CDLL(_SO)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        L.ora_flatten_layout.argtypes = [vp, i32, i32, vp, vp]
        L.ora_shard_of.argtypes = [i64, i32, i64]
        L.ora_shard_of.restype = i32
        L.ora_shard_segments.argtypes = [vp, i32, vp, i32, vp, ctypes.POINTER(i32)]
        L.ora_state_bytes.argtypes = [i64, i32, i32, ctypes.POINTER(_Bytes)]
        L.ora_widen16.argtypes = [ctypes.c_uint16, i32]
        L.ora_widen16.restype = ctypes.c_float
        L.ora_round16.argtypes = [ctypes.c_float, i32]
        L.ora_round16.restype = ctypes.c_uint16
        L.ora_round16_array.argtypes = [vp, i64, i32, vp]
        L.ora_widen16_array.argtypes = [vp, i64, i32, vp]
        L.ora_grad_reduce.argtypes = [vp, i32, i32, i64, ctypes.c_float, i32, vp]
        L.ora_adamw.argtypes = [ctypes.POINTER(_HP), i64, vp, ctypes.c_float, vp, vp, vp, vp, i32]
        L.ora_unshard.argtypes = [vp, vp, i32, i32, vp]
        L.ora_reshard.argtypes = [vp, vp, i32, i32, vp]
        L.ora_sumsq.argtypes = [vp, i64]
        L.ora_sumsq.restype = ctypes.c_double
        L.ora_clip_coef.argtypes = [ctypes.c_double, ctypes.c_float]
        L.ora_clip_coef.restype = ctypes.c_float
        L.ora_all_finite.argtypes = [vp, i64]
        L.ora_all_finite.restype = i32
        L.ora_set_threads.argtypes = [i32]
        L.ora_max_threads.restype = i32
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"{what}: oracle error {rc}")


def set_threads(n: int) -> None:
    lib().ora_set_threads(n)


def max_threads() -> int:
    return int(lib().ora_max_threads())


# ---------------------------------------------------------------------- layout

def flatten_layout(numels, n_ranks: int):
    """(tensor offsets[T+1], shard bounds[N+1]) of a unit, both int64."""
    numels = np.ascontiguousarray(np.asarray(numels, dtype=np.int64))
    offsets = np.zeros(numels.size + 1, dtype=np.int64)
    bounds = np.zeros(n_ranks + 1, dtype=np.int64)
    _check(lib().ora_flatten_layout(_ptr(numels) if numels.size else None, numels.size, n_ranks,
                                    _ptr(offsets), _ptr(bounds)), "flatten_layout")
    return offsets, bounds


def shard_of(P: int, n_ranks: int, i: int) -> int:
    return int(lib().ora_shard_of(P, n_ranks, i))


def shard_segments(offsets: np.ndarray, bounds: np.ndarray, shard: int):
    """List of (tensor, tensor_offset, shard_offset, length) of one shard."""
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    bounds = np.ascontiguousarray(bounds, dtype=np.int64)
    cnt = ctypes.c_int32(0)
    _check(lib().ora_shard_segments(_ptr(offsets), offsets.size - 1, _ptr(bounds), shard, None,
                                    ctypes.byref(cnt)), "shard_segments")
    segs = (_Segment * max(cnt.value, 1))()
    _check(lib().ora_shard_segments(_ptr(offsets), offsets.size - 1, _ptr(bounds), shard,
                                    ctypes.cast(segs, ctypes.c_void_p), ctypes.byref(cnt)), "shard_segments")
    return [(s.tensor, s.tensor_offset, s.shard_offset, s.length) for s in segs[:cnt.value]]


def state_bytes(P: int, n_ranks: int, n_units: int) -> dict:
    b = _Bytes()
    _check(lib().ora_state_bytes(P, n_ranks, n_units, ctypes.byref(b)), "state_bytes")
    return {f: getattr(b, f) for f in _BYTES_FIELDS}


# --------------------------------------------------------------------- formats

def widen16(bits: np.ndarray, dtype: int) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.size, dtype=np.float32)
    _check(lib().ora_widen16_array(_ptr(bits), bits.size, dtype, _ptr(out)), "widen16")
    return out.reshape(bits.shape)


def round16(x: np.ndarray, dtype: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.size, dtype=np.uint16)
    _check(lib().ora_round16_array(_ptr(x), x.size, dtype, _ptr(out)), "round16")
    return out.reshape(x.shape)


# ---------------------------------------------------------------------- reduce

def grad_reduce(rank_bits, dtype: int, post_scale: float = 1.0, accumulate_into: np.ndarray | None = None):
    """fp32 rank-ordered sum of N 16-bit gradient arrays (bit patterns)."""
    arrs = [np.ascontiguousarray(a, dtype=np.uint16) for a in rank_bits]
    n = arrs[0].size
    assert all(a.size == n for a in arrs)
    ptrs = (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])
    if accumulate_into is not None:
        out = accumulate_into
        assert out.dtype == np.float32 and out.size == n and out.flags.c_contiguous
    else:
        out = np.empty(n, dtype=np.float32)
    _check(lib().ora_grad_reduce(ctypes.cast(ptrs, ctypes.c_void_p), len(arrs), dtype, n,
                                 float(np.float32(post_scale)), int(accumulate_into is not None), _ptr(out)),
           "grad_reduce")
    return out


# ----------------------------------------------------------------------- AdamW

def adamw(lr, beta1, beta2, eps, weight_decay, step, g, master, m, v, p16_dtype=None, grad_scale=1.0):
    """One AdamW step in place on fp32 master/m/v; returns the 16-bit params (or None)."""
    for a in (g, master, m, v):
        assert a.dtype == np.float32 and a.flags.c_contiguous and a.size == g.size
    hp = _HP(*(float(np.float32(x)) for x in (lr, beta1, beta2, eps, weight_decay)), 0, int(step))
    p16 = np.empty(g.size, dtype=np.uint16) if p16_dtype is not None else None
    _check(lib().ora_adamw(ctypes.byref(hp), g.size, _ptr(g), float(np.float32(grad_scale)), _ptr(master), _ptr(m),
                           _ptr(v), _ptr(p16) if p16 is not None else None,
                           p16_dtype if p16_dtype is not None else BF16), "adamw")
    return p16


# --------------------------------------------------------------------- unshard

def unshard(shards, bounds: np.ndarray) -> np.ndarray:
    shards = [np.ascontiguousarray(s) for s in shards]
    bounds = np.ascontiguousarray(bounds, dtype=np.int64)
    es = shards[0].dtype.itemsize
    flat = np.empty(int(bounds[-1]), dtype=shards[0].dtype)
    ptrs = (ctypes.c_void_p * len(shards))(*[_ptr(s) if s.size else _ptr(flat) for s in shards])
    _check(lib().ora_unshard(ctypes.cast(ptrs, ctypes.c_void_p), _ptr(bounds), len(shards), es, _ptr(flat)),
           "unshard")
    return flat


def reshard(flat: np.ndarray, bounds: np.ndarray):
    flat = np.ascontiguousarray(flat)
    bounds = np.ascontiguousarray(bounds, dtype=np.int64)
    n = bounds.size - 1
    shards = [np.empty(int(bounds[k + 1] - bounds[k]), dtype=flat.dtype) for k in range(n)]
    scratch = np.empty(1, dtype=flat.dtype)
    ptrs = (ctypes.c_void_p * n)(*[_ptr(s) if s.size else _ptr(scratch) for s in shards])
    _check(lib().ora_reshard(_ptr(flat), _ptr(bounds), n, flat.dtype.itemsize, ctypes.cast(ptrs, ctypes.c_void_p)),
           "reshard")
    return shards


# --------------------------------------------------------- clipping / overflow

def sumsq(g: np.ndarray) -> float:
    g = np.ascontiguousarray(g, dtype=np.float32)
    return float(lib().ora_sumsq(_ptr(g), g.size))


def clip_coef(total_sumsq: float, max_norm: float) -> float:
    return float(lib().ora_clip_coef(float(total_sumsq), float(np.float32(max_norm))))


def all_finite(g: np.ndarray) -> bool:
    g = np.ascontiguousarray(g, dtype=np.float32)
    return bool(lib().ora_all_finite(_ptr(g), g.size))
