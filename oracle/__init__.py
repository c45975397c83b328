"""ctypes wrapper around the host oracle of the ZeRO-1/2 step (zero_oracle.cpp).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package. The CUDA product path never
imports it, and it never imports the product.

Low-precision arrays are passed as ``numpy.uint16`` bit patterns; fp32 arrays
as ``numpy.float32``. Parity is unpinned for nothing here: every function has a
pin in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess

import numpy as np

F32, F16, BF16 = 0, 1, 2
_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboracle_zero.so")
SRC_PATH = os.path.join(_HERE, "zero_oracle.cpp")


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (host code only, no fused multiply-adds)."""
    stale = (not os.path.exists(LIB_PATH)
             or os.path.getmtime(LIB_PATH) < max(os.path.getmtime(SRC_PATH),
                                                 os.path.getmtime(os.path.join(_HERE, "zero_oracle.h"))))
    if force or stale:
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
               "-o", LIB_PATH, SRC_PATH]
        subprocess.run(cmd, check=True)
    return LIB_PATH


class _Hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double),
                ("max_grad_norm", ctypes.c_double), ("grad_divisor", ctypes.c_double)]


class _Scaler(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_double), ("counter", ctypes.c_int64), ("t", ctypes.c_int64),
                ("dynamic", ctypes.c_int32), ("_pad", ctypes.c_int32),
                ("growth_interval", ctypes.c_int64), ("growth_factor", ctypes.c_double),
                ("backoff_factor", ctypes.c_double), ("min_scale", ctypes.c_double)]


class _Info(ctypes.Structure):
    _fields_ = [("overflow", ctypes.c_int32), ("skipped", ctypes.c_int32),
                ("norm_sq_raw", ctypes.c_double), ("grad_norm", ctypes.c_double),
                ("clip_coef", ctypes.c_double), ("gscale", ctypes.c_double),
                ("bc1", ctypes.c_double), ("bc2", ctypes.c_double)]


@dataclasses.dataclass
class Hparams:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    max_grad_norm: float = 1.0
    grad_divisor: float = 0.0  # <= 0: the world size

    def _c(self) -> _Hparams:
        return _Hparams(**dataclasses.asdict(self))


@dataclasses.dataclass
class Scaler:
    scale: float = 1.0
    counter: int = 0
    t: int = 0
    dynamic: bool = False
    growth_interval: int = 1000
    growth_factor: float = 2.0
    backoff_factor: float = 0.5
    min_scale: float = 1.0

    def _c(self) -> _Scaler:
        return _Scaler(self.scale, self.counter, self.t, int(self.dynamic), 0,
                       self.growth_interval, self.growth_factor, self.backoff_factor,
                       self.min_scale)

    def _update(self, c: _Scaler) -> None:
        self.scale, self.counter, self.t = c.scale, c.counter, c.t


@dataclasses.dataclass
class Info:
    overflow: int
    skipped: int
    norm_sq_raw: float
    grad_norm: float
    clip_coef: float
    gscale: float
    bc1: float
    bc2: float


def _info(c: _Info) -> Info:
    return Info(c.overflow, c.skipped, c.norm_sq_raw, c.grad_norm, c.clip_coef, c.gscale,
                c.bc1, c.bc2)


_lib = None


def _open(path: str) -> ctypes.CDLL:
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64, I32, D = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    L.orc_layout.argtypes = [P, I32, I32, I64, I32, P, P, P, P, P, P]
    L.orc_encode.argtypes = [P, I64, I32, P]
    L.orc_decode.argtypes = [P, I64, I32, P]
    L.orc_reduce.argtypes = [P, I32, I32, I64, I64, P, I32, P]
    L.orc_overflow_sumsq.argtypes = [P, I32, I64, P, P, P]
    L.orc_finalize.argtypes = [D, I32, I32, P, P, P]
    L.orc_adamw.argtypes = [P, I32, I64, P, P, P, P, P]
    L.orc_accumulate.argtypes = [P, I32, P, I64, P, I32]
    L.orc_ddp_step.argtypes = [I32, I64, I32, I32, I32, P, P, P, P, P, P, P, P]
    L.orc_ddp_step.restype = I32
    L.orc_zero_step.argtypes = [P, I32, I32, I32, I64, I32, I32, I32, P, P, P, P, P, P,
                                P, P, P]
    L.orc_zero_step.restype = I32
    L.orc_layout.restype = I32
    return L


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        _lib = _open(LIB_PATH)
    return _lib


def build_variant(src: str, out: str) -> str:
    """Compile another source of the oracle (the planted-mistake variants of
    the mutation tests) with the same flags."""
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
           "-I", _HERE, "-o", out, src]
    subprocess.run(cmd, check=True, capture_output=True)
    return out


def use_library(path: str | None):
    """Route every call through the build at `path` (None: the oracle's own
    build). Returns the library used before, for restoring. A test hook: the
    mutation tests plant one mistake at a time this way."""
    global _lib
    before = _lib
    _lib = _open(path) if path is not None else None
    return before


def restore_library(before) -> None:
    global _lib
    _lib = before


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _ptr_array(arrays) -> ctypes.Array:
    return (ctypes.c_void_p * len(arrays))(*[_ptr(a) for a in arrays])


def storage_dtype(dtype: int):
    return np.float32 if dtype == F32 else np.uint16


# ---------------------------------------------------------------------------
# Layout
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Layout:
    numel: np.ndarray          # int64 [P]
    world: int
    param_offset: np.ndarray   # int64 [P]
    param_bucket: np.ndarray   # int32 [P]
    bucket_start: np.ndarray   # int64 [B]
    bucket_len: np.ndarray     # int64 [B]
    np_total: int

    @property
    def shard_total(self) -> int:
        return self.np_total // self.world

    def real_mask(self) -> np.ndarray:
        mask = np.zeros(self.np_total, dtype=np.uint8)
        for off, n in zip(self.param_offset, self.numel):
            mask[off:off + n] = 1
        return mask

    def shard_ranges(self):
        """Yield (bucket, rank, flat_begin, shard_offset, length) in rank-major order."""
        for r in range(self.world):
            at = r * self.shard_total
            for b, (b0, bl) in enumerate(zip(self.bucket_start, self.bucket_len)):
                sl = int(bl) // self.world
                yield b, r, int(b0) + r * sl, at, sl
                at += sl

    def flat_of_shard(self) -> np.ndarray:
        """flat index of every rank-major shard position (int64 [np_total])."""
        out = np.empty(self.np_total, dtype=np.int64)
        for _, _, f0, s0, ln in self.shard_ranges():
            out[s0:s0 + ln] = np.arange(f0, f0 + ln, dtype=np.int64)
        return out


def layout(numel, world: int, bucket_bytes: int, grad_bytes: int) -> Layout:
    numel = np.ascontiguousarray(np.asarray(numel, dtype=np.int64))
    n = len(numel)
    poff = np.zeros(n, dtype=np.int64)
    pb = np.zeros(n, dtype=np.int32)
    bs = np.zeros(n + 1, dtype=np.int64)
    bl = np.zeros(n + 1, dtype=np.int64)
    nb = ctypes.c_int(0)
    npt = ctypes.c_int64(0)
    rc = lib().orc_layout(_ptr(numel), n, world, bucket_bytes, grad_bytes, _ptr(poff), _ptr(pb),
                          _ptr(bs), _ptr(bl), ctypes.byref(nb), ctypes.byref(npt))
    if rc != 0:
        raise ValueError("invalid layout arguments")
    return Layout(numel, world, poff, pb, bs[:nb.value].copy(), bl[:nb.value].copy(), npt.value)


# ---------------------------------------------------------------------------
# Conversions and individual steps
# ---------------------------------------------------------------------------

def encode(x: np.ndarray, dtype: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=storage_dtype(dtype))
    lib().orc_encode(_ptr(x), x.size, dtype, _ptr(out))
    return out


def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=storage_dtype(dtype))
    out = np.empty(bits.shape, dtype=np.float32)
    lib().orc_decode(_ptr(bits), bits.size, dtype, _ptr(out))
    return out


def reduce(grads, grad_dtype: int, comm_dtype: int, begin: int = 0, end: int | None = None,
           real_mask: np.ndarray | None = None) -> np.ndarray:
    grads = [np.ascontiguousarray(g) for g in grads]
    if end is None:
        end = grads[0].size
    out = np.empty(end - begin, dtype=storage_dtype(comm_dtype))
    mask_p = _ptr(real_mask) if real_mask is not None else None
    lib().orc_reduce(_ptr_array(grads), len(grads), grad_dtype, begin, end, mask_p, comm_dtype,
                     _ptr(out))
    return out


def overflow_sumsq(reduced: np.ndarray, comm_dtype: int, real_mask: np.ndarray | None = None):
    reduced = np.ascontiguousarray(reduced)
    ovf = ctypes.c_int32(0)
    s = ctypes.c_double(0)
    lib().orc_overflow_sumsq(_ptr(reduced), comm_dtype, reduced.size,
                             _ptr(real_mask) if real_mask is not None else None,
                             ctypes.byref(ovf), ctypes.byref(s))
    return int(ovf.value), float(s.value)


def finalize(norm_sq_raw: float, overflow: int, world: int, hp: Hparams, scaler: Scaler) -> Info:
    c_hp, c_sc, c_info = hp._c(), scaler._c(), _Info()
    lib().orc_finalize(norm_sq_raw, overflow, world, ctypes.byref(c_hp), ctypes.byref(c_sc),
                       ctypes.byref(c_info))
    scaler._update(c_sc)
    return _info(c_info)


def adamw(reduced: np.ndarray, comm_dtype: int, hp: Hparams, info: Info, master: np.ndarray,
          m: np.ndarray, v: np.ndarray) -> None:
    """In-place update of fp32 master/m/v from reduced (communication-dtype) values."""
    reduced = np.ascontiguousarray(reduced)
    c_info = _Info(info.overflow, info.skipped, info.norm_sq_raw, info.grad_norm, info.clip_coef,
                   info.gscale, info.bc1, info.bc2)
    c_hp = hp._c()
    lib().orc_adamw(_ptr(reduced), comm_dtype, reduced.size, ctypes.byref(c_hp),
                    ctypes.byref(c_info), _ptr(master), _ptr(m), _ptr(v))


def accumulate(micro: np.ndarray, micro_dtype: int, main: np.ndarray, first: bool,
               real_mask: np.ndarray | None = None) -> None:
    """In place: main = (first ? 0 : main) + fp32(micro) over real elements."""
    micro = np.ascontiguousarray(micro)
    lib().orc_accumulate(_ptr(micro), micro_dtype, _ptr(main), main.size,
                         _ptr(real_mask) if real_mask is not None else None, int(first))


# ---------------------------------------------------------------------------
# Composed steps
# ---------------------------------------------------------------------------

def ddp_step(grads, grad_dtype: int, comm_dtype: int, param_dtype: int, master, m, v, params,
             hp: Hparams, scaler: Scaler) -> Info:
    """Unpartitioned step; grads are W arrays of N elements (parameters concatenated)."""
    c_hp, c_sc, c_info = hp._c(), scaler._c(), _Info()
    rc = lib().orc_ddp_step(len(grads), master.size, grad_dtype, comm_dtype, param_dtype,
                            _ptr_array(grads), _ptr(master), _ptr(m), _ptr(v), _ptr(params),
                            ctypes.byref(c_hp), ctypes.byref(c_sc), ctypes.byref(c_info))
    if rc != 0:
        raise ValueError("oracle ddp step rejected its arguments")
    scaler._update(c_sc)
    return _info(c_info)


def zero_step(numel, world: int, stage: int, bucket_bytes: int, grad_dtype: int, comm_dtype: int,
              param_dtype: int, grads, master_shards, m_shards, v_shards, params_flat,
              hp: Hparams, scaler: Scaler, allreduce_out=None) -> Info:
    """Partitioned step; grads are W flat-layout arrays; state arrays are rank-major."""
    numel = np.ascontiguousarray(np.asarray(numel, dtype=np.int64))
    c_hp, c_sc, c_info = hp._c(), scaler._c(), _Info()
    ar = _ptr_array(allreduce_out) if allreduce_out is not None else None
    rc = lib().orc_zero_step(_ptr(numel), len(numel), world, stage, bucket_bytes, grad_dtype,
                             comm_dtype, param_dtype, _ptr_array(grads), ar, _ptr(master_shards),
                             _ptr(m_shards), _ptr(v_shards), _ptr(params_flat),
                             ctypes.byref(c_hp), ctypes.byref(c_sc), ctypes.byref(c_info))
    if rc != 0:
        raise ValueError("oracle zero step rejected its arguments")
    scaler._update(c_sc)
    return _info(c_info)
