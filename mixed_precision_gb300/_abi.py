"""ctypes binding of the C ABI in include/zero.h, entry point for entry point.

Argument marshalling only: every function here converts Python values to the
C types, calls the entry point of the same name in libzero_gb300.so, and turns
a non-zero status into ZeroError. Device pointers and streams are plain ints
(``tensor.data_ptr()``, ``torch.cuda.current_stream().cuda_stream``).

There is no fallback: if the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzero_gb300.so")

ZERO_OK, ZERO_ERR_INVALID, ZERO_ERR_CUDA, ZERO_ERR_OOM, ZERO_ERR_TIMEOUT, ZERO_ERR_STATE = range(6)
ZERO_F32, ZERO_F16, ZERO_BF16 = 0, 1, 2
ZERO_MAX_WORLD = 64
ZERO_MAX_ELEMS = 1 << 36
ZERO_STATE_BLOB_BYTES = 256
STATUS_NAME = {0: "ZERO_OK", 1: "ZERO_ERR_INVALID", 2: "ZERO_ERR_CUDA", 3: "ZERO_ERR_OOM",
               4: "ZERO_ERR_TIMEOUT", 5: "ZERO_ERR_STATE"}


class ZeroError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS_NAME.get(code, code)}: {message}")
        self.code = code


class zero_config(ctypes.Structure):
    _fields_ = [("world", ctypes.c_int32), ("stage", ctypes.c_int32),
                ("bucket_bytes", ctypes.c_int64), ("grad_dtype", ctypes.c_int32),
                ("param_dtype", ctypes.c_int32), ("comm_dtype", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class zero_layout_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "n_params", "n_real", "n_padded", "shard_elems", "n_buckets", "n_tiles", "grad_bytes",
        "state_bytes", "params_bytes", "scratch_bytes", "allreduce_bytes", "device_bytes_owned")] + \
        [("ledger_bytes_per_param", ctypes.c_double), ("step_bytes_per_elem", ctypes.c_double),
         ("state_blob_used", ctypes.c_int64)]


class zero_scaler_cfg(ctypes.Structure):
    _fields_ = [("init_scale", ctypes.c_double), ("dynamic", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("growth_interval", ctypes.c_int64),
                ("growth_factor", ctypes.c_double), ("backoff_factor", ctypes.c_double),
                ("min_scale", ctypes.c_double)]


class zero_hparams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in (
        "lr", "beta1", "beta2", "eps", "weight_decay", "max_grad_norm", "grad_divisor")]


class zero_scaler_state(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_double), ("counter", ctypes.c_int64), ("t", ctypes.c_int64),
                ("overflow", ctypes.c_int32), ("skipped", ctypes.c_int32),
                ("grad_norm", ctypes.c_double), ("clip_coef", ctypes.c_double),
                ("norm_sq_raw", ctypes.c_double), ("steps", ctypes.c_int64),
                ("state_set", ctypes.c_int32), ("fast_path", ctypes.c_int32)]


ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p)
FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p)

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        PP = ctypes.POINTER(ctypes.c_void_p)
        sig = {
            "zero_layout_create": [ctypes.POINTER(ctypes.POINTER(ctypes.c_int64)),
                                   ctypes.POINTER(ctypes.c_int), I, ctypes.POINTER(zero_config),
                                   ctypes.POINTER(P)],
            "zero_layout_destroy": [P],
            "zero_layout_query": [P, ctypes.POINTER(zero_layout_info)],
            "zero_param_offset": [P, I, ctypes.POINTER(I64)],
            "zero_bucket_range": [P, I, ctypes.POINTER(I64), ctypes.POINTER(I64)],
            "zero_shard_range": [P, I, I, ctypes.POINTER(I64), ctypes.POINTER(I64),
                                 ctypes.POINTER(I64)],
            "zero_state_bind": [P, P, P, P, P, P],
            "zero_state_init": [P, P, ctypes.POINTER(zero_scaler_cfg), P],
            "zero_state_bind_alternate": [P, P, P, P],
            "zero_step_speculative": [P, PP, ctypes.POINTER(zero_hparams), P],
            "zero_step_speculative_allreduce": [P, PP, PP, ctypes.POINTER(zero_hparams), P],
            "zero_step_speculative_tensors": [P, PP, ctypes.POINTER(zero_hparams), P],
            "zero_step": [P, PP, PP, ctypes.POINTER(zero_hparams), P],
            "zero_step_tensors": [P, PP, PP, ctypes.POINTER(zero_hparams), P],
            "zero_step_per_tensor_launch": [P, PP, PP, ctypes.POINTER(zero_hparams), P],
            "zero_step_host": [P, PP, PP, PP, ctypes.POINTER(zero_hparams), P],
            "zero_loss_scale_state": [P, P, ctypes.POINTER(zero_scaler_state)],
            "zero_gather_params": [P, PP, I, P],
            "zero_state_export": [P, P, P, P, P],
            "zero_state_import": [P, P, P, P, P],
            "zero_layout_set_allocator": [P, ALLOC_FN, FREE_FN, P],
            "zero_set_step_events": [P, PP],
            "zero_reduce_norm_noalloc": [PP, I, I64, I, I, P, P, P, P],
            "zero_selftest_wait_timeout": [ctypes.c_uint32, P],
            "zero_selftest_layout_timeout": [P, ctypes.c_uint32, P],
            "zero_accumulate": [P, PP, I, PP, I, P],
            "zero_state_export_params": [P, P, P, P, P],
            "zero_state_import_params": [P, P, P, P, P],
            "zero_scaler_restore": [P, ctypes.POINTER(zero_scaler_state), P],
            "zero_gather_bucket": [P, I, P, P],
            "zero_loss_scale_state_async": [P, P, P],
            "zero_state_blob_decode": [P, ctypes.POINTER(zero_scaler_state)],
            "zero_dist_set_rank": [P, I],
            "zero_dist_shard_norm": [P, P, P, P],
            "zero_dist_finalize": [P, P, ctypes.POINTER(zero_hparams), P],
            "zero_dist_update": [P, P, P],
            "zero_dist_update_buckets": [P, P, I, I, P],
            "zero_dist_widen": [P, P, P, P],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.zero_last_error.argtypes = []
        L.zero_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def zero_last_error() -> str:
    return lib().zero_last_error().decode()


def _check(rc: int) -> None:
    if rc != ZERO_OK:
        raise ZeroError(rc, zero_last_error())


def _ptrs(values) -> ctypes.Array:
    return (ctypes.c_void_p * len(values))(*[int(v) if v else None for v in values])


def zero_layout_create(shapes, cfg: zero_config) -> int:
    n = len(shapes)
    dims = [(ctypes.c_int64 * max(1, len(s)))(*[int(d) for d in s]) for s in shapes]
    shape_ptrs = (ctypes.POINTER(ctypes.c_int64) * max(1, n))(
        *[ctypes.cast(d, ctypes.POINTER(ctypes.c_int64)) for d in dims])
    ndims = (ctypes.c_int * max(1, n))(*[len(s) for s in shapes])
    out = ctypes.c_void_p()
    _check(lib().zero_layout_create(shape_ptrs, ndims, n, ctypes.byref(cfg), ctypes.byref(out)))
    return out.value


def zero_layout_destroy(layout: int) -> None:
    _check(lib().zero_layout_destroy(layout))


def zero_layout_query(layout: int) -> zero_layout_info:
    info = zero_layout_info()
    _check(lib().zero_layout_query(layout, ctypes.byref(info)))
    return info


def zero_param_offset(layout: int, param: int) -> int:
    off = ctypes.c_int64()
    _check(lib().zero_param_offset(layout, param, ctypes.byref(off)))
    return off.value


def zero_bucket_range(layout: int, bucket: int):
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().zero_bucket_range(layout, bucket, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def zero_shard_range(layout: int, bucket: int, rank: int):
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().zero_shard_range(layout, bucket, rank, ctypes.byref(a), ctypes.byref(b),
                                  ctypes.byref(c)))
    return a.value, b.value, c.value


def zero_state_bind(layout: int, master: int, m: int, v: int, params_flat: int, scratch: int) -> None:
    _check(lib().zero_state_bind(layout, master, m, v, params_flat, scratch or None))


def zero_state_init(layout: int, master_init_flat: int, cfg: zero_scaler_cfg, stream: int) -> None:
    _check(lib().zero_state_init(layout, master_init_flat, ctypes.byref(cfg), stream or None))


def zero_step(layout: int, grads, allreduce_out, hp: zero_hparams, stream: int) -> None:
    ar = _ptrs(allreduce_out) if allreduce_out is not None else None
    _check(lib().zero_step(layout, _ptrs(grads), ar, ctypes.byref(hp), stream or None))


def zero_state_bind_alternate(layout: int, master2: int, m2: int, v2: int) -> None:
    _check(lib().zero_state_bind_alternate(layout, master2, m2, v2))


def zero_step_speculative(layout: int, grads, hp: zero_hparams, stream: int) -> None:
    _check(lib().zero_step_speculative(layout, _ptrs(grads), ctypes.byref(hp), stream or None))


def zero_step_speculative_allreduce(layout: int, grads, allreduce_out, hp: zero_hparams,
                                    stream: int) -> None:
    _check(lib().zero_step_speculative_allreduce(
        layout, _ptrs(grads), _ptrs(allreduce_out) if allreduce_out is not None else None,
        ctypes.byref(hp), stream or None))


def zero_step_speculative_tensors(layout: int, grad_ptrs, hp: zero_hparams, stream: int) -> None:
    _check(lib().zero_step_speculative_tensors(layout, _ptrs(grad_ptrs), ctypes.byref(hp),
                                               stream or None))


def zero_step_per_tensor_launch(layout: int, grads, allreduce_out, hp: zero_hparams,
                                stream: int) -> None:
    ar = _ptrs(allreduce_out) if allreduce_out is not None else None
    _check(lib().zero_step_per_tensor_launch(layout, _ptrs(grads), ar, ctypes.byref(hp),
                                             stream or None))


def zero_step_tensors(layout: int, grad_ptrs, allreduce_out, hp: zero_hparams, stream: int) -> None:
    ar = _ptrs(allreduce_out) if allreduce_out is not None else None
    _check(lib().zero_step_tensors(layout, _ptrs(grad_ptrs), ar, ctypes.byref(hp), stream or None))


def zero_step_host(layout: int, host_grads, dev_grads, allreduce_out, hp: zero_hparams,
                   stream: int) -> None:
    ar = _ptrs(allreduce_out) if allreduce_out is not None else None
    _check(lib().zero_step_host(layout, _ptrs(host_grads), _ptrs(dev_grads), ar, ctypes.byref(hp),
                                stream or None))


def zero_loss_scale_state(layout: int, stream: int) -> zero_scaler_state:
    st = zero_scaler_state()
    _check(lib().zero_loss_scale_state(layout, stream or None, ctypes.byref(st)))
    return st


def zero_gather_params(layout: int, dst, n_replicas: int, stream: int) -> None:
    _check(lib().zero_gather_params(layout, _ptrs(dst), n_replicas, stream or None))


def zero_state_export(layout: int, master_flat: int, m_flat: int, v_flat: int, stream: int) -> None:
    _check(lib().zero_state_export(layout, master_flat or None, m_flat or None, v_flat or None,
                                   stream or None))


def zero_state_import(layout: int, master_flat: int, m_flat: int, v_flat: int, stream: int) -> None:
    _check(lib().zero_state_import(layout, master_flat or None, m_flat or None, v_flat or None,
                                   stream or None))


def zero_set_step_events(layout: int, events) -> None:
    """events: four cudaEvent_t handles (ints), or None to turn the hook off."""
    _check(lib().zero_set_step_events(layout, _ptrs(events) if events is not None else None))


def zero_layout_set_allocator(layout: int, alloc, free_fn, ctx: int = 0) -> None:
    """alloc/free_fn: ALLOC_FN / FREE_FN instances (keep them alive), or None for the default."""
    _check(lib().zero_layout_set_allocator(layout, alloc or ALLOC_FN(), free_fn or FREE_FN(),
                                           ctx or None))


def zero_reduce_norm_noalloc(grads, n: int, grad_dtype: int, comm_dtype: int, reduced_out: int,
                             norm_sq_out: int, overflow_out: int, stream: int) -> None:
    """grads: W device pointers; outputs are device pointers (reduced_out may be 0)."""
    _check(lib().zero_reduce_norm_noalloc(_ptrs(grads), len(grads), n, grad_dtype, comm_dtype,
                                          reduced_out or None, norm_sq_out, overflow_out,
                                          stream or None))


def zero_selftest_wait_timeout(spin_limit: int, stream: int) -> None:
    _check(lib().zero_selftest_wait_timeout(spin_limit, stream or None))


def zero_selftest_layout_timeout(layout: int, spin_limit: int, stream: int) -> None:
    _check(lib().zero_selftest_layout_timeout(layout, spin_limit, stream or None))


def zero_accumulate(layout: int, micro, micro_dtype: int, main, first: bool, stream: int) -> None:
    _check(lib().zero_accumulate(layout, _ptrs(micro), micro_dtype, _ptrs(main), int(first),
                                 stream or None))


def zero_state_export_params(layout: int, master_pm: int, m_pm: int, v_pm: int, stream: int) -> None:
    _check(lib().zero_state_export_params(layout, master_pm or None, m_pm or None, v_pm or None,
                                          stream or None))


def zero_state_import_params(layout: int, master_pm: int, m_pm: int, v_pm: int, stream: int) -> None:
    _check(lib().zero_state_import_params(layout, master_pm or None, m_pm or None, v_pm or None,
                                          stream or None))


def zero_scaler_restore(layout: int, st: zero_scaler_state, stream: int) -> None:
    _check(lib().zero_scaler_restore(layout, ctypes.byref(st), stream or None))


def zero_gather_bucket(layout: int, bucket: int, dst: int, stream: int) -> None:
    _check(lib().zero_gather_bucket(layout, bucket, dst, stream or None))


def zero_loss_scale_state_async(layout: int, blob: int, stream: int) -> None:
    _check(lib().zero_loss_scale_state_async(layout, blob, stream or None))


def zero_state_blob_decode(blob: int) -> zero_scaler_state:
    st = zero_scaler_state()
    _check(lib().zero_state_blob_decode(blob, ctypes.byref(st)))
    return st


def zero_dist_set_rank(layout: int, rank: int) -> None:
    _check(lib().zero_dist_set_rank(layout, rank))


def zero_dist_shard_norm(layout: int, allreduced: int, norm_pair: int, stream: int) -> None:
    _check(lib().zero_dist_shard_norm(layout, allreduced or None, norm_pair, stream or None))


def zero_dist_finalize(layout: int, norm_pair: int, hp: zero_hparams, stream: int) -> None:
    _check(lib().zero_dist_finalize(layout, norm_pair, ctypes.byref(hp), stream or None))


def zero_dist_update(layout: int, allreduced: int, stream: int) -> None:
    _check(lib().zero_dist_update(layout, allreduced or None, stream or None))


def zero_dist_update_buckets(layout: int, allreduced: int, first_bucket: int, n_buckets: int,
                             stream: int) -> None:
    _check(lib().zero_dist_update_buckets(layout, allreduced or None, first_bucket, n_buckets,
                                          stream or None))


def zero_dist_widen(layout: int, grads: int, out: int, stream: int) -> None:
    _check(lib().zero_dist_widen(layout, grads, out, stream or None))
