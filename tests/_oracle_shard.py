"""This rank's local steps of the sharded ZeRO step, computed by the oracle.

A stand-in for mixed_precision_gb300.sharded.LibraryShard on CPU tensors:
the same buffers (master/m/v and scratch of this rank's shard, the parameter
buffer, the norm pair), filled by the oracle's functions instead of the
library's kernels. With it, the schedule of ShardedZeroStep (the bucket
loop and the collectives) runs under gloo on CPU and can be compared with the
oracle's own partitioned step.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TORCH_DTYPE = {oracle.F32: torch.float32, oracle.F16: torch.float16, oracle.BF16: torch.bfloat16}


def bits(t: torch.Tensor) -> np.ndarray:
    """The tensor's storage as numpy (fp32 values, or 16-bit patterns); shares memory."""
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


class OracleShard:
    def __init__(self, z):
        self.z = z
        W, r = z.world, z.rank
        n_shard = z.shard_elems
        self.master = torch.zeros(max(n_shard, 8), dtype=torch.float32)
        self.m = torch.zeros_like(self.master)
        self.v = torch.zeros_like(self.master)
        n_params = n_shard if z.stage == 3 else z.np
        self.params = torch.zeros(max(n_params, 8), dtype=TORCH_DTYPE[z.param_dtype])
        self.scratch = (torch.zeros(max(n_shard, 8), dtype=TORCH_DTYPE[z.comm_dtype])
                        if z.stage != 1 else None)
        self.norm_pair = torch.zeros(2, dtype=torch.float64)
        # flat index of every position of this rank's shard, and which are real
        L = oracle.layout(z.numels, W, z.bucket_bytes, 4 if z.grad_dtype == oracle.F32 else 2)
        assert L.np_total == z.np
        self.flat = L.flat_of_shard()[r * n_shard:(r + 1) * n_shard]
        self.real = L.real_mask()[self.flat].astype(bool)
        self.info = None
        self.scaler = None
        self.hp = None

    def init(self, master_init_flat: torch.Tensor, cfg) -> None:
        n = self.z.shard_elems
        mi = bits(master_init_flat.contiguous())
        self.master[:n] = torch.from_numpy(np.where(self.real, mi[self.flat], 0).astype(np.float32))
        self.m.zero_()
        self.v.zero_()
        self.params.zero_()
        self._cast_params()
        self.scaler = oracle.Scaler(scale=cfg.init_scale, dynamic=bool(cfg.dynamic),
                                    growth_interval=cfg.growth_interval,
                                    growth_factor=cfg.growth_factor,
                                    backoff_factor=cfg.backoff_factor, min_scale=cfg.min_scale)

    def to_comm(self, grads):
        """The buffer the collectives reduce (fp32 comm: the exact widening,
        by the oracle's own decode)."""
        if self.z.comm_dtype == self.z.grad_dtype:
            return grads
        return torch.from_numpy(oracle.decode(bits(grads.contiguous()), self.z.grad_dtype))

    def _local_reduced(self, allreduced) -> np.ndarray:
        """This rank's reduced values in shard order; padding read as zero."""
        src = bits(allreduced)[self.flat] if allreduced is not None else \
            bits(self.scratch)[:self.z.shard_elems].copy()
        src[~self.real] = 0
        return np.ascontiguousarray(src)

    def shard_norm(self, allreduced) -> None:
        r = self._local_reduced(allreduced)
        o, s = oracle.overflow_sumsq(r, self.z.comm_dtype, self.real.astype(np.uint8))
        self.norm_pair[0] = s
        self.norm_pair[1] = 1.0 if o else 0.0

    def finalize(self, hp) -> None:
        self.hp = oracle.Hparams(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay,
                                 hp.max_grad_norm, hp.grad_divisor)
        self.info = oracle.finalize(float(self.norm_pair[0]), int(self.norm_pair[1] != 0.0),
                                    self.z.world, self.hp, self.scaler)

    def update(self, allreduced) -> None:
        if self.info.skipped:
            return
        n = self.z.shard_elems
        r = self._local_reduced(allreduced)
        ms, mm, vv = (bits(t)[:n] for t in (self.master, self.m, self.v))
        oracle.adamw(r, self.z.comm_dtype, self.hp, self.info, ms, mm, vv)
        self._cast_params()

    def update_buckets(self, first: int, count: int, allreduced) -> None:
        """The update of this rank's slices of buckets [first, first + count)
        only (element-wise, so the same numbers as one whole update); only
        their parameters are recast."""
        if self.info.skipped or count == 0:
            return
        bs = self.z.buckets
        lo = bs[first].local
        hi = bs[first + count - 1].local + bs[first + count - 1].slice_len(self.z.world)
        r = self._local_reduced(allreduced)[lo:hi]
        ms, mm, vv = (bits(t)[lo:hi] for t in (self.master, self.m, self.v))
        oracle.adamw(np.ascontiguousarray(r), self.z.comm_dtype, self.hp, self.info, ms, mm, vv)
        enc = oracle.encode(bits(self.master)[lo:hi], self.z.param_dtype)
        enc[~self.real[lo:hi]] = 0
        p = bits(self.params)
        if self.z.stage == 3:
            p[lo:hi] = enc
        else:
            p[self.flat[lo:hi]] = enc

    def _cast_params(self) -> None:
        n = self.z.shard_elems
        enc = oracle.encode(bits(self.master)[:n], self.z.param_dtype)
        enc[~self.real] = 0
        p = bits(self.params)
        if self.z.stage == 3:
            p[:n] = enc
        else:
            p[self.flat] = enc

    def _pm_index(self):
        """Parameter-major index of every real element of this rank's shard."""
        if not hasattr(self, "_pm"):
            offs = np.asarray(self.z.offsets, np.int64)
            nums = np.asarray(self.z.numels, np.int64)
            starts = np.concatenate([[0], np.cumsum(nums)[:-1]])
            f = self.flat[self.real]
            p = np.searchsorted(offs, f, side="right") - 1
            self._pm = starts[p] + (f - offs[p])
        return self._pm

    def export_params(self, master_pm, m_pm, v_pm) -> None:
        n = self.z.shard_elems
        for src, dst in zip((self.master, self.m, self.v), (master_pm, m_pm, v_pm)):
            d = bits(dst)
            d[:] = 0
            d[self._pm_index()] = bits(src)[:n][self.real]

    def import_params(self, master_pm, m_pm, v_pm) -> None:
        n = self.z.shard_elems
        for dst, src in zip((self.master, self.m, self.v), (master_pm, m_pm, v_pm)):
            d = bits(dst)[:n]
            d[self.real] = bits(src)[self._pm_index()]
        self._cast_params()

    def scaler_restore(self, st: dict) -> None:
        self.scaler.scale, self.scaler.counter, self.scaler.t = st["scale"], st["counter"], st["t"]

    def scaler_state(self) -> dict:
        info = self.info
        return {"scale": self.scaler.scale, "counter": self.scaler.counter, "t": self.scaler.t,
                "overflow": info.overflow if info else 0, "skipped": info.skipped if info else 0}
