"""The sharded ZeRO step: one process per GPU, each holding one rank's shard.

leetllm "Deep dive: Megatron", section "Distributed optimizer: trade
replicated state for collectives": each bucket of gradients is
reduce-scattered so that every rank receives the sum of its own slice, every
rank updates its FP32 master slice and moments, and the parameters are
all-gathered back bucket by bucket. One 16-byte all-reduce of {sum of
squares, overflow} between the two makes the norm, the clip coefficient and
the loss-scale decision global.

The collectives run through a communicator (``TorchComm``: torch.distributed,
NCCL between GPUs); everything between them runs in the library's kernels
(``zero_dist_shard_norm``, ``zero_dist_finalize``, ``zero_dist_update``,
through ``LibraryShard``). Nothing here computes a step of the method: this
module allocates buffers, slices bucket views and orders the calls.
"""
from __future__ import annotations

import dataclasses

import torch

from . import _abi as abi
from .engine import Hparams

TORCH_DTYPE = {abi.ZERO_F32: torch.float32, abi.ZERO_F16: torch.float16,
               abi.ZERO_BF16: torch.bfloat16}


class TorchComm:
    """The step's three collectives through torch.distributed (sum)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist, self.group = dist, group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def reduce_scatter(self, out: torch.Tensor, inp: torch.Tensor) -> None:
        """out (len/W) <- this rank's slice of the sum of every rank's inp (len)."""
        self.dist.reduce_scatter_tensor(out, inp, op=self.dist.ReduceOp.SUM, group=self.group)

    def all_reduce(self, t: torch.Tensor) -> None:
        self.dist.all_reduce(t, op=self.dist.ReduceOp.SUM, group=self.group)

    def all_gather(self, out: torch.Tensor, inp: torch.Tensor) -> None:
        """out (len) <- every rank's inp (len/W), in rank order."""
        self.dist.all_gather_into_tensor(out, inp, group=self.group)

    def all_gather_async(self, out: torch.Tensor, inp: torch.Tensor):
        """The same, started after the work already on the current stream and
        running beside what is enqueued next; .wait() joins it."""
        return self.dist.all_gather_into_tensor(out, inp, group=self.group, async_op=True)


@dataclasses.dataclass
class Bucket:
    start: int        # flat offset of the bucket
    length: int       # padded length (a multiple of W * 128)
    local: int        # offset of this rank's slice in the shard buffers

    def slice_len(self, world: int) -> int:
        return self.length // world


class LibraryShard:
    """This rank's device buffers, bound to its layout, and the library's
    kernels for the steps between the collectives."""

    def __init__(self, z: "ShardedZeroStep", device):
        self.z = z
        n_shard = max(z.shard_elems, 8)
        dev = torch.device(device)
        self.master = torch.empty(n_shard, dtype=torch.float32, device=dev)
        self.m = torch.empty(n_shard, dtype=torch.float32, device=dev)
        self.v = torch.empty(n_shard, dtype=torch.float32, device=dev)
        n_params = n_shard if z.stage == 3 else max(z.np, 8)
        self.params = torch.empty(n_params, dtype=TORCH_DTYPE[z.param_dtype], device=dev)
        self.scratch = (torch.empty(n_shard, dtype=TORCH_DTYPE[z.comm_dtype], device=dev)
                        if z.stage != 1 else None)
        # an fp32 collective of 16-bit gradients: this rank's widened copy
        self.comm_buf = (torch.empty(max(z.np, 8), dtype=torch.float32, device=dev)
                         if z.comm_dtype != z.grad_dtype else None)
        self.norm_pair = torch.zeros(2, dtype=torch.float64, device=dev)
        abi.zero_state_bind(z.handle, self.master.data_ptr(), self.m.data_ptr(), self.v.data_ptr(),
                            self.params.data_ptr(),
                            self.scratch.data_ptr() if self.scratch is not None else 0)

    @staticmethod
    def _stream() -> int:
        return int(torch.cuda.current_stream().cuda_stream)

    def init(self, master_init_flat: torch.Tensor, cfg: abi.zero_scaler_cfg) -> None:
        abi.zero_state_init(self.z.handle, master_init_flat.data_ptr(), cfg, self._stream())

    def to_comm(self, grads: torch.Tensor) -> torch.Tensor:
        """The buffer the collectives reduce: the gradients themselves, or
        their exact fp32 widening when the communication dtype is fp32."""
        if self.comm_buf is None:
            return grads
        abi.zero_dist_widen(self.z.handle, grads.data_ptr(), self.comm_buf.data_ptr(), self._stream())
        return self.comm_buf

    def shard_norm(self, allreduced) -> None:
        abi.zero_dist_shard_norm(self.z.handle, allreduced.data_ptr() if allreduced is not None else 0,
                                 self.norm_pair.data_ptr(), self._stream())

    def finalize(self, hp: Hparams) -> None:
        abi.zero_dist_finalize(self.z.handle, self.norm_pair.data_ptr(), hp.c(), self._stream())

    def update(self, allreduced) -> None:
        abi.zero_dist_update(self.z.handle, allreduced.data_ptr() if allreduced is not None else 0,
                             self._stream())

    def update_buckets(self, first: int, count: int, allreduced) -> None:
        abi.zero_dist_update_buckets(self.z.handle,
                                     allreduced.data_ptr() if allreduced is not None else 0,
                                     first, count, self._stream())

    def scaler_state(self) -> dict:
        st = abi.zero_loss_scale_state(self.z.handle, self._stream())
        return {f: getattr(st, f) for f, _ in abi.zero_scaler_state._fields_}

    def export_params(self, master_pm, m_pm, v_pm) -> None:
        """This rank's fp32 state into parameter-major buffers (N elements
        each); the other ranks' elements are written as zero."""
        abi.zero_state_export_params(self.z.handle, master_pm.data_ptr(), m_pm.data_ptr(),
                                     v_pm.data_ptr(), self._stream())

    def import_params(self, master_pm, m_pm, v_pm) -> None:
        """This rank's elements from whole parameter-major buffers; its
        parameter slices are recast."""
        abi.zero_state_import_params(self.z.handle, master_pm.data_ptr(), m_pm.data_ptr(),
                                     v_pm.data_ptr(), self._stream())

    def scaler_restore(self, st: dict) -> None:
        abi.zero_scaler_restore(self.z.handle, abi.zero_scaler_state(
            st["scale"], st["counter"], st["t"], 0, 0, 0.0, 0.0, 0.0, 0, 0, 0), self._stream())


class ShardedZeroStep:
    """Rank `rank` of a W-GPU data-parallel ZeRO-1/2/3 optimizer.

    The layout is the library's (zero_layout_create with world = W), made
    this rank's with zero_dist_set_rank. ``local`` builds the object that
    holds this rank's buffers and runs the local steps; by default the
    library's kernels on `device` (``LibraryShard``). ``comm`` runs the
    collectives; by default torch.distributed's default group.
    """

    def __init__(self, shapes, stage: int = 2, bucket_bytes: int = 500_000_000,
                 grad_dtype: int = abi.ZERO_BF16, param_dtype: int = abi.ZERO_BF16, comm=None,
                 local=None, device="cuda", comm_dtype: int = -1):
        self.comm = comm if comm is not None else TorchComm()
        self.rank, self.world = self.comm.rank, self.comm.world
        self.shapes = [tuple(int(d) for d in s) for s in shapes]
        self.stage, self.grad_dtype, self.param_dtype = stage, grad_dtype, param_dtype
        # the collectives' dtype: the gradients' own, or fp32 (abi.ZERO_F32)
        self.comm_dtype = grad_dtype if comm_dtype < 0 else comm_dtype
        self.bucket_bytes = int(bucket_bytes)
        cfg = abi.zero_config(self.world, stage, int(bucket_bytes), grad_dtype, param_dtype,
                              self.comm_dtype, 0)
        self.handle = abi.zero_layout_create(self.shapes, cfg)
        abi.zero_dist_set_rank(self.handle, self.rank)
        self.info = abi.zero_layout_query(self.handle)
        self.np = self.info.n_padded
        self.shard_elems = self.info.shard_elems
        self.offsets = [abi.zero_param_offset(self.handle, p) for p in range(len(self.shapes))]
        self.numels = [int(torch.Size(s).numel()) for s in self.shapes]
        self.buckets = []
        for b in range(self.info.n_buckets):
            start, length = abi.zero_bucket_range(self.handle, b)
            _, shard_off, _ = abi.zero_shard_range(self.handle, b, self.rank)
            self.buckets.append(Bucket(start, length, shard_off - self.rank * self.shard_elems))
        self.local = local(self) if local is not None else LibraryShard(self, device)

    # ---- state ------------------------------------------------------------
    def init(self, master_init_flat: torch.Tensor, init_scale: float = 1.0, dynamic: bool = False,
             growth_interval: int = 1000, growth_factor: float = 2.0, backoff_factor: float = 0.5,
             min_scale: float = 1.0) -> None:
        """This rank's slices of master <- master_init_flat (the whole flat
        buffer, Np fp32), m = v = 0, its parameters cast; then one all-gather
        gives every rank the whole parameter buffer (stages 1/2)."""
        cfg = abi.zero_scaler_cfg(init_scale, int(dynamic), 0, growth_interval, growth_factor,
                                  backoff_factor, min_scale)
        self.local.init(master_init_flat, cfg)
        self.all_gather_params()

    def scaler_state(self) -> dict:
        return self.local.scaler_state()

    # ---- the step -----------------------------------------------------------
    def step(self, grads: torch.Tensor, hp: Hparams) -> None:
        """One step from this rank's gradients (flat layout, Np elements of the
        gradient dtype). Stages 2/3: reduce-scatter bucket by bucket into this
        rank's scratch. Stage 1: all-reduce bucket by bucket, in place (on
        `grads`, which then hold the summed gradient, or on the fp32 copy
        with an fp32 communication dtype). Then this rank's
        norm share, its all-reduce, the finalize, the local update, and the
        all-gather of the parameters (stages 1/2), bucket by bucket with each
        bucket's all-gather beside the next bucket's update when the
        communicator can start one asynchronously."""
        W = self.world
        allreduced = None
        src = self.local.to_comm(grads)
        for b in self.buckets:
            g = src[b.start:b.start + b.length]
            if self.stage == 1:
                self.comm.all_reduce(g)
            else:
                n = b.slice_len(W)
                self.comm.reduce_scatter(self.local.scratch[b.local:b.local + n], g)
        if self.stage == 1:
            allreduced = src
        self.local.shard_norm(allreduced)
        self.comm.all_reduce(self.local.norm_pair)
        self.local.finalize(hp)
        gather_async = getattr(self.comm, "all_gather_async", None)
        if self.stage == 3 or gather_async is None:
            self.local.update(allreduced)
            self.all_gather_params()
            return
        # Bucket by bucket: bucket b's all-gather starts once its update is
        # done and runs while bucket b + 1 is updated.
        works = []
        for i, b in enumerate(self.buckets):
            self.local.update_buckets(i, 1, allreduced)
            n = b.slice_len(W)
            p = self.local.params
            works.append(gather_async(p[b.start:b.start + b.length],
                                      p[b.start + self.rank * n:b.start + (self.rank + 1) * n]))
        for w in works:
            w.wait()

    def all_gather_params(self) -> None:
        """Every rank's updated parameter slices into every rank's flat
        parameter buffer, bucket by bucket (in place; stage 3 keeps them
        sharded and gathers nothing)."""
        if self.stage == 3:
            return
        W, p = self.world, self.local.params
        for b in self.buckets:
            n = b.slice_len(W)
            mine = p[b.start + self.rank * n:b.start + (self.rank + 1) * n]
            self.comm.all_gather(p[b.start:b.start + b.length], mine)

    def gather_bucket(self, b: int, out: torch.Tensor) -> None:
        """Stage 3: bucket b's parameters from every rank's slice into `out`
        (its padded length, flat order) -- what a forward pass fetches
        bucket by bucket."""
        n = self.buckets[b].slice_len(self.world)
        loc = self.buckets[b].local
        self.comm.all_gather(out[:self.buckets[b].length], self.local.params[loc:loc + n])

    # ---- checkpoints independent of W -------------------------------------
    def export_params(self):
        """(master, m, v) in parameter-major order -- N fp32 elements each, the
        same for any W, stage or bucket size -- whole on every rank. Each
        rank exports its own elements (zeros elsewhere); one all-reduce per
        tensor sums their 32-bit patterns, exactly one rank contributing
        each element."""
        n = max(self.info.n_real, 1)
        dev = self.local.master.device
        out = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(3)]
        self.local.export_params(*out)
        for t in out:
            self.comm.all_reduce(t.view(torch.int32))
        return out

    def import_params(self, master_pm, m_pm, v_pm, scaler: dict | None = None) -> None:
        """This rank's elements from whole parameter-major buffers (exported by
        a job of any W, stage or bucket size), its parameters recast and
        all-gathered; `scaler` (scale, counter, t) restores the loss scaler.
        Call after init (which sets the scaler's configuration)."""
        self.local.import_params(master_pm, m_pm, v_pm)
        if scaler is not None:
            self.local.scaler_restore(scaler)
        self.all_gather_params()

    def close(self) -> None:
        if self.handle:
            abi.zero_layout_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
