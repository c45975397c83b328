"""ZeroStep: a small owner of the device buffers one layout needs.

PyTorch is used only to allocate device memory and to name streams; every
step of the path runs in the library's CUDA kernels through the C ABI
(mixed_precision_gb300._abi). The flat buffers follow the layout of
``zero_layout_create``: parameters at 64-aligned offsets, buckets padded to a
multiple of W*128 elements; master/m/v are rank-major shard buffers.
"""
from __future__ import annotations

import dataclasses

import torch

from . import _abi as abi

TORCH_DTYPE = {abi.ZERO_F32: torch.float32, abi.ZERO_F16: torch.float16,
               abi.ZERO_BF16: torch.bfloat16}


@dataclasses.dataclass
class Hparams:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    max_grad_norm: float = 1.0
    grad_divisor: float = 0.0  # <= 0: the world size

    def c(self) -> abi.zero_hparams:
        return abi.zero_hparams(**dataclasses.asdict(self))


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


class ZeroStep:
    """One simulated W-rank ZeRO-1/2 optimizer over a parameter-shape list."""

    def __init__(self, shapes, world: int, stage: int = 2, bucket_bytes: int = 500_000_000,
                 grad_dtype: int = abi.ZERO_BF16, param_dtype: int = abi.ZERO_BF16,
                 comm_dtype: int = -1, device="cuda"):
        self.shapes = [tuple(int(d) for d in s) for s in shapes]
        self.cfg = abi.zero_config(world, stage, int(bucket_bytes), grad_dtype, param_dtype,
                                   comm_dtype, 0)
        self.handle = abi.zero_layout_create(self.shapes, self.cfg)
        self.info = abi.zero_layout_query(self.handle)
        self.world, self.stage = world, stage
        self.grad_dtype, self.param_dtype = grad_dtype, param_dtype
        self.comm_dtype = grad_dtype if comm_dtype < 0 else comm_dtype
        self.np = self.info.n_padded
        self.device = torch.device(device)
        self.offsets = [abi.zero_param_offset(self.handle, p) for p in range(len(self.shapes))]
        self.numels = [int(torch.Size(s).numel()) for s in self.shapes]
        self._bound = False

    # ---- buffers ------------------------------------------------------------
    def allocate(self, speculative: bool = False) -> None:
        """Allocate master/m/v, the flat params, the stage-2 scratch or the
        stage-1 all-reduce outputs, and bind them; with `speculative`, also a
        second master/m/v set for step_speculative."""
        dev = self.device
        n = max(self.np, 8)  # an empty model still gets non-NULL buffers
        self.master = torch.empty(n, dtype=torch.float32, device=dev)
        self.m = torch.empty(n, dtype=torch.float32, device=dev)
        self.v = torch.empty(n, dtype=torch.float32, device=dev)
        self.params_flat = torch.empty(n, dtype=TORCH_DTYPE[self.param_dtype], device=dev)
        self.scratch = None
        self.allreduce_out = None
        if self.stage != 1:
            self.scratch = torch.empty(n, dtype=TORCH_DTYPE[self.comm_dtype], device=dev)
        else:
            self.allreduce_out = [torch.empty(n, dtype=TORCH_DTYPE[self.comm_dtype], device=dev)
                                  for _ in range(self.world)]
        self.bind(self.master, self.m, self.v, self.params_flat, self.scratch)
        if speculative:
            self.bind_alternate(*[torch.empty(n, dtype=torch.float32, device=dev) for _ in range(3)])

    def bind_alternate(self, master2, m2, v2) -> None:
        """Bind the second master/m/v set (before init)."""
        abi.zero_state_bind_alternate(self.handle, master2.data_ptr(), m2.data_ptr(), v2.data_ptr())
        self.master2, self.m2, self.v2 = master2, m2, v2

    def current_state(self, stream=None):
        """(master, m, v) of the state set that holds the current state."""
        if self.scaler_state(stream)["state_set"] == 1:
            return self.master2, self.m2, self.v2
        return self.master, self.m, self.v

    def bind(self, master, m, v, params_flat, scratch=None) -> None:
        abi.zero_state_bind(self.handle, master.data_ptr(), m.data_ptr(), v.data_ptr(),
                            params_flat.data_ptr(), scratch.data_ptr() if scratch is not None else 0)
        self._bound = True

    def new_grad_buffers(self):
        """W flat gradient buffers of the layout (contents undefined)."""
        return [torch.empty(max(self.np, 8), dtype=TORCH_DTYPE[self.grad_dtype], device=self.device)
                for _ in range(self.world)]

    def param_view(self, flat: torch.Tensor, p: int) -> torch.Tensor:
        off, n = self.offsets[p], self.numels[p]
        return flat[off:off + n].view(self.shapes[p])

    # ---- state --------------------------------------------------------------
    def init(self, master_init_flat: torch.Tensor, init_scale: float = 1.0, dynamic: bool = False,
             growth_interval: int = 1000, growth_factor: float = 2.0, backoff_factor: float = 0.5,
             min_scale: float = 1.0, stream=None) -> None:
        cfg = abi.zero_scaler_cfg(init_scale, int(dynamic), 0, growth_interval, growth_factor,
                                  backoff_factor, min_scale)
        abi.zero_state_init(self.handle, master_init_flat.data_ptr(), cfg, _stream_handle(stream))

    def scaler_state(self, stream=None) -> dict:
        st = abi.zero_loss_scale_state(self.handle, _stream_handle(stream))
        return {f: getattr(st, f) for f, _ in abi.zero_scaler_state._fields_}

    # ---- the step -----------------------------------------------------------
    def step(self, grads, hp: Hparams, stream=None, allreduce_out=None) -> None:
        ar = None
        if self.stage == 1:
            outs = allreduce_out if allreduce_out is not None else self.allreduce_out
            ar = [t.data_ptr() for t in outs]
        abi.zero_step(self.handle, [g.data_ptr() for g in grads], ar, hp.c(), _stream_handle(stream))

    def step_speculative(self, grads, hp: Hparams, stream=None) -> None:
        """The step as one pass when clipping stays inactive and nothing
        overflows (bit-identical to step); otherwise skip or two-pass fallback.
        Stage 1 also writes the all-reduce outputs, as step does."""
        if self.stage == 1:
            abi.zero_step_speculative_allreduce(self.handle, [g.data_ptr() for g in grads],
                                                [t.data_ptr() for t in self.allreduce_out],
                                                hp.c(), _stream_handle(stream))
        else:
            abi.zero_step_speculative(self.handle, [g.data_ptr() for g in grads], hp.c(),
                                      _stream_handle(stream))

    def step_speculative_tensors(self, grads_per_rank, hp: Hparams, stream=None) -> None:
        """step_speculative from per-tensor gradients: grads_per_rank[w][p] is
        a tensor or None (all-zero gradient, never read)."""
        ptrs = [(g.data_ptr() if g is not None else 0) for row in grads_per_rank for g in row]
        abi.zero_step_speculative_tensors(self.handle, ptrs, hp.c(), _stream_handle(stream))

    def step_per_tensor_launch(self, grads, hp: Hparams, stream=None) -> None:
        """The same step launched tensor by tensor (the hook-style baseline)."""
        ar = [t.data_ptr() for t in self.allreduce_out] if self.stage == 1 else None
        abi.zero_step_per_tensor_launch(self.handle, [g.data_ptr() for g in grads], ar, hp.c(),
                                        _stream_handle(stream))

    def step_tensors(self, grads_per_rank, hp: Hparams, stream=None) -> None:
        """grads_per_rank[w][p]: a tensor or None (all-zero gradient)."""
        ptrs = [(g.data_ptr() if g is not None else 0) for row in grads_per_rank for g in row]
        ar = [t.data_ptr() for t in self.allreduce_out] if self.stage == 1 else None
        abi.zero_step_tensors(self.handle, ptrs, ar, hp.c(), _stream_handle(stream))

    def step_host(self, host_grads, dev_grads, hp: Hparams, stream=None) -> None:
        ar = [t.data_ptr() for t in self.allreduce_out] if self.stage == 1 else None
        abi.zero_step_host(self.handle, [h.data_ptr() for h in host_grads],
                           [d.data_ptr() for d in dev_grads], ar, hp.c(), _stream_handle(stream))

    def gather(self, dst_per_replica, stream=None) -> None:
        """dst_per_replica[k][p]: tensors of the param dtype and each parameter's numel."""
        ptrs = [t.data_ptr() for row in dst_per_replica for t in row]
        abi.zero_gather_params(self.handle, ptrs, len(dst_per_replica), _stream_handle(stream))

    def export_state(self, stream=None):
        out = [torch.empty(self.np, dtype=torch.float32, device=self.device) for _ in range(3)]
        abi.zero_state_export(self.handle, *[t.data_ptr() for t in out], _stream_handle(stream))
        return out

    def import_state(self, master_flat, m_flat, v_flat, stream=None) -> None:
        abi.zero_state_import(self.handle, master_flat.data_ptr(), m_flat.data_ptr(),
                              v_flat.data_ptr(), _stream_handle(stream))

    def close(self) -> None:
        if self.handle:
            abi.zero_layout_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
