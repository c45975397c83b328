"""Run the CUDA step and the oracle step side by side on the same seeded inputs.

The CUDA side goes through the C ABI (mixed_precision_gb300); the oracle side
through its own ctypes wrapper. The two share only the seeded input generators
(workloads). The oracle's state evolves from its own results; nothing measured
on the GPU is ever fed back into it.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as wl
from _util import params_close, plain_param_stats, plain_state_stats, rel_err, scaled_err, ulp_diff16
from mixed_precision_gb300.engine import Hparams, ZeroStep

INF_BITS = {wl.BF16: 0x7F80, wl.F16: 0x7C00}


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def same_bits_or_both_nan(a: np.ndarray, b: np.ndarray, dtype: int) -> bool:
    if np.array_equal(a, b):
        return True
    fa, fb = oracle.decode(a, dtype), oracle.decode(b, dtype)
    diff = a != b
    return bool(np.all(np.isnan(fa[diff]) & np.isnan(fb[diff])))


class Pair:
    def __init__(self, shapes, world, stage, bucket_bytes, grad_dtype, param_dtype, comm_dtype=-1,
                 init_scale=1.0, dynamic=False, growth_interval=1000, index=9, master_sigma=0.02,
                 speculative=False):
        self.shapes = shapes
        self.numel = wl.numels(shapes)
        self.W, self.stage, self.bucket = world, stage, bucket_bytes
        self.gdt, self.pdt = grad_dtype, param_dtype
        self.cdt = grad_dtype if comm_dtype < 0 else comm_dtype
        self.index = index
        self.z = ZeroStep(shapes, world, stage, bucket_bytes, grad_dtype, param_dtype, comm_dtype)
        self.z.allocate(speculative=speculative)
        self.last_mode = None
        self.L = oracle.layout(self.numel, world, bucket_bytes, wl.ELEM_BYTES[grad_dtype])
        assert self.z.np == self.L.np_total
        # Inputs are laid out with the oracle's own offsets; the library's
        # must be the same (they are tested bit for bit on the host as well).
        self.offsets = [int(o) for o in self.L.param_offset]
        assert list(self.z.offsets) == self.offsets
        self.np = self.L.np_total
        master0 = wl.master_init(self.offsets, self.numel, self.np, master_sigma,
                                 wl.master_seed(index))
        m0 = master0.cuda() if self.np else torch.zeros(8, device="cuda")
        self.z.init(m0, init_scale=init_scale, dynamic=dynamic,
                    growth_interval=growth_interval)
        self.perm = self.L.flat_of_shard()
        self.mask_flat = self.L.real_mask().astype(bool)
        self.mask_shard = self.mask_flat[self.perm]
        self.o_master = master0.numpy()[self.perm].copy()
        self.o_m = np.zeros(self.np, np.float32)
        self.o_v = np.zeros(self.np, np.float32)
        self.o_params = oracle.encode(master0.numpy(), param_dtype)
        self.o_params[~self.mask_flat] = 0
        self.o_scaler = oracle.Scaler(scale=init_scale, dynamic=dynamic,
                                      growth_interval=growth_interval)
        # Largest magnitude each element of master/m/v has held so far (oracle values).
        self.hist = [np.abs(self.o_master), np.zeros(self.np, np.float32),
                     np.zeros(self.np, np.float32)]
        self.o_out = None
        if stage == 1:
            self.o_out = [np.zeros(self.np, oracle.storage_dtype(self.cdt)) for _ in range(world)]

    def grads(self, step: int, sigma: float, zero_params=(), inject=None):
        """Seeded flat gradients (CPU) for this step; inject = [(rank, flat_index, bits)]."""
        out = []
        for r in range(self.W):
            g = wl.flat_grads(self.offsets, self.numel, self.np, sigma,
                              wl.grad_seed(self.index, r, step), self.gdt,
                              zero_params=zero_params)
            out.append(g)
        for rank, idx, bits in (inject or []):
            out[rank].view(torch.int16)[idx] = int(np.array(bits, np.uint16).view(np.int16))
        return out

    def step(self, grads_cpu, hp: Hparams, mode: str = "flat", dev=None):
        """One step on both sides. `dev`: the GPU side's own device gradients
        (default: grads_cpu uploaded)."""
        if dev is None:
            dev = [g.cuda() if g.numel() else torch.empty(8, dtype=g.dtype, device="cuda")
                   for g in grads_cpu]
        if mode == "flat":
            self.z.step(dev, hp)
        elif mode == "tensors":
            per = []
            for r in range(self.W):
                row = []
                for p, (off, n) in enumerate(zip(self.offsets, self.numel)):
                    t = grads_cpu[r][off:off + n]
                    row.append(None if (n == 0 or not t.any()) else t.clone().cuda())
                per.append(row)
            self.z.step_tensors(per, hp)
        elif mode == "per_tensor_launch":
            self.z.step_per_tensor_launch(dev, hp)
        elif mode == "speculative":
            self.z.step_speculative(dev, hp)
        elif mode == "speculative_tensors":
            per = []
            for r in range(self.W):
                row = []
                for off, n in zip(self.offsets, self.numel):
                    t = grads_cpu[r][off:off + n]
                    row.append(None if (n == 0 or not t.any()) else t.clone().cuda())
                per.append(row)
            self.z.step_speculative_tensors(per, hp)
        elif mode == "host":
            pinned = [(g if g.numel() else torch.empty(8, dtype=g.dtype)).pin_memory()
                      for g in grads_cpu]
            self.z.step_host(pinned, dev, hp)
        else:
            raise ValueError(mode)
        self.last_mode = mode
        torch.cuda.synchronize()
        gpu_state = self.z.scaler_state()
        o_hp = oracle.Hparams(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.max_grad_norm,
                              hp.grad_divisor)
        # stage 3 has stage 2's arithmetic; only where the parameters live differs
        info = oracle.zero_step(self.numel, self.W, min(self.stage, 2), self.bucket, self.gdt, self.cdt,
                                self.pdt, [to_np(g) for g in grads_cpu], self.o_master, self.o_m,
                                self.o_v, self.o_params, o_hp, self.o_scaler,
                                allreduce_out=self.o_out)
        for h, x in zip(self.hist, (self.o_master, self.o_m, self.o_v)):
            np.maximum(h, np.abs(x), out=h)
        return gpu_state, info, grads_cpu

    def check(self, gpu_state, info, grads_cpu, rtol=1e-5):
        """Every acceptance check of one step; returns the worst relative error.

        fp32 state: |gpu - oracle| <= rtol * (largest |oracle| the element has
        held so far, this step included). Every fp32 operation's rounding error
        is relative to its operands, and fp32 state carries it from step to
        step, so near a zero crossing (an update cancelling the value it was
        computed from) the result's own magnitude is not the scale of the
        error; the magnitudes the element passed through are."""
        sc = self.o_scaler
        assert gpu_state["overflow"] == info.overflow
        assert gpu_state["skipped"] == info.skipped
        assert gpu_state["scale"] == sc.scale
        assert gpu_state["counter"] == sc.counter
        assert gpu_state["t"] == sc.t
        if np.isfinite(info.grad_norm):
            assert abs(gpu_state["grad_norm"] - info.grad_norm) <= 1e-6 * max(info.grad_norm, 1e-300)
        if not info.skipped:
            assert abs(gpu_state["clip_coef"] - info.clip_coef) <= 1e-6 * info.clip_coef
        # reduced values: bit-exact (a committed or skipped speculative step
        # never stores them in stages 2/3; its fallback does; in stage 1 the
        # single pass writes the all-reduce outputs every step)
        spec_no_reduce = (self.last_mode or "").startswith("speculative") and (
            gpu_state["fast_path"] or gpu_state["skipped"]) and self.stage != 1
        if spec_no_reduce:
            pass
        elif self.stage != 1:
            got = to_np(self.z.scratch)[:self.np]
            exp = np.zeros(self.np, oracle.storage_dtype(self.cdt))
            gn = [to_np(g) for g in grads_cpu]
            for _, _, f0, s0, ln in self.L.shard_ranges():
                exp[s0:s0 + ln] = oracle.reduce(gn, self.gdt, self.cdt, f0, f0 + ln, self.L.real_mask())
            assert same_bits_or_both_nan(got[self.mask_shard], exp[self.mask_shard], self.cdt)
        else:
            for w in range(self.W):
                got = to_np(self.z.allreduce_out[w])[:self.np]
                assert same_bits_or_both_nan(got[self.mask_flat], self.o_out[w][self.mask_flat],
                                             self.cdt)
        worst = 0.0
        cur = self.z.current_state() if hasattr(self.z, "master2") else (self.z.master, self.z.m,
                                                                        self.z.v)
        for name, gpu_t, ref, hist in zip(("master", "m", "v"), cur,
                                          (self.o_master, self.o_m, self.o_v), self.hist):
            got = to_np(gpu_t)[:self.np][self.mask_shard]
            r, h = ref[self.mask_shard], hist[self.mask_shard]
            e = scaled_err(got, r, h)
            worst = max(worst, float(e.max()) if e.size else 0.0)
            # Plain element-wise relative error holds everywhere except where the
            # element has fallen to under 10% of the largest value it held.
            plain = rel_err(got, r)
            bad = plain > rtol
            assert np.all(np.abs(r[bad]) < 0.1 * h[bad]), f"{name}: mismatch away from a cancellation"
            plain_state_stats("parity", name, got, r, rtol)
        assert worst <= rtol, worst
        p = to_np(self.z.params_flat)[:self.np]
        if self.stage == 3:  # sharded parameters: put them back in flat order
            flat = np.zeros(self.np, np.uint16)
            flat[self.perm] = p
            p = flat
        # master error bound in flat order: rtol x the largest |master| held
        bound = np.zeros(self.np)
        bound[self.perm] = rtol * self.hist[0].astype(np.float64)
        ok = params_close(p, self.o_params, oracle.decode(self.o_params, self.pdt),
                          oracle.decode(p, self.pdt), bound, self.pdt == wl.BF16)
        plain_param_stats("parity", p, self.o_params, self.mask_flat)
        bad = np.nonzero(~ok & self.mask_flat)[0]
        if len(bad):
            offs = np.array(self.offsets)
            pid = np.searchsorted(offs, bad, side="right") - 1
            raise AssertionError(
                f"{len(bad)} params beyond tolerance; first flat {bad[:6].tolist()} params "
                f"{pid[:6].tolist()} gpu {p[bad[:6]].tolist()} oracle {self.o_params[bad[:6]].tolist()}")
        return worst
