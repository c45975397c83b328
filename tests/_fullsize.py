"""Full-size parity on sampled outputs.

At the workloads' full sizes the oracle cannot run a whole step in the test's
time, but it can run the parts that decide everything globally (the reduce,
overflow flag and squared norm over every element, bucket by bucket) and then
the element-wise update for a sample of elements, one by one. The oracle's
state at the sampled elements evolves from its own results across steps.
"""
from __future__ import annotations

import concurrent.futures
import math
import os

import numpy as np
import torch

import oracle
import workloads as wl
from _parity import to_np
from _util import params_close, plain_param_stats, plain_state_stats, rel_err, scaled_err
from mixed_precision_gb300 import _abi as abi


def shard_position(z, flat_idx: np.ndarray) -> np.ndarray:
    """Rank-major shard offset of each flat index, from the library's shard ranges."""
    starts, lens = [], []
    for b in range(z.info.n_buckets):
        s, ln = abi.zero_bucket_range(z.handle, b)
        starts.append(s)
        lens.append(ln)
    starts, lens = np.array(starts), np.array(lens)
    b = np.searchsorted(starts, flat_idx, side="right") - 1
    out = np.empty_like(flat_idx)
    for bi in np.unique(b):
        sel = b == bi
        sl = lens[bi] // z.world
        r = (flat_idx[sel] - starts[bi]) // sl
        base = np.array([abi.zero_shard_range(z.handle, int(bi), int(rr))[1] for rr in range(z.world)])
        out[sel] = base[r] + (flat_idx[sel] - starts[bi] - r * sl)
    return out


def sample_indices(z, numel, n_random: int, seed: int) -> np.ndarray:
    """Random real flat indices plus the first and last real element of every
    (bucket, rank) slice and of every parameter."""
    rng = np.random.default_rng(seed)
    offs = np.array(z.offsets, np.int64)
    nums = np.array(numel, np.int64)
    live = nums > 0
    cum = np.cumsum(nums[live])
    pick = rng.integers(0, int(cum[-1]), size=n_random)
    p = np.searchsorted(cum, pick, side="right")
    before = np.concatenate([[0], cum[:-1]])
    idx = [offs[live][p] + (pick - before[p])]
    idx.append(offs[live])
    idx.append(offs[live] + nums[live] - 1)
    for b in range(z.info.n_buckets):
        for r in range(z.world):
            f0, _, ln = abi.zero_shard_range(z.handle, b, r)
            # real elements at the slice edges: first param start >= f0 ...
            inside = (offs < f0 + ln) & (offs + nums > f0) & live
            for q in np.nonzero(inside)[0]:
                a, e = max(f0, offs[q]), min(f0 + ln, offs[q] + nums[q])
                idx.append(np.array([a, e - 1]))
    return np.unique(np.concatenate(idx))


class SampledOracle:
    """Oracle state at sampled flat indices, stepped with global scalars from
    a full bucket-by-bucket reduce."""

    def __init__(self, z, numel, master0_gpu: torch.Tensor, idx: np.ndarray, init_scale, dynamic,
                 growth_interval):
        self.z, self.numel, self.idx = z, numel, idx
        self.shard = shard_position(z, idx)
        idx_t = torch.from_numpy(idx).to(master0_gpu.device)
        self.master = master0_gpu[idx_t].cpu().numpy().copy()
        self.m = np.zeros_like(self.master)
        self.v = np.zeros_like(self.master)
        self.hist = [np.abs(self.master), np.zeros_like(self.master), np.zeros_like(self.master)]
        self.scaler = oracle.Scaler(scale=init_scale, dynamic=dynamic,
                                    growth_interval=growth_interval)
        L = oracle.layout(numel, z.world, z.cfg.bucket_bytes, wl.ELEM_BYTES[z.grad_dtype])
        assert L.np_total == z.np
        # the tests lay their inputs out at the library's offsets: the oracle's own
        # layout must agree (it is also checked bit for bit on the host)
        assert list(z.offsets) == [int(o) for o in L.param_offset]
        self.L = L

    def global_reduce(self, grads_gpu):
        """Overflow flag and sum of squares over every real element (bucket by
        bucket, slices copied to the host), and the reduced values at the samples."""
        cdt, gdt = self.z.comm_dtype, self.z.grad_dtype
        ovf, sumsq = 0, 0.0
        red_at = np.zeros(len(self.idx), oracle.storage_dtype(cdt))
        for b in range(len(self.L.bucket_start)):
            b0, bl = int(self.L.bucket_start[b]), int(self.L.bucket_len[b])
            mask = np.zeros(bl, np.uint8)
            for off, n in zip(self.L.param_offset, self.numel):
                a, e = max(int(off), b0), min(int(off) + int(n), b0 + bl)
                if a < e:
                    mask[a - b0:e - b0] = 1
            host = [to_np(g[b0:b0 + bl]) for g in grads_gpu]
            # the plain oracle on disjoint chunks, in parallel host threads
            # (ctypes releases the GIL during each call); combined in chunk order
            n_chunks = max(1, min(32, bl // (1 << 20)))
            edges = [bl * k // n_chunks for k in range(n_chunks + 1)]

            def part(k):
                a, e = edges[k], edges[k + 1]
                r = oracle.reduce(host, gdt, cdt, a, e, mask)
                o, s = oracle.overflow_sumsq(r, cdt, mask[a:e])
                return r, o, s

            with concurrent.futures.ThreadPoolExecutor(min(16, os.cpu_count() or 4)) as ex:
                parts = list(ex.map(part, range(n_chunks)))
            red = np.concatenate([r for r, _, _ in parts])
            for _, o, s in parts:
                ovf |= o
                sumsq += s
            sel = (self.idx >= b0) & (self.idx < b0 + bl)
            red_at[sel] = red[self.idx[sel] - b0]
        return ovf, sumsq, red_at

    def step(self, grads_gpu, hp):
        ovf, sumsq, red_at = self.global_reduce(grads_gpu)
        self.last_reduce = (ovf, sumsq, red_at)
        return self._apply(ovf, sumsq, red_at, hp)

    def step_repeat(self, hp, ovf=None, sumsq=None):
        """A step on the same gradients as the last `step` (its global reduce
        reused), optionally with another overflow flag and sum of squares: an
        injected non-finite value changes those and, on a skipped step,
        nothing else."""
        o, sq, red_at = self.last_reduce
        return self._apply(o if ovf is None else ovf, sq if sumsq is None else sumsq, red_at, hp)

    def _apply(self, ovf, sumsq, red_at, hp):
        o_hp = oracle.Hparams(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.max_grad_norm,
                              hp.grad_divisor)
        info = oracle.finalize(sumsq, ovf, self.z.world, o_hp, self.scaler)
        oracle.adamw(red_at, self.z.comm_dtype, o_hp, info, self.master, self.m, self.v)
        for h, x in zip(self.hist, (self.master, self.m, self.v)):
            np.maximum(h, np.abs(x), out=h)
        return info, red_at

    def check(self, gpu_state, info, red_at, rtol=1e-5, reduced=True):
        """`reduced`: also compare the stored reduced gradients (a committed or
        skipped speculative step stores none)."""
        z, sc = self.z, self.scaler
        assert gpu_state["overflow"] == info.overflow and gpu_state["skipped"] == info.skipped
        assert gpu_state["scale"] == sc.scale and gpu_state["counter"] == sc.counter
        assert gpu_state["t"] == sc.t
        if math.isfinite(info.grad_norm):
            assert abs(gpu_state["grad_norm"] - info.grad_norm) <= 1e-6 * info.grad_norm
        dev = z.master.device
        sh = torch.from_numpy(self.shard).to(dev)
        fl = torch.from_numpy(self.idx).to(dev)
        if not reduced:
            pass
        elif z.stage == 2:
            assert np.array_equal(to_np(z.scratch[sh]), red_at)
        else:
            for out in z.allreduce_out:
                assert np.array_equal(to_np(out[fl]), red_at)
        worst = 0.0
        cur = z.current_state() if hasattr(z, "master2") else (z.master, z.m, z.v)
        for name, t, ref, h in zip(("master", "m", "v"), cur, (self.master, self.m, self.v),
                                   self.hist):
            got = t[sh].cpu().numpy()
            e = scaled_err(got, ref, h)
            worst = max(worst, float(e.max()))
            bad = rel_err(got, ref) > rtol
            assert np.all(np.abs(ref[bad]) < 0.1 * h[bad])
            plain_state_stats("fullsize", name, got, ref, rtol)
        assert worst <= rtol, worst
        p = to_np(z.params_flat[fl])
        exp = oracle.encode(self.master, z.param_dtype)
        plain_param_stats("fullsize", p, exp)
        ok = params_close(p, exp, oracle.decode(exp, z.param_dtype), oracle.decode(p, z.param_dtype),
                          rtol * self.hist[0].astype(np.float64), z.param_dtype == wl.BF16)
        assert ok.all(), int((~ok).sum())
        return worst
