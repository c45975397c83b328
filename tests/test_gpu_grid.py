"""The grid size of the streaming kernels does not change the step.

Every streaming kernel walks its tiles grid-stride, and the grid is a tuning
choice read at bind (ZERO_*_GRID_MULT). Two layouts bound with different
grids step on the same gradients: the reduced gradients, the overflow flag,
the loss scale, master/m/v and the parameters must be bit-identical, because
each element's arithmetic does not depend on which block runs it. Only the
norm is grouped differently: each warp's compensated fp32 running sum and
each block's partial cover other elements, so the norms agree to the norm's
tolerance (1e-6 relative, as against the oracle), not bit for bit. Clipping
is kept inactive (a threshold far above the norm): the clip coefficient is
then exactly 1 on both sides, whatever the last bits of the norm.
"""
import pytest
import torch

import workloads as wl
from mixed_precision_gb300 import _abi as abi
from mixed_precision_gb300.engine import Hparams, ZeroStep

pytestmark = pytest.mark.gpu

KNOBS = ("ZERO_REDUCE_GRID_MULT", "ZERO_UPDATE_GRID_MULT", "ZERO_SPEC_GRID_MULT",
         "ZERO_COPY_GRID_MULT")
KEYS = ("scale", "counter", "t", "overflow", "skipped", "clip_coef", "steps")


def _shapes():
    # about 12.6M elements: some 1500 tiles, more than one grid of resident
    # blocks and fewer than 64 grids' worth
    return [(1024, 1024)] * 12 + [(1000,), (3000, 7), (129, 257)]


def _layout(monkeypatch, mult, W, gdt, spec, stage=2):
    for k in KNOBS:
        monkeypatch.setenv(k, str(mult))
    z = ZeroStep(_shapes(), W, stage, 8_000_000, gdt, gdt)
    z.allocate(speculative=spec)
    master0 = wl.master_init(z.offsets, z.numels, z.np, 0.02, wl.master_seed(91), device="cuda")
    z.init(master0, init_scale=2.0 ** 12, dynamic=True, growth_interval=1000)
    return z


def _real_shard_mask(z):
    mask = torch.zeros(max(z.np, 8), dtype=torch.bool, device="cuda")
    for b in range(z.info.n_buckets):
        for r in range(z.world):
            f0, s0, ln = abi.zero_shard_range(z.handle, b, r)
            for off, n in zip(z.offsets, z.numels):
                lo, hi = max(off, f0), min(off + n, f0 + ln)
                if lo < hi:
                    mask[s0 + lo - f0:s0 + hi - f0] = True
    return mask


@pytest.mark.parametrize("spec,W,gdt,stage", [(False, 2, wl.BF16, 2), (False, 8, wl.F16, 2),
                                              (True, 2, wl.BF16, 2), (True, 4, wl.F16, 2),
                                              (False, 4, wl.BF16, 1), (True, 8, wl.F16, 1)])
def test_grid_size_does_not_change_the_step(monkeypatch, spec, W, gdt, stage):
    small = _layout(monkeypatch, 1, W, gdt, spec, stage)
    large = _layout(monkeypatch, 64, W, gdt, spec, stage)
    mask = _real_shard_mask(small)
    rank, idx = wl.inject_position(small.numels, small.offsets, W, seed=17)
    hp = Hparams(max_grad_norm=1e9)
    for step, kind in enumerate(["clean", "clean", "inf", "clean"]):
        g = [wl.flat_grads(small.offsets, small.numels, small.np, 1e-3, wl.grad_seed(900, r, step), gdt,
                           device="cuda") for r in range(W)]
        if kind == "inf":
            g[rank][idx] = float("inf")
        for z in (small, large):
            if spec:
                z.step_speculative(g, hp)
            else:
                z.step(g, hp)
        torch.cuda.synchronize()
        sa, sb = small.scaler_state(), large.scaler_state()
        for k in KEYS:
            assert sa[k] == sb[k], (step, k, sa, sb)
        assert sa["skipped"] == (1 if kind == "inf" else 0)
        if kind != "inf":
            assert sa["clip_coef"] == 1.0
            assert abs(sa["grad_norm"] - sb["grad_norm"]) <= 1e-6 * sb["grad_norm"]
            if spec:
                assert sa["fast_path"] == sb["fast_path"]
        if stage == 1:
            # every rank's all-reduce output (written by the single pass too)
            flat = torch.zeros(max(small.np, 8), dtype=torch.bool, device="cuda")
            for off, n in zip(small.offsets, small.numels):
                flat[off:off + n] = True
            for x, y in zip(small.allreduce_out, large.allreduce_out):
                assert torch.equal(x.view(torch.int16)[flat], y.view(torch.int16)[flat])
        elif not spec:
            # the reduced gradients, rank-major like the state
            assert torch.equal(small.scratch[mask].view(torch.int16), large.scratch[mask].view(torch.int16))
        for x, y in zip(small.current_state(), large.current_state()):
            assert torch.equal(x[mask].view(torch.int32), y[mask].view(torch.int32)), step
        assert torch.equal(small.params_flat.view(torch.int16), large.params_flat.view(torch.int16))
    small.close()
    large.close()


@pytest.mark.parametrize("W,gdt", [(2, wl.BF16), (8, wl.F16)])
def test_update_tile_schedules_agree(monkeypatch, W, gdt):
    """The update kernel's two tile schedules -- one block per tile, and a
    device counter handing tiles to a grid of the resident blocks -- write
    bit-identical state and parameters over clean, clipped and skipped steps.
    The counter wraps back to 0 after every launch: were it left anywhere
    else, the next step's update would skip tiles and the states would part."""
    def layout(sched):
        monkeypatch.setenv("ZERO_UPDATE_SCHED", sched)
        z = ZeroStep(_shapes(), W, 2, 8_000_000, gdt, gdt)
        z.allocate()
        master0 = wl.master_init(z.offsets, z.numels, z.np, 0.02, wl.master_seed(92), device="cuda")
        z.init(master0, init_scale=2.0 ** 12, dynamic=True, growth_interval=1000)
        return z

    per_tile, counter = layout("static"), layout("dynamic")
    mask = _real_shard_mask(per_tile)
    rank, idx = wl.inject_position(per_tile.numels, per_tile.offsets, W, seed=18)
    for step, kind in enumerate(["clean", "clip", "inf", "clean", "clip", "clean"]):
        g = [wl.flat_grads(per_tile.offsets, per_tile.numels, per_tile.np, 1e-3,
                           wl.grad_seed(901, r, step), gdt, device="cuda") for r in range(W)]
        if kind == "inf":
            g[rank][idx] = float("inf")
        hp = Hparams(max_grad_norm=1e-5 if kind == "clip" else 1e9)
        for z in (per_tile, counter):
            z.step(g, hp)
        torch.cuda.synchronize()
        sa, sb = per_tile.scaler_state(), counter.scaler_state()
        for k in KEYS + ("grad_norm",):
            assert sa[k] == sb[k], (step, k)
        assert (sa["clip_coef"] < 1.0) == (kind == "clip") or kind == "inf"
        for x, y in zip((per_tile.master, per_tile.m, per_tile.v), (counter.master, counter.m, counter.v)):
            assert torch.equal(x[mask].view(torch.int32), y[mask].view(torch.int32)), step
        assert torch.equal(per_tile.params_flat.view(torch.int16), counter.params_flat.view(torch.int16))
    per_tile.close()
    counter.close()
