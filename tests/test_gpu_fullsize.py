"""Full-size parity of the named workloads, in the launch configuration the
benchmark times, on sampled outputs (see _fullsize.py).

- Qwen3-0.6B-shaped, W=2, ZeRO-2, bf16 (the benchmark's workload): two steps.
- Qwen3-0.6B-shaped, W=8, fp16 dynamic loss scaling, ZeRO-1 and ZeRO-2:
  the two stages bit-identical; sampled parity; 200 steps with +inf at steps
  50/100/150/200 and the scale/counter/t trajectory bit-exact.
- MoE ~3.9B, W=4, bf16, 14 of 16 experts' gradients zero per rank and layer:
  sampled parity, and the per-tensor entry point (NULL for the zero experts)
  bit-identical to the flat one.
- The layout sweep's 2000 ragged tensors (1.69G elements; 1 MB buckets at
  W=2, 1 GB buckets at W=8): sampled parity of the flat step and of the step
  launched tensor by tensor, which must also store the same reduced values.
- The speculative step at full size, in the launch configuration
  `bench.py --speculative` times: fp16 W=8 (clipping inactive) commits, skips
  on +inf and commits again, in stage 2 and in stage 1 (where the single pass
  also writes the all-reduce outputs); Qwen3 bf16 W=2 at clip 1.0 (clipping active)
  falls back, then is predicted to. Sampled parity on every step.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _fullsize import SampledOracle, sample_indices
from _parity import INF_BITS, to_np
from mixed_precision_gb300.engine import Hparams, ZeroStep

pytestmark = pytest.mark.gpu


def _setup(w, stage=None, speculative=False):
    stage = w.stage if stage is None else stage
    z = ZeroStep(w.shapes, w.world, stage, w.bucket_bytes, w.grad_dtype, w.param_dtype, w.comm_dtype)
    z.allocate(speculative=speculative)
    numel = wl.numels(w.shapes)
    master0 = wl.master_init(z.offsets, numel, z.np, w.master_sigma, wl.master_seed(w.index),
                             device="cuda")
    z.init(master0, init_scale=w.init_scale, dynamic=w.dynamic, growth_interval=w.growth_interval)
    return z, numel, master0


def _grads(z, w, numel, step):
    return [wl.flat_grads(z.offsets, numel, z.np, w.grad_sigma, wl.grad_seed(w.index, r, step),
                          w.grad_dtype, device="cuda", zero_params=wl.zero_params(w, r))
            for r in range(w.world)]


def _hp(w):
    return Hparams(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                   max_grad_norm=w.max_grad_norm)


def test_fullsize_qwen3_bf16_w2():
    w = wl.workload("qwen3_0.6b_bf16_w2")
    z, numel, master0 = _setup(w)
    so = SampledOracle(z, numel, master0, sample_indices(z, numel, 200_000, 1), w.init_scale,
                       w.dynamic, w.growth_interval)
    del master0
    for step in range(2):
        g = _grads(z, w, numel, step)
        z.step(g, _hp(w))
        torch.cuda.synchronize()
        st = z.scaler_state()
        info, red_at = so.step(g, _hp(w))
        so.check(st, info, red_at)
        del g
    z.close()


def test_fullsize_qwen3_fp16_w8_stages_and_trajectory():
    w = wl.workload("qwen3_0.6b_fp16_w8")
    z2, numel, master0 = _setup(w, stage=2)
    z1, _, _ = _setup(w, stage=1)
    so = SampledOracle(z2, numel, master0, sample_indices(z2, numel, 100_000, 2), w.init_scale,
                       w.dynamic, w.growth_interval)
    del master0
    g = _grads(z2, w, numel, 0)
    hp = _hp(w)
    # step 1: sampled parity, and ZeRO-1 == ZeRO-2 bit for bit
    z2.step(g, hp)
    z1.step(g, hp)
    torch.cuda.synchronize()
    st = z2.scaler_state()
    assert st == z1.scaler_state()
    info, red_at = so.step(g, hp)
    so.check(st, info, red_at)
    for a, b in ((z1.master, z2.master), (z1.m, z2.m), (z1.v, z2.v), (z1.params_flat, z2.params_flat)):
        assert torch.equal(a.view(torch.int32 if a.dtype == torch.float32 else torch.int16),
                           b.view(torch.int32 if b.dtype == torch.float32 else torch.int16))
    z1.close()
    # 199 more steps on the same gradients, +inf at 1-indexed steps 50/100/150/200
    rank, idx = wl.inject_position(numel, z2.offsets, w.world, seed=3)
    bits = INF_BITS[wl.F16]
    vals = [to_np(g[r][idx:idx + 1]) for r in range(w.world)]
    vals[rank] = np.array([bits], np.uint16)
    # the injected element's reduced value is +inf, so is the step's sum of squares
    inj_ovf, inj_sq = oracle.overflow_sumsq(oracle.reduce(vals, wl.F16, wl.F16), wl.F16)
    saved = g[rank][idx].clone()
    for step in range(2, 201):
        inject = step % 50 == 0
        if inject:
            g[rank].view(torch.int16)[idx] = int(np.array(bits, np.uint16).view(np.int16))
        z2.step(g, hp)
        st = z2.scaler_state()
        if inject:
            g[rank][idx] = saved
        # the sampled oracle steps on the same gradients: the first step's
        # global reduce, with the injected step's overflow flag
        o_info, red_at = so.step_repeat(hp, *((inj_ovf, inj_sq) if inject else ()))
        assert (st["overflow"], st["skipped"]) == (o_info.overflow, o_info.skipped)
        assert (st["scale"], st["counter"], st["t"]) == (so.scaler.scale, so.scaler.counter,
                                                         so.scaler.t)
        if step == 199:  # the last clean step: the sampled state after 196 updates
            so.check(st, o_info, red_at)
    assert so.scaler.scale == 2.0 ** 12 and so.scaler.t == 196
    # the skipped step 200 left the state as step 199 did
    so.check(st, o_info, red_at, reduced=False)
    z2.close()


def test_fullsize_moe_w4_flat_and_tensors():
    w = wl.workload("moe_3.9b_bf16_w4")
    z, numel, master0 = _setup(w)
    so = SampledOracle(z, numel, master0, sample_indices(z, numel, 100_000, 3), w.init_scale,
                       w.dynamic, w.growth_interval)
    del master0
    g = _grads(z, w, numel, 0)
    hp = _hp(w)
    z.step(g, hp)
    torch.cuda.synchronize()
    st = z.scaler_state()
    info, red_at = so.step(g, hp)
    so.check(st, info, red_at)
    # the same step from per-tensor pointers, the zero experts passed as NULL
    zt, _, master0 = _setup(w)
    del master0
    per = []
    for r in range(w.world):
        zero = set(wl.zero_params(w, r))
        per.append([None if p in zero else g[r][off:off + n]
                    for p, (off, n) in enumerate(zip(zt.offsets, numel))])
    zt.step_tensors(per, hp)
    torch.cuda.synchronize()
    assert zt.scaler_state() == st
    for a, b in ((z.master, zt.master), (z.m, zt.m), (z.v, zt.v)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(z.params_flat.view(torch.int16), zt.params_flat.view(torch.int16))
    zt.close()
    z.close()


@pytest.mark.parametrize("world,bucket", [(2, 1 << 20), (8, 1 << 30)])
def test_fullsize_ragged_2000_flat_and_per_tensor_launch(world, bucket):
    w = wl.workload("ragged_2000", world=world, bucket_bytes=bucket)
    z, numel, master0 = _setup(w)
    # the greedy packing: 955 buckets of 1 MB (a tensor larger than the bucket
    # gets one of its own), or 4 of 1 GB
    assert z.info.n_buckets == (955 if bucket == 1 << 20 else 4)
    idx = sample_indices(z, numel, 100_000, 5)
    so = SampledOracle(z, numel, master0, idx, w.init_scale, w.dynamic, w.growth_interval)
    del master0
    g = _grads(z, w, numel, 0)
    hp = _hp(w)
    z.step(g, hp)
    torch.cuda.synchronize()
    st = z.scaler_state()
    info, red_at = so.step(g, hp)
    assert info.clip_coef < 1.0  # clip 1.0 is active on this workload
    so.check(st, info, red_at)
    z.close()
    del z
    # the same step with two kernel launches per parameter: the same oracle
    # step from the same initial state (its global reduce reused)
    zt, _, master0 = _setup(w)
    sot = SampledOracle(zt, numel, master0, idx, w.init_scale, w.dynamic, w.growth_interval)
    del master0
    zt.step_per_tensor_launch(g, hp)
    torch.cuda.synchronize()
    stt = zt.scaler_state()
    sot.last_reduce = so.last_reduce
    info_t, _ = sot.step_repeat(hp)
    sot.check(stt, info_t, red_at)
    zt.close()


@pytest.mark.parametrize("name,stage,plan", [
    ("qwen3_0.6b_fp16_w8", 2, ["commit", "skip", "commit"]),
    ("qwen3_0.6b_fp16_w8", 1, ["commit", "skip", "commit"]),  # also writes the all-reduce outputs
    ("qwen3_0.6b_bf16_w2", 2, ["fallback", "predicted"]),
])
def test_fullsize_speculative(name, stage, plan):
    w = wl.workload(name)
    z, numel, master0 = _setup(w, stage=stage, speculative=True)
    so = SampledOracle(z, numel, master0, sample_indices(z, numel, 100_000, 4), w.init_scale,
                       w.dynamic, w.growth_interval)
    del master0
    hp = _hp(w)
    rank, idx = wl.inject_position(numel, z.offsets, w.world, seed=9)
    for step, kind in enumerate(plan):
        g = _grads(z, w, numel, step)
        if kind == "skip":
            g[rank][idx] = float("inf")
        z.step_speculative(g, hp)
        torch.cuda.synchronize()
        st = z.scaler_state()
        assert st["fast_path"] == (kind == "commit")
        assert st["skipped"] == (kind == "skip")
        info, red_at = so.step(g, hp)
        so.check(st, info, red_at, reduced=stage == 1 or kind in ("fallback", "predicted"))
        if kind in ("fallback", "predicted"):
            assert st["clip_coef"] < 1.0
        del g
    z.close()


def test_tensor_past_2_31_elements():
    """One parameter of 2^31 + 200 elements between two small ones, W=2,
    ZeRO-2, bf16: offsets inside that parameter pass 2^31 in the per-tensor
    pointer mode and in the per-tensor gather. The flat and per-tensor entry
    points agree bit for bit, the sampled oracle agrees (the samples include
    the parameter's last element), and the gathered tensors equal the flat
    parameters."""
    shapes = [(300,), ((1 << 31) + 200,), (77,)]
    W = 2

    def setup():
        z = ZeroStep(shapes, W, 2, 1 << 30, wl.BF16, wl.BF16)
        z.allocate()
        m0 = wl.master_init(z.offsets, numel, z.np, 0.02, wl.master_seed(150), device="cuda")
        z.init(m0)
        return z, m0

    numel = wl.numels(shapes)
    za, master0 = setup()
    zb, m0b = setup()
    del m0b
    assert za.offsets[1] + numel[1] > 1 << 31
    so = SampledOracle(za, numel, master0, sample_indices(za, numel, 20_000, 5), 1.0, False, 1000)
    del master0
    g = [wl.flat_grads(za.offsets, numel, za.np, 1e-4, wl.grad_seed(150, r, 0), wl.BF16,
                       device="cuda") for r in range(W)]
    hp = Hparams()
    za.step(g, hp)
    zb.step_tensors([[zb.param_view(g[r], p) for p in range(len(shapes))] for r in range(W)], hp)
    torch.cuda.synchronize()
    st = za.scaler_state()
    assert st == zb.scaler_state()
    for a, b in ((za.master, zb.master), (za.m, zb.m), (za.v, zb.v)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(za.params_flat.view(torch.int16), zb.params_flat.view(torch.int16))
    zb.close()
    del zb
    info, red_at = so.step(g, hp)
    so.check(st, info, red_at)
    del g
    dst = [[torch.empty(n, dtype=torch.bfloat16, device="cuda") for n in numel]]
    za.gather(dst)
    torch.cuda.synchronize()
    for p in range(len(shapes)):
        assert torch.equal(dst[0][p].view(torch.int16),
                           za.param_view(za.params_flat, p).view(torch.int16))
    za.close()
