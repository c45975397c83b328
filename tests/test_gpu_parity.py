"""CUDA path versus the oracle, element by element, through the C ABI.

Acceptance: reduced (communication-dtype) values, the overflow flag and the
loss-scale/step-count trajectory bit-exact; fp32 master/m/v within 1e-5
relative error (absolute below 1e-30); cast-out parameters within 1 ulp.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _parity import INF_BITS, Pair, to_np
from mixed_precision_gb300 import ZeroError
from mixed_precision_gb300 import _abi as abi
from mixed_precision_gb300.engine import Hparams

pytestmark = pytest.mark.gpu


def small_qwen_shapes():
    return wl.qwen3_0_6b_shapes(vocab=1000, hidden=128, layers=2, q_dim=256, kv_dim=128, ffn=384,
                                head_dim=32)


def test_tiny_four_steps_with_inf():
    """The tiny fp16 workload: W=2, ZeRO-2, S0 = 2^16, +inf in step 3."""
    w = wl.workload("tiny")
    pr = Pair(w.shapes, w.world, w.stage, w.bucket_bytes, w.grad_dtype, w.param_dtype,
              init_scale=w.init_scale, dynamic=True, index=w.index)
    hp = Hparams(lr=w.lr, weight_decay=w.weight_decay, max_grad_norm=w.max_grad_norm)
    rank, idx = wl.inject_position(pr.numel, pr.z.offsets, w.world, seed=1234)
    scales, ts = [], []
    for step in range(1, 5):
        inj = [(rank, idx, INF_BITS[wl.F16])] if step == 3 else None
        g = pr.grads(step, w.grad_sigma, inject=inj)
        st, info, gc = pr.step(g, hp)
        pr.check(st, info, gc)
        scales.append(st["scale"])
        ts.append(st["t"])
        assert st["overflow"] == (1 if step == 3 else 0)
    assert ts == [1, 2, 2, 3]
    assert scales == [2.0 ** 16, 2.0 ** 16, 2.0 ** 15, 2.0 ** 15]


@pytest.mark.parametrize("W,stage,gdt,cdt,pdt,bucket", [
    (2, 2, wl.BF16, -1, wl.BF16, 64_000),
    (2, 1, wl.BF16, -1, wl.BF16, 64_000),
    (4, 2, wl.F16, wl.F32, wl.F16, 200_000),
    (8, 2, wl.BF16, -1, wl.BF16, 500_000_000),
    (3, 2, wl.BF16, -1, wl.F16, 30_000),
    (5, 1, wl.F32, wl.BF16, wl.BF16, 100_000),
    (1, 2, wl.F16, -1, wl.F16, 50_000),
])
def test_small_qwen_shaped(W, stage, gdt, cdt, pdt, bucket):
    pr = Pair(small_qwen_shapes(), W, stage, bucket, gdt, pdt, cdt, init_scale=8.0, index=20 + W)
    for step, hp in enumerate([Hparams(), Hparams(max_grad_norm=0.0, grad_divisor=1.0),
                               Hparams(lr=3e-4, weight_decay=0.1, max_grad_norm=1e-3)]):
        st, info, gc = pr.step(pr.grads(step, 1e-3), hp)
        pr.check(st, info, gc)
        assert st["t"] == step + 1


def test_stage1_equals_stage2_bitwise():
    shapes = small_qwen_shapes()
    res = []
    for stage in (1, 2):
        pr = Pair(shapes, 8, stage, 100_000, wl.F16, wl.F16, init_scale=2.0 ** 16, dynamic=True,
                  index=31)
        for step in range(3):
            st, info, gc = pr.step(pr.grads(step, 1e-4), Hparams())
            pr.check(st, info, gc)
        res.append([to_np(t) for t in (pr.z.master, pr.z.m, pr.z.v, pr.z.params_flat)] + [st])
    for a, b in zip(res[0][:4], res[1][:4]):
        assert np.array_equal(a, b)
    assert res[0][4] == res[1][4]


@pytest.mark.parametrize("W", [3, 16, 64])
def test_generic_world_and_ragged(W):
    """Odd and large W (the runtime-W kernel path), 1-element, empty and ragged
    parameters that straddle bucket and shard boundaries."""
    rng = np.random.default_rng(W)
    sizes = [1, 0, 7, 63, 64, 65, 129, 8191, 8193, 20000, 3, 1]
    sizes += [int(x) for x in rng.integers(1, 3000, size=10)]
    shapes = [(s,) for s in sizes]
    pr = Pair(shapes, W, 2, 4096 * 2, wl.BF16, wl.BF16, index=40 + W)
    for step in range(2):
        st, info, gc = pr.step(pr.grads(step, 1e-2), Hparams(max_grad_norm=0.5))
        pr.check(st, info, gc)


def test_pointer_table_mode_matches_flat():
    """Per-tensor gradient pointers (NULL = all-zero) give the same bits as the
    flat buffers with those parameters zeroed."""
    shapes = small_qwen_shapes()
    zero = (1, 4, 7)
    outs = []
    for mode in ("flat", "tensors"):
        pr = Pair(shapes, 4, 2, 80_000, wl.BF16, wl.BF16, index=50)
        for step in range(2):
            g = pr.grads(step, 1e-3, zero_params=zero)
            st, info, gc = pr.step(g, Hparams(), mode=mode)
            pr.check(st, info, gc)
        outs.append([to_np(t) for t in (pr.z.master, pr.z.m, pr.z.v, pr.z.params_flat)])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("W,gdt,cdt,stage", [(3, wl.BF16, wl.BF16, 2), (4, wl.BF16, wl.BF16, 2),
                                             (8, wl.F16, wl.F16, 2), (4, wl.BF16, wl.F32, 2),
                                             (5, wl.F32, wl.F32, 2), (4, wl.BF16, wl.BF16, 1)])
def test_pointer_table_partial_nulls_match_flat_and_oracle(W, gdt, cdt, stage):
    """Gradients that are NULL on some ranks only (the routed-experts
    pattern): a tile's live ranks take longer chunks in the reduce's stages.
    Every live count from 0 to W occurs (each rank drops about half of the
    parameters); tensors span several tiles, with ragged tails. The result
    matches the oracle and equals the flat step's, norm included, bit for
    bit."""
    rng = np.random.default_rng(300 + W)
    sizes = [int(x) for x in rng.integers(1, 40_000, size=30)] + [8192, 8193, 24_577, 7, 1]
    shapes = [(n,) for n in sizes]
    P = len(shapes)
    # parameter 0 dropped everywhere, parameter 1 nowhere
    dropped = [(set(int(p) for p in rng.choice(P, size=P // 2, replace=False)) | {0}) - {1}
               for _ in range(W)]
    live = [sum(p not in d for d in dropped) for p in range(P)]
    assert 0 in live and W in live and any(0 < c < W for c in live)
    pdt = wl.F16 if gdt == wl.F16 else wl.BF16
    outs = []
    for mode in ("flat", "tensors"):
        pr = Pair(shapes, W, stage, 150_000, gdt, pdt, comm_dtype=cdt, index=60 + W)
        for step in range(2):
            g = pr.grads(step, 1e-3)
            for r in range(W):
                for p in dropped[r]:
                    g[r][pr.offsets[p]:pr.offsets[p] + sizes[p]] = 0
            st, info, gc = pr.step(g, Hparams(max_grad_norm=0.05), mode=mode)
            pr.check(st, info, gc)
        assert info.clip_coef < 1.0
        outs.append([to_np(t) for t in (pr.z.master, pr.z.m, pr.z.v, pr.z.params_flat)]
                    + [st["grad_norm"], st["norm_sq_raw"]])
    for a, b in zip(outs[0][:4], outs[1][:4]):
        assert np.array_equal(a, b)
    assert outs[0][4:] == outs[1][4:]


@pytest.mark.parametrize("stage", [1, 2])
def test_per_tensor_launch_matches_oracle(stage):
    """The tensor-by-tensor launch sequence (the hook-style baseline) computes
    the same step: ragged tensors across several buckets and rank slices."""
    rng = np.random.default_rng(stage)
    shapes = [(int(x),) for x in rng.integers(1, 30000, size=25)] + [(0,), (70000,)]
    pr = Pair(shapes, 4, stage, 100_000, wl.BF16, wl.BF16, init_scale=4.0, dynamic=True, index=110)
    for step in range(3):
        inj = [(0, pr.z.offsets[3], INF_BITS[wl.BF16])] if step == 1 else None
        st, info, gc = pr.step(pr.grads(step, 1e-3, inject=inj), Hparams(), mode="per_tensor_launch")
        pr.check(st, info, gc)


def test_host_entry_point_matches_device():
    shapes = small_qwen_shapes()
    outs = []
    for mode in ("flat", "host"):
        pr = Pair(shapes, 2, 2, 500_000_000, wl.BF16, wl.BF16, index=60)
        st, info, gc = pr.step(pr.grads(0, 1e-3), Hparams(), mode=mode)
        pr.check(st, info, gc)
        outs.append([to_np(t) for t in (pr.z.master, pr.z.params_flat)])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("stage", [1, 2])
def test_host_steps_back_to_back_overlap(stage):
    """Two zero_step_host calls with different gradients into the same device
    buffers, no synchronisation between them: the second step's copies may
    overlap the first step's update kernel (stage 2) but never its reduce.
    The final state matches two oracle steps."""
    import oracle as orc
    from _parity import to_np
    shapes = small_qwen_shapes()
    pr = Pair(shapes, 2, stage, 100_000, wl.BF16, wl.BF16, index=160)
    g0, g1 = pr.grads(0, 1e-3), pr.grads(1, 1e-3)
    dev = [torch.empty(pr.np, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    pin0, pin1 = [x.pin_memory() for x in g0], [x.pin_memory() for x in g1]
    hp = Hparams()
    pr.z.step_host(pin0, dev, hp)
    pr.z.step_host(pin1, dev, hp)
    torch.cuda.synchronize()
    st = pr.z.scaler_state()
    o_hp = orc.Hparams(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.max_grad_norm,
                       hp.grad_divisor)
    for g in (g0, g1):
        info = orc.zero_step(pr.numel, pr.W, stage, pr.bucket, pr.gdt, pr.cdt, pr.pdt,
                             [to_np(x) for x in g], pr.o_master, pr.o_m, pr.o_v, pr.o_params, o_hp,
                             pr.o_scaler, allreduce_out=pr.o_out)
        for h, x in zip(pr.hist, (pr.o_master, pr.o_m, pr.o_v)):
            np.maximum(h, np.abs(x), out=h)
    assert st["t"] == 2
    pr.check(st, info, g1)


def test_host_steps_alternating_device_sets():
    """Three zero_step_host calls alternating two device gradient sets (A, B,
    A) without synchronising: each copy waits only for the reduce kernel that
    last read its own set. The final state matches three oracle steps."""
    import oracle as orc
    shapes = small_qwen_shapes()
    pr = Pair(shapes, 3, 2, 100_000, wl.BF16, wl.BF16, index=161)
    gs = [pr.grads(k, 1e-3) for k in range(3)]
    sets = [[torch.empty(pr.np, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
            for _ in range(2)]
    pins = [[x.pin_memory() for x in g] for g in gs]
    hp = Hparams()
    for k in range(3):
        pr.z.step_host(pins[k], sets[k % 2], hp)
    torch.cuda.synchronize()
    st = pr.z.scaler_state()
    o_hp = orc.Hparams(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.max_grad_norm,
                       hp.grad_divisor)
    for g in gs:
        info = orc.zero_step(pr.numel, pr.W, 2, pr.bucket, pr.gdt, pr.cdt, pr.pdt,
                             [to_np(x) for x in g], pr.o_master, pr.o_m, pr.o_v, pr.o_params, o_hp,
                             pr.o_scaler, allreduce_out=pr.o_out)
        for h, x in zip(pr.hist, (pr.o_master, pr.o_m, pr.o_v)):
            np.maximum(h, np.abs(x), out=h)
    assert st["t"] == 3
    pr.check(st, info, gs[2])
    # the device sets hold the last gradients copied into each
    for k in (1, 2):
        for r in range(3):
            assert np.array_equal(to_np(sets[k % 2][r]), to_np(gs[k][r]))


def test_overflow_at_shard_edges_skips():
    """+inf / -inf / NaN at the first or last real element of shards in the
    first and last rank: flag set, step skipped, state untouched, scale halved."""
    shapes = [(300,), (64,), (513,), (1000,)]
    pr = Pair(shapes, 3, 2, 1024, wl.F16, wl.F16, init_scale=1024.0, dynamic=True, index=70)
    st, info, gc = pr.step(pr.grads(0, 1e-2), Hparams())
    pr.check(st, info, gc)
    positions = []
    for _, _, f0, _, ln in pr.L.shard_ranges():
        real = np.nonzero(pr.mask_flat[f0:f0 + ln])[0]
        if len(real):
            positions += [f0 + int(real[0]), f0 + int(real[-1])]
    bad_bits = [0x7C00, 0xFC00, 0x7E00]
    for k, pos in enumerate(positions[:8]):
        before = [to_np(t).copy() for t in (pr.z.master, pr.z.m, pr.z.v, pr.z.params_flat)]
        rank = 0 if k % 2 == 0 else pr.W - 1
        g = pr.grads(k + 1, 1e-2, inject=[(rank, pos, bad_bits[k % 3])])
        st, info, gc = pr.step(g, Hparams())
        assert st["overflow"] == 1 and st["skipped"] == 1
        pr.check(st, info, gc)
        after = [to_np(t) for t in (pr.z.master, pr.z.m, pr.z.v, pr.z.params_flat)]
        for a, b in zip(before, after):
            assert np.array_equal(a, b)


def test_fp16_overflow_only_after_reduction():
    """Finite fp16 inputs whose fp32 sum rounds past 65504 overflow in fp16
    communication but not in fp32 communication."""
    shapes = [(4096,), (100,)]
    for cdt, expect in ((wl.F16, 1), (wl.F32, 0)):
        pr = Pair(shapes, 2, 2, 1 << 20, wl.F16, wl.F16, cdt, init_scale=4.0, dynamic=True, index=80)
        g = pr.grads(0, 1e-2)
        for r in range(2):
            g[r][17] = 40000.0
        st, info, gc = pr.step(g, Hparams())
        assert st["overflow"] == expect
        pr.check(st, info, gc)


def test_padding_garbage_is_ignored():
    """The gradient buffers' padding holds NaN (the generator's default) and the
    step still matches the oracle, which never reads padding."""
    pr = Pair([(100,), (30,), (200,)], 2, 2, 512, wl.BF16, wl.BF16, index=90)
    st, info, gc = pr.step(pr.grads(0, 1e-2), Hparams())
    assert np.isnan(gc[0][100].float().item())
    assert st["overflow"] == 0
    pr.check(st, info, gc)


def test_scaler_growth_and_long_trajectory():
    """fp16, W=8, dynamic scaling with growth after N=10 clean steps and an
    +inf every 13th step: 40 steps (growth at 10, 23, 36; backoff at 13, 26,
    39), scale/counter/t bit-exact every step."""
    shapes = [(1000,), (129,), (4000,)]
    pr = Pair(shapes, 8, 2, 4096, wl.F16, wl.F16, init_scale=2.0 ** 10, dynamic=True,
              growth_interval=10, index=95)
    rank, idx = wl.inject_position(pr.numel, pr.z.offsets, 8, seed=5)
    seen_growth = False
    prev = 2.0 ** 10
    for step in range(1, 41):
        inj = [(rank, idx, INF_BITS[wl.F16])] if step % 13 == 0 else None
        st, info, gc = pr.step(pr.grads(step, 1e-3, inject=inj), Hparams())
        pr.check(st, info, gc)
        seen_growth |= st["scale"] > prev
        prev = st["scale"]
        if step in (10, 23, 36):
            assert st["counter"] == 0 and st["overflow"] == 0
    assert seen_growth
    assert st["scale"] == 2.0 ** 10  # three doublings, three halvings


def test_empty_model():
    """All parameters empty: no element work, the step still advances t."""
    pr = Pair([(0,), (0, 5)], 2, 2, 1024, wl.BF16, wl.BF16, index=99)
    st, info, gc = pr.step(pr.grads(0, 1e-3), Hparams())
    assert st["t"] == 1 and info.grad_norm == 0.0


def test_gather_export_import():
    shapes = small_qwen_shapes()
    pr = Pair(shapes, 4, 2, 100_000, wl.BF16, wl.BF16, index=101)
    st, info, gc = pr.step(pr.grads(0, 1e-3), Hparams())
    pr.check(st, info, gc)
    z = pr.z
    # K4: two replicas of per-tensor storage, one of them deliberately offset by
    # one element (2-byte aligned only) to take the unaligned path
    backing = torch.empty(z.np + 64, dtype=torch.bfloat16, device="cuda")
    rep0 = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in shapes]
    rep1, at = [], 1
    for s, n in zip(shapes, pr.numel):
        rep1.append(backing[at:at + n].view(s))
        at += n + 1
    z.gather([rep0, rep1])
    torch.cuda.synchronize()
    for p in range(len(shapes)):
        ref = z.param_view(z.params_flat, p)
        assert torch.equal(rep0[p].view(torch.int16), ref.view(torch.int16))
        assert torch.equal(rep1[p].view(torch.int16), ref.view(torch.int16))
    # export to flat order and back
    master_f, m_f, v_f = z.export_state()
    for flat_t, shard_t in ((master_f, z.master), (m_f, z.m), (v_f, z.v)):
        exp = np.zeros(z.np, np.float32)
        exp[pr.perm] = to_np(shard_t)[:z.np]  # the GPU's own rank-major state, permuted
        got = to_np(flat_t)
        assert np.array_equal(got[pr.mask_flat], exp[pr.mask_flat])
        assert np.all(got[~pr.mask_flat] == 0)
    saved = [to_np(t).copy() for t in (z.master, z.m, z.v)]
    z.master.zero_(), z.m.zero_(), z.v.zero_()
    z.import_state(master_f, m_f, v_f)
    torch.cuda.synchronize()
    for t, s in zip((z.master, z.m, z.v), saved):
        assert np.array_equal(to_np(t)[pr.mask_shard], s[pr.mask_shard])


def test_invalid_device_arguments():
    pr = Pair([(100,)], 2, 2, 1024, wl.BF16, wl.BF16, index=102)
    g = [x.cuda() for x in pr.grads(0, 1e-3)]
    hp = Hparams()
    with pytest.raises(ZeroError) as e:
        pr.z.step([g[0], g[1][1:]], hp)  # 2-byte offset: not 16-byte aligned
    assert e.value.code == 1
    with pytest.raises(ZeroError) as e:
        pr.z.step(g, Hparams(beta1=1.0))
    assert e.value.code == 1
    # nothing was enqueued: a valid step afterwards is the first one
    pr.z.step(g, hp)
    torch.cuda.synchronize()
    assert pr.z.scaler_state()["t"] == 1


def test_deterministic_across_runs():
    """The reductions run in a fixed order, so two identical runs give
    identical bits (norm included)."""
    outs = []
    for _ in range(2):
        pr = Pair(small_qwen_shapes(), 4, 2, 80_000, wl.BF16, wl.BF16, index=180)
        for step in range(2):
            st, info, gc = pr.step(pr.grads(step, 1e-3), Hparams())
        outs.append([to_np(t) for t in (pr.z.master, pr.z.m, pr.z.v, pr.z.params_flat)]
                    + [to_np(pr.z.scratch)[:pr.np][pr.mask_shard]]  # padding is never written
                    + [st["grad_norm"], st["norm_sq_raw"]])
    for a, b in zip(outs[0][:5], outs[1][:5]):
        assert np.array_equal(a, b)
    assert outs[0][5:] == outs[1][5:]


def test_runs_on_the_given_stream():
    """Work goes to the stream passed in: a side stream, joined afterwards."""
    pr = Pair(small_qwen_shapes(), 2, 2, 80_000, wl.BF16, wl.BF16, index=181)
    g = pr.grads(0, 1e-3)
    dev = [x.cuda() for x in g]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        pr.z.step(dev, Hparams(), stream=side)
        st_side = pr.z.scaler_state(stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    # the oracle side of the same step
    import oracle as orc
    o_hp = orc.Hparams()
    info = orc.zero_step(pr.numel, 2, 2, pr.bucket, pr.gdt, pr.cdt, pr.pdt, [to_np(x) for x in g],
                         pr.o_master, pr.o_m, pr.o_v, pr.o_params, o_hp, pr.o_scaler)
    for h, x in zip(pr.hist, (pr.o_master, pr.o_m, pr.o_v)):
        np.maximum(h, np.abs(x), out=h)
    pr.check(st_side, info, g)


def test_stage1_in_place_allreduce():
    """ZeRO-1 with the all-reduce outputs aliasing the gradient buffers: each
    rank's buffer ends up holding the reduced gradient; the step matches a
    run with separate outputs."""
    shapes = small_qwen_shapes()
    a = Pair(shapes, 4, 1, 80_000, wl.F16, wl.F16, index=182)
    b = Pair(shapes, 4, 1, 80_000, wl.F16, wl.F16, index=182)
    g = a.grads(0, 1e-3)
    st_a, info, gc = a.step(g, Hparams())
    a.check(st_a, info, gc)
    dev = [x.cuda() for x in g]
    b.z.step(dev, Hparams(), allreduce_out=dev)
    torch.cuda.synchronize()
    for t_a, t_b in ((a.z.master, b.z.master), (a.z.params_flat, b.z.params_flat)):
        assert np.array_equal(to_np(t_a), to_np(t_b))
    for w in range(4):
        assert np.array_equal(to_np(dev[w])[a.mask_flat], to_np(a.z.allreduce_out[w])[a.mask_flat])


def test_rebind_state_buffers():
    """Binding new buffers redirects the step; the library's own block is reused."""
    pr = Pair([(5000,), (300,)], 2, 2, 1 << 20, wl.BF16, wl.BF16, index=183)
    z = pr.z
    owned = abi.zero_layout_query(z.handle).device_bytes_owned
    old = (z.master, z.m, z.v, z.params_flat, z.scratch)
    old_bits = [to_np(t).copy() for t in old]
    copies = [t.clone() for t in old]
    z.bind(*copies)
    z.master, z.m, z.v, z.params_flat, z.scratch = copies
    z.init(torch.zeros(z.np, dtype=torch.float32, device="cuda"))
    st, info, gc = pr.step(pr.grads(0, 1e-3), Hparams(max_grad_norm=0.0))
    assert abi.zero_layout_query(z.handle).device_bytes_owned == owned
    assert st["t"] == 1
    assert np.count_nonzero(to_np(z.master)[pr.mask_shard]) > 0  # the new buffers were stepped
    for t, bits in zip(old, old_bits):  # the old ones were not touched
        assert np.array_equal(to_np(t), bits)
