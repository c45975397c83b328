"""GPU tests of the rows beyond the step itself: gradient accumulation into
fp32 main gradients, and the bounded-wait failure path."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _parity import Pair, to_np
from mixed_precision_gb300 import ZeroError
from mixed_precision_gb300 import _abi as abi
from mixed_precision_gb300.engine import Hparams

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    """A wait on data that never arrives gives up after its retry limit and is
    reported as ZERO_ERR_TIMEOUT; the next step runs normally."""
    stream = torch.cuda.current_stream().cuda_stream
    with pytest.raises(ZeroError) as e:
        abi.zero_selftest_wait_timeout(2000, stream)
    assert e.value.code == abi.ZERO_ERR_TIMEOUT
    pr = Pair([(1000,), (77,)], 2, 2, 1 << 20, wl.BF16, wl.BF16, index=120)
    st, info, gc = pr.step(pr.grads(0, 1e-3), Hparams())
    pr.check(st, info, gc)


def test_layout_timeout_freezes_every_step_until_init():
    """A bounded wait that gives up inside a layout (the self-test records it
    in the layout's device error word, as a step kernel does) is reported as
    ZERO_ERR_TIMEOUT by the next state read. Every step entry point then
    leaves master, m, v, the parameters and the scaler as they were, and
    zero_state_init makes the layout usable again: its next step matches a
    fresh layout's bit for bit."""
    from mixed_precision_gb300.engine import ZeroStep
    shapes = [(3000,), (129,), (40000,), (1,)]
    W = 2
    hp = Hparams()
    stream = torch.cuda.current_stream().cuda_stream

    def fresh():
        z = ZeroStep(shapes, W, 2, 100_000, wl.BF16, wl.BF16)
        z.allocate(speculative=True)
        z.init(wl.master_init(z.offsets, z.numels, z.np, 0.02, wl.master_seed(140), device="cuda"))
        return z

    def grads(z, step):
        return [wl.flat_grads(z.offsets, z.numels, z.np, 1e-3, wl.grad_seed(140, r, step), wl.BF16,
                              device="cuda") for r in range(W)]

    def snapshot(z):  # both state sets (no state read: it would report the error)
        return [t.clone() for t in (z.master, z.m, z.v, z.master2, z.m2, z.v2, z.params_flat)]

    z = fresh()
    z.step(grads(z, 0), hp)
    st0 = z.scaler_state()
    assert st0["t"] == 1
    before = snapshot(z)
    with pytest.raises(ZeroError) as e:
        abi.zero_selftest_layout_timeout(z.handle, 2000, stream)
    assert e.value.code == abi.ZERO_ERR_TIMEOUT
    g = grads(z, 1)
    per_tensor = [[z.param_view(g[w], p) for p in range(len(shapes))] for w in range(W)]
    host = [t.cpu().pin_memory() for t in g]
    dev = z.new_grad_buffers()
    z.step(g, hp)
    z.step_speculative(g, hp)
    z.step_tensors(per_tensor, hp)
    z.step_speculative_tensors(per_tensor, hp)
    z.step_per_tensor_launch(g, hp)
    z.step_host(host, dev, hp)
    torch.cuda.synchronize()
    with pytest.raises(ZeroError) as e:
        z.scaler_state()
    assert e.value.code == abi.ZERO_ERR_TIMEOUT
    for a, b in zip(before, snapshot(z)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # initialised again: the error is gone and the layout steps like a new one
    z.init(wl.master_init(z.offsets, z.numels, z.np, 0.02, wl.master_seed(140), device="cuda"))
    ref = fresh()
    for k in range(2):
        gk = grads(z, k)
        z.step(gk, hp)
        ref.step(gk, hp)
    torch.cuda.synchronize()
    sa, sb = z.scaler_state(), ref.scaler_state()
    assert sa["t"] == sb["t"] == 2 and sa["scale"] == sb["scale"]
    mask = torch.zeros(z.np, dtype=torch.bool, device="cuda")
    for b in range(z.info.n_buckets):
        for r in range(W):
            f0, s0, ln = abi.zero_shard_range(z.handle, b, r)
            for off, n in zip(z.offsets, z.numels):
                lo, hi = max(off, f0), min(off + n, f0 + ln)
                if lo < hi:
                    mask[s0 + lo - f0:s0 + hi - f0] = True
    for a, b in zip(z.current_state(), ref.current_state()):
        assert torch.equal(a[:z.np][mask].view(torch.int32), b[:z.np][mask].view(torch.int32))
    assert torch.equal(z.params_flat.view(torch.int16), ref.params_flat.view(torch.int16))
    z.close()
    ref.close()


@pytest.mark.parametrize("micro_dtype,comm", [(wl.BF16, wl.BF16), (wl.F16, wl.F32)])
def test_accumulate_then_boundary_step(micro_dtype, comm):
    """Three bf16/fp16 micro-steps accumulated into fp32 main gradients (bit
    for bit against the oracle), then the boundary step over the fp32 main
    gradients (the 18-byte ledger layout) against the oracle's step."""
    shapes = [(3000,), (129,), (40000,), (1,), (9000,)]
    W = 2
    pr = Pair(shapes, W, 2, 100_000, wl.F32, wl.BF16, comm, index=130)
    mask = pr.L.real_mask()
    main_dev = [torch.zeros(pr.np, dtype=torch.float32, device="cuda") for _ in range(W)]
    main_np = [np.zeros(pr.np, np.float32) for _ in range(W)]
    stream = torch.cuda.current_stream().cuda_stream
    for k in range(3):
        micro = [wl.flat_grads(pr.z.offsets, pr.numel, pr.np, 1e-3, wl.grad_seed(130, r, k),
                               micro_dtype) for r in range(W)]
        micro_dev = [m.cuda() for m in micro]
        abi.zero_accumulate(pr.z.handle, [m.data_ptr() for m in micro_dev], micro_dtype,
                            [m.data_ptr() for m in main_dev], k == 0, stream)
        for r in range(W):
            oracle.accumulate(to_np(micro[r]), micro_dtype, main_np[r], k == 0, mask)
    torch.cuda.synchronize()
    real = mask.astype(bool)
    for r in range(W):
        assert np.array_equal(to_np(main_dev[r])[real], main_np[r][real])
    st, info, gc = pr.step([torch.from_numpy(m) for m in main_np], Hparams(), dev=main_dev)
    pr.check(st, info, gc)


def _pm_from_shards(L, numel, shards):
    flat = np.zeros(L.np_total, np.float32)
    flat[L.flat_of_shard()] = shards
    return np.concatenate([flat[off:off + n] for off, n in zip(L.param_offset, numel)])


def _shards_from_pm(L, numel, pm):
    flat = np.zeros(L.np_total, np.float32)
    at = 0
    for off, n in zip(L.param_offset, numel):
        flat[off:off + n] = pm[at:at + n]
        at += n
    return flat[L.flat_of_shard()].copy()


def test_checkpoint_reshard_w4_to_w2():
    """Train 2 steps with W=4 / ZeRO-2 / 80 KB buckets, export the fp32 state in
    parameter-major order plus the scaler, import it into W=2 / ZeRO-1 / 1 MB
    buckets, and continue: the imported state is bit-identical per parameter
    and the next step matches the oracle continued from its own state."""
    shapes = wl.qwen3_0_6b_shapes(vocab=1000, hidden=128, layers=2, q_dim=256, kv_dim=128,
                                  ffn=384, head_dim=32)
    numel = wl.numels(shapes)
    n = sum(numel)
    stream = torch.cuda.current_stream().cuda_stream
    a = Pair(shapes, 4, 2, 80_000, wl.F16, wl.F16, init_scale=1024.0, dynamic=True,
             growth_interval=3, index=140)
    for step in range(2):
        st, info, gc = a.step(a.grads(step, 1e-3), Hparams())
        a.check(st, info, gc)
    pm = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(3)]
    abi.zero_state_export_params(a.z.handle, *[t.data_ptr() for t in pm], stream)
    saved = abi.zero_loss_scale_state(a.z.handle, stream)
    # the export is the GPU's own state, reordered
    for t, shard_t in zip(pm, (a.z.master, a.z.m, a.z.v)):
        assert np.array_equal(to_np(t), _pm_from_shards(a.L, numel, to_np(shard_t)[:a.np]))

    b = Pair(shapes, 2, 1, 1_000_000, wl.F16, wl.F16, init_scale=1.0, dynamic=True,
             growth_interval=3, index=141)
    abi.zero_state_import_params(b.z.handle, *[t.data_ptr() for t in pm], stream)
    abi.zero_scaler_restore(b.z.handle, saved, stream)
    torch.cuda.synchronize()
    pm_b = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(3)]
    abi.zero_state_export_params(b.z.handle, *[t.data_ptr() for t in pm_b], stream)
    torch.cuda.synchronize()
    for x, y in zip(pm, pm_b):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    for p in range(len(shapes)):
        assert torch.equal(a.z.param_view(a.z.params_flat, p).view(torch.int16),
                           b.z.param_view(b.z.params_flat, p).view(torch.int16))
    st_b = b.z.scaler_state()
    assert (st_b["scale"], st_b["counter"], st_b["t"]) == (saved.scale, saved.counter, saved.t)

    # the oracle side goes through the same reshard, from the oracle's own state
    o_pm = [_pm_from_shards(a.L, numel, x) for x in (a.o_master, a.o_m, a.o_v)]
    b.o_master, b.o_m, b.o_v = [_shards_from_pm(b.L, numel, x) for x in o_pm]
    b.hist = [_shards_from_pm(b.L, numel, _pm_from_shards(a.L, numel, h)) for h in a.hist]
    flat_master = np.zeros(b.np, np.float32)
    flat_master[b.perm] = b.o_master
    b.o_params = oracle.encode(flat_master, wl.F16)
    b.o_params[~b.mask_flat] = 0
    b.o_scaler = oracle.Scaler(scale=a.o_scaler.scale, counter=a.o_scaler.counter, t=a.o_scaler.t,
                               dynamic=True, growth_interval=3)
    st, info, gc = b.step(b.grads(5, 1e-3), Hparams())
    b.check(st, info, gc)


def test_zero3_sharded_params_and_bucket_gather_with_prefetch():
    """Stage 3: the cast-out parameters stay in rank-major shards; all-gathering
    every bucket (the next one prefetched on a second stream while the
    current one is "in use") rebuilds exactly the flat parameters the oracle
    computes, step after step."""
    shapes = wl.qwen3_0_6b_shapes(vocab=1000, hidden=128, layers=2, q_dim=256, kv_dim=128,
                                  ffn=384, head_dim=32)
    pr = Pair(shapes, 4, 3, 120_000, wl.BF16, wl.BF16, index=150)
    info_q = abi.zero_layout_query(pr.z.handle)
    assert info_q.ledger_bytes_per_param == pytest.approx(16.0 / 4)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    gathered = torch.zeros(pr.np, dtype=torch.bfloat16, device="cuda")
    n_b = info_q.n_buckets
    assert n_b >= 3
    for step in range(2):
        st, info, gc = pr.step(pr.grads(step, 1e-3), Hparams())
        pr.check(st, info, gc)
        gathered.zero_()
        ready = [torch.cuda.Event() for _ in range(n_b)]
        abi.zero_gather_bucket(pr.z.handle, 0, gathered.data_ptr(), main.cuda_stream)
        ready[0].record(main)
        side.wait_stream(main)
        for b in range(n_b):
            if b + 1 < n_b:  # prefetch the next bucket on the side stream
                abi.zero_gather_bucket(pr.z.handle, b + 1, gathered.data_ptr(), side.cuda_stream)
                ready[b + 1].record(side)
            main.wait_event(ready[b])
            # bucket b is in use here (a forward would read it on `main`)
        torch.cuda.synchronize()
        got = to_np(gathered)
        assert _gather_matches_shards(pr, got)  # bit for bit; pr.check compared with the oracle
        assert np.all(got[~pr.mask_flat] == 0)
    with pytest.raises(ZeroError) as e:
        abi.zero_gather_bucket(pr.z.handle, n_b, gathered.data_ptr(), main.cuda_stream)
    assert e.value.code == abi.ZERO_ERR_INVALID


def _gather_matches_shards(pr, got):
    """The gathered params equal the GPU's own shards put back in flat order
    (those were checked against the oracle's parameters by pr.check)."""
    flat = np.zeros(pr.np, np.uint16)
    flat[pr.perm] = to_np(pr.z.params_flat)[:pr.np]
    return np.array_equal(got[pr.mask_flat], flat[pr.mask_flat])
