"""The sharded step on the GPU: R ranks of one job as threads of one process.

Each thread is one rank: its own layout made rank r's with
zero_dist_set_rank, its own shard buffers, and the library's kernels for the
local steps (ShardedZeroStep with LibraryShard). The collectives are carried
out on the host between the ranks' kernels (ThreadComm): every rank
synchronises its GPU work, the ranks meet at a barrier, and each takes its
result from all ranks' snapshots -- the sum in rank order in fp32, rounded
once to the buffer's dtype (the reading the oracle takes of the
reduce-scatter), fp64 for the norm pair. No kernel waits for another rank's
kernel: the only waits are host barriers with a timeout.

Every rank's master/m/v shard, parameters and scaler are compared with the
oracle's partitioned step (orc_zero_step) on all ranks' gradients, at the
tolerances of the other parity tests.
"""
import concurrent.futures
import threading

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _parity import to_np
from _util import params_close, rel_err, scaled_err
from mixed_precision_gb300.engine import Hparams
from mixed_precision_gb300.sharded import ShardedZeroStep

pytestmark = pytest.mark.gpu


class _Shared:
    def __init__(self, world):
        self.world = world
        self.slots = [None] * world
        self.barrier = threading.Barrier(world, timeout=120)


class ThreadComm:
    """The three collectives among R threads of one process (see above)."""

    def __init__(self, shared: _Shared, rank: int):
        self.shared, self.rank, self.world = shared, rank, shared.world

    def _gather(self, t):
        torch.cuda.synchronize()
        self.shared.slots[self.rank] = t.clone()
        self.shared.barrier.wait()
        snaps = list(self.shared.slots)
        self.shared.barrier.wait()  # every rank holds the snapshots before any slot changes
        return snaps

    @staticmethod
    def _sum(parts):
        dt = parts[0].dtype
        acc_t = (torch.int64 if not dt.is_floating_point else
                 torch.float64 if dt == torch.float64 else torch.float32)
        acc = parts[0].to(acc_t)
        for x in parts[1:]:
            acc = acc + x.to(acc_t)
        return acc.to(dt)

    def reduce_scatter(self, out, inp):
        snaps = self._gather(inp)
        n = out.numel()
        out.copy_(self._sum([s[self.rank * n:(self.rank + 1) * n] for s in snaps]))
        torch.cuda.synchronize()

    def all_reduce(self, t):
        t.copy_(self._sum(self._gather(t)))
        torch.cuda.synchronize()

    def all_gather(self, out, inp):
        out.copy_(torch.cat(self._gather(inp)))
        torch.cuda.synchronize()

    class _Done:
        @staticmethod
        def wait():
            pass

    def all_gather_async(self, out, inp):
        """all_gather, complete when it returns: the step then takes its
        bucket-by-bucket path (zero_dist_update_buckets)."""
        self.all_gather(out, inp)
        return self._Done


SHAPES = [(96, 40), (7,), (300, 33), (1,), (64, 64), (1000,), (0,), (129, 3), (8200,)]


def _run_rank(rank, shared, stage, gdt, bucket, steps, hp, cdt=-1):
    torch.cuda.set_device(0)
    pdt = wl.F16 if gdt == wl.F16 else wl.BF16
    dynamic = gdt == wl.F16
    scale0 = 2.0 ** 10 if dynamic else 1.0
    z = ShardedZeroStep(SHAPES, stage, bucket, gdt, pdt, comm=ThreadComm(shared, rank),
                        comm_dtype=cdt)
    numel = wl.numels(SHAPES)
    master0 = wl.master_init(z.offsets, numel, z.np, 0.02, wl.master_seed(50)).cuda()
    z.init(master0, init_scale=scale0, dynamic=dynamic, growth_interval=3)
    out = []
    for step in range(steps):
        g = _grads(z, numel, shared.world, step, gdt, scale0)[rank].cuda()
        z.step(g, hp)
        torch.cuda.synchronize()
        out.append((z.scaler_state(), [to_np(t) for t in (z.local.master, z.local.m, z.local.v)],
                    to_np(z.local.params)))
    gathered = []
    if stage == 3:  # every bucket's parameters, all-gathered from the ranks' slices
        for b, bk in enumerate(z.buckets):
            buf = torch.empty(bk.length, dtype=z.local.params.dtype, device="cuda")
            z.gather_bucket(b, buf)
            gathered.append((bk.start, to_np(buf)))
    z.close()
    return out, gathered


def _grads(z, numel, world, step, gdt, scale0):
    g = [wl.flat_grads(z.offsets, numel, z.np, 1e-3 * scale0, wl.grad_seed(51, w, step), gdt)
         for w in range(world)]
    if step == 2:  # one non-finite value on the last rank: every rank skips
        g[world - 1][z.offsets[2] + 5] = float("inf")
    return g


@pytest.mark.parametrize("world,stage,gdt,cdt", [(2, 2, wl.BF16, -1), (3, 2, wl.F16, -1),
                                                 (4, 1, wl.BF16, -1), (2, 3, wl.F16, -1),
                                                 (4, 3, wl.BF16, -1), (1, 2, wl.BF16, -1),
                                                 (3, 2, wl.BF16, wl.F32), (4, 1, wl.F16, wl.F32)])
def test_sharded_ranks_match_oracle(world, stage, gdt, cdt):
    """cdt F32: fp32 collectives of the widened 16-bit gradients."""
    bucket, steps = 24_000, 5
    hp = Hparams(max_grad_norm=0.05 if world == 4 else 1.0)  # clipping active at W = 4
    shared = _Shared(world)
    with concurrent.futures.ThreadPoolExecutor(world) as ex:
        futs = [ex.submit(_run_rank, r, shared, stage, gdt, bucket, steps, hp, cdt)
                for r in range(world)]
        results = [f.result(timeout=600) for f in futs]
    per_rank = [r[0] for r in results]

    # the oracle's partitioned step on every rank's gradients
    pdt = wl.F16 if gdt == wl.F16 else wl.BF16
    dynamic = gdt == wl.F16
    scale0 = 2.0 ** 10 if dynamic else 1.0
    numel = wl.numels(SHAPES)
    L = oracle.layout(numel, world, bucket, wl.ELEM_BYTES[gdt])
    n, npad = L.shard_total, L.np_total
    perm = L.flat_of_shard()
    real_shard = L.real_mask().astype(bool)[perm]
    offs = [int(o) for o in L.param_offset]
    master0 = wl.master_init(offs, numel, npad, 0.02, wl.master_seed(50)).numpy()
    ms, mm, vv = master0[perm].copy(), np.zeros(npad, np.float32), np.zeros(npad, np.float32)
    hist = [np.abs(ms), np.zeros(npad, np.float32), np.zeros(npad, np.float32)]
    params = oracle.encode(master0, pdt)
    params[~L.real_mask().astype(bool)] = 0
    sc = oracle.Scaler(scale=scale0, dynamic=dynamic, growth_interval=3)
    o_hp = oracle.Hparams(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.max_grad_norm,
                          hp.grad_divisor)

    class _Z:  # what _grads needs of a step object
        offsets = offs
        np = npad

    for step in range(steps):
        g = [to_np(x) for x in _grads(_Z, numel, world, step, gdt, scale0)]
        c_eff = gdt if cdt < 0 else cdt
        outs = [np.zeros(npad, oracle.storage_dtype(c_eff)) for _ in range(world)] if stage == 1 else None
        info = oracle.zero_step(numel, world, min(stage, 2), bucket, gdt, c_eff, pdt, g, ms, mm, vv,
                                params, o_hp, sc, allreduce_out=outs)
        for h, x in zip(hist, (ms, mm, vv)):
            np.maximum(h, np.abs(x), out=h)
        for r in range(world):
            st, state, p = per_rank[r][step]
            assert (st["scale"], st["counter"], st["t"]) == (sc.scale, sc.counter, sc.t), (r, step)
            assert st["overflow"] == info.overflow and st["skipped"] == info.skipped
            if np.isfinite(info.grad_norm):
                assert abs(st["grad_norm"] - info.grad_norm) <= 1e-6 * info.grad_norm
            sl = slice(r * n, (r + 1) * n)
            real = real_shard[sl]
            for got, ref, h in zip(state, (ms, mm, vv), hist):
                got, ref, h = got[:n][real], ref[sl][real], h[sl][real]
                assert scaled_err(got, ref, h).max(initial=0.0) <= 1e-5, (r, step)
                bad = rel_err(got, ref) > 1e-5
                assert np.all(np.abs(ref[bad]) < 0.1 * h[bad])
            bound = 1e-5 * hist[0][sl].astype(np.float64)
            if stage == 3:
                exp = params[perm[sl]]
                ok = params_close(p[:n], exp, oracle.decode(exp, pdt), oracle.decode(p[:n], pdt),
                                  bound, pdt == wl.BF16)
                assert ok[real].all(), (r, step)
            else:
                b_flat = np.zeros(npad)
                b_flat[perm] = 1e-5 * hist[0].astype(np.float64)
                ok = params_close(p[:npad], params, oracle.decode(params, pdt),
                                  oracle.decode(p[:npad], pdt), b_flat, pdt == wl.BF16)
                assert ok[L.real_mask().astype(bool)].all(), (r, step)
                assert np.all(p[:npad][~L.real_mask().astype(bool)] == 0)
    if stage == 3:  # the gathered buckets: the flat parameters, on every rank alike
        b_flat = np.zeros(npad)
        b_flat[perm] = 1e-5 * hist[0].astype(np.float64)
        real_flat = L.real_mask().astype(bool)
        for r in range(world):
            assert len(results[r][1]) == len(L.bucket_start)
            for (b0, got), bl in zip(results[r][1], L.bucket_len):
                sl = slice(b0, b0 + int(bl))
                ok = params_close(got, params[sl], oracle.decode(params[sl], pdt),
                                  oracle.decode(got, pdt), b_flat[sl], pdt == wl.BF16)
                assert ok[real_flat[sl]].all(), (r, b0)
                assert np.array_equal(got, results[0][1][[x[0] for x in results[0][1]].index(b0)][1])


def test_sharded_layout_refuses_single_process_steps():
    """A layout that holds one rank's shard refuses the entry points that
    step all W ranks in one process, and the sharded calls need a sharded
    layout."""
    from mixed_precision_gb300 import ZeroError
    from mixed_precision_gb300 import _abi as abi
    from mixed_precision_gb300.engine import ZeroStep

    shared = _Shared(1)
    z = ShardedZeroStep(SHAPES, 2, 24_000, wl.BF16, wl.BF16, comm=ThreadComm(shared, 0))
    master0 = torch.zeros(z.np, dtype=torch.float32, device="cuda")
    z.init(master0)
    g = torch.zeros(z.np, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    with pytest.raises(ZeroError) as e:
        abi.zero_step(z.handle, [g.data_ptr()], None, Hparams().c(), stream)
    assert e.value.code == abi.ZERO_ERR_STATE
    with pytest.raises(ZeroError) as e:  # stages 2/3 read the bound scratch
        abi.zero_dist_update(z.handle, g.data_ptr(), stream)
    assert e.value.code == abi.ZERO_ERR_INVALID
    nb = len(z.buckets)
    for first, count in ((-1, 1), (0, nb + 1), (nb, 1), (1, -1)):  # outside the layout's buckets
        with pytest.raises(ZeroError) as e:
            abi.zero_dist_update_buckets(z.handle, 0, first, count, stream)
        assert e.value.code == abi.ZERO_ERR_INVALID, (first, count)
    abi.zero_dist_update_buckets(z.handle, 0, nb, 0, stream)  # an empty range enqueues nothing
    z.close()
    plain = ZeroStep(SHAPES, 1, 2, 24_000, wl.BF16, wl.BF16)
    plain.allocate()
    plain.init(master0)
    pair = torch.zeros(2, dtype=torch.float64, device="cuda")
    with pytest.raises(ZeroError) as e:
        abi.zero_dist_shard_norm(plain.handle, 0, pair.data_ptr(), stream)
    assert e.value.code == abi.ZERO_ERR_STATE
    plain.close()


def _run_ranks(world, fn):
    shared = _Shared(world)
    with concurrent.futures.ThreadPoolExecutor(world) as ex:
        futs = [ex.submit(fn, r, ThreadComm(shared, r)) for r in range(world)]
        return [f.result(timeout=600) for f in futs]


def test_checkpoint_across_gpu_counts():
    """A 2-rank job (bucket 24 KB) steps, then assembles a parameter-major
    checkpoint: each rank exports its elements, the all-reduce of the 32-bit
    patterns joins them. A 4-rank job with 60 KB buckets imports it (and the
    scaler); its own export is the same checkpoint bit for bit, and its next
    step matches the oracle restarted from that state on its layout."""
    gdt = pdt = wl.BF16
    numel = wl.numels(SHAPES)
    hp = Hparams()

    def job_a(rank, comm):
        torch.cuda.set_device(0)
        z = ShardedZeroStep(SHAPES, 2, 24_000, gdt, pdt, comm=comm)
        z.init(wl.master_init(z.offsets, numel, z.np, 0.02, wl.master_seed(52)).cuda())
        for step in range(3):
            g = wl.flat_grads(z.offsets, numel, z.np, 1e-3, wl.grad_seed(53, rank, step), gdt).cuda()
            z.step(g, hp)
        ex = z.export_params()
        st = z.scaler_state()
        torch.cuda.synchronize()
        z.close()
        return [t.clone() for t in ex], st

    res_a = _run_ranks(2, job_a)
    ex, st = res_a[0]
    for other, _ in res_a[1:]:  # every rank holds the same whole checkpoint
        for x, y in zip(ex, other):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert st["t"] == 3

    def job_b(rank, comm):
        torch.cuda.set_device(0)
        z = ShardedZeroStep(SHAPES, 2, 60_000, gdt, pdt, comm=comm)
        z.init(torch.zeros(max(z.np, 8), device="cuda"))
        z.import_params(*ex, scaler=st)
        again = [t.clone() for t in z.export_params()]
        g = wl.flat_grads(z.offsets, numel, z.np, 1e-3, wl.grad_seed(53, rank, 3), gdt).cuda()
        z.step(g, hp)
        torch.cuda.synchronize()
        out = (again, z.scaler_state(), [to_np(t) for t in (z.local.master, z.local.m, z.local.v)],
               to_np(z.local.params))
        z.close()
        return out

    res_b = _run_ranks(4, job_b)
    for again, _, _, _ in res_b:
        for x, y in zip(ex, again):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))

    # the oracle restarted from the checkpoint on the 4-rank layout
    L = oracle.layout(numel, 4, 60_000, 2)
    n, npad = L.shard_total, L.np_total
    perm = L.flat_of_shard()
    flats = []
    for t in ex:
        pm, flat, at = t.cpu().numpy(), np.zeros(npad, np.float32), 0
        for o, k in zip(L.param_offset, numel):
            flat[o:o + k] = pm[at:at + k]
            at += k
        flats.append(flat)
    ms, mm, vv = (f[perm].copy() for f in flats)
    hist = [np.maximum(np.abs(ms), 0), np.abs(mm), np.abs(vv)]
    params = oracle.encode(flats[0], pdt)
    params[~L.real_mask().astype(bool)] = 0
    sc = oracle.Scaler(scale=st["scale"], counter=st["counter"], t=st["t"])
    offs = [int(o) for o in L.param_offset]
    g = [to_np(wl.flat_grads(offs, numel, npad, 1e-3, wl.grad_seed(53, r, 3), gdt)) for r in range(4)]
    oracle.zero_step(numel, 4, 2, 60_000, gdt, gdt, pdt, g, ms, mm, vv, params, oracle.Hparams(), sc)
    for h, x in zip(hist, (ms, mm, vv)):
        np.maximum(h, np.abs(x), out=h)
    real_shard = L.real_mask().astype(bool)[perm]
    for r, (_, st_b, state, p) in enumerate(res_b):
        assert (st_b["scale"], st_b["counter"], st_b["t"]) == (sc.scale, sc.counter, sc.t)
        sl = slice(r * n, (r + 1) * n)
        real = real_shard[sl]
        for got, ref, h in zip(state, (ms, mm, vv), hist):
            assert scaled_err(got[:n][real], ref[sl][real], h[sl][real]).max(initial=0.0) <= 1e-5
        b_flat = np.zeros(npad)
        b_flat[perm] = 1e-5 * hist[0].astype(np.float64)
        ok = params_close(p[:npad], params, oracle.decode(params, pdt), oracle.decode(p[:npad], pdt),
                          b_flat, True)
        assert ok[L.real_mask().astype(bool)].all()


def test_fullsize_two_ranks_equal_the_single_process_step():
    """The full Qwen3-0.6B-shaped list (596M parameters), W = 2, ZeRO-2,
    bf16: two sharded ranks (threads, host-barrier collectives) against the
    library's single-process step on the same gradients. With clipping off
    the clip coefficient is exactly 1 on both sides and a two-term sum has
    one order, so every rank's master/m/v slice and the gathered parameters
    equal the single-process step's bit for bit over two steps (the second
    with every element's moments non-zero); the norms agree within 1e-6
    (their partial sums are grouped differently)."""
    from mixed_precision_gb300 import _abi as abi
    from mixed_precision_gb300.engine import ZeroStep

    w = wl.workload("qwen3_0.6b_bf16_w2", max_grad_norm=0.0)
    numel = wl.numels(w.shapes)
    hp = Hparams(max_grad_norm=0.0)
    ref = ZeroStep(w.shapes, 2, 2, w.bucket_bytes, w.grad_dtype, w.param_dtype)
    ref.allocate()
    m0 = wl.master_init(ref.offsets, numel, ref.np, w.master_sigma, wl.master_seed(w.index),
                        device="cuda")
    ref.init(m0)
    grads = [[wl.flat_grads(ref.offsets, numel, ref.np, w.grad_sigma, wl.grad_seed(w.index, r, s),
                            w.grad_dtype, device="cuda") for r in range(2)] for s in range(2)]
    for s in range(2):
        ref.step(grads[s], hp)
    torch.cuda.synchronize()
    ref_st = ref.scaler_state()

    def rank_job(rank, comm):
        torch.cuda.set_device(0)
        z = ShardedZeroStep(w.shapes, 2, w.bucket_bytes, w.grad_dtype, w.param_dtype, comm=comm)
        z.init(m0)
        for s in range(2):
            z.step(grads[s][rank].clone(), hp)
        torch.cuda.synchronize()
        n = z.shard_elems
        lo = rank * n
        same = [torch.equal(mine[:n].view(torch.int32), full[lo:lo + n].view(torch.int32))
                for mine, full in zip((z.local.master, z.local.m, z.local.v),
                                      (ref.master, ref.m, ref.v))]
        params_same = torch.equal(z.local.params[:z.np].view(torch.int16),
                                  ref.params_flat[:ref.np].view(torch.int16))
        st = z.scaler_state()
        z.close()
        return same, params_same, st

    for same, params_same, st in _run_ranks(2, rank_job):
        assert all(same) and params_same
        assert st["t"] == ref_st["t"] == 2 and st["overflow"] == 0
        assert abs(st["grad_norm"] - ref_st["grad_norm"]) <= 1e-6 * ref_st["grad_norm"]
    assert abi.zero_layout_query(ref.handle).n_real == 596_049_920
    ref.close()
