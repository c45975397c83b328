"""The sharded step's schedule across processes, on CPU (gloo, world size 2).

ShardedZeroStep (mixed_precision_gb300/sharded.py) runs one rank per process:
per bucket a reduce-scatter (stages 2/3) or an all-reduce (stage 1), this
rank's share of the norm and overflow flag, one all-reduce of that pair, the
finalize, the update of this rank's shard, and the per-bucket all-gather of
the parameters. Here the local steps are the oracle's (tests/_oracle_shard.py)
and the collectives are gloo's, so the test checks the schedule itself: which
slices travel, in which buffers they land, and that the global decisions come
out the same on every rank. Each rank compares its shard of master/m/v, its
parameter buffer and its scaler with the oracle's own partitioned step
(orc_zero_step) run on every rank's gradients, bit for bit. At W = 2 a
two-term sum has one order, so the collectives' sums are the oracle's (leetllm
"Deep dive: Megatron", "Distributed optimizer": the reduce-scatter sums each
rank's slice; the all-gather rebuilds the parameter buffer). Then the ranks
assemble a parameter-major checkpoint (each exports its own elements, an
all-reduce of the 32-bit patterns joins them), which must equal the oracle's
state, and restart a job with another bucket size from it, which must keep
stepping like the oracle.
"""
import os
import socket
import traceback

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


SHAPES = [(96, 40), (7,), (300, 33), (1,), (64, 64), (1000,), (0,), (129, 3)]


def _worker(rank, world, port, stage, gdt, q, cdt=-1):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        import torch
        import torch.distributed as dist
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import oracle
        import workloads as wl
        from _oracle_shard import TORCH_DTYPE, OracleShard, bits
        from mixed_precision_gb300.engine import Hparams
        from mixed_precision_gb300.sharded import ShardedZeroStep

        pdt = wl.F16 if gdt == wl.F16 else wl.BF16
        dynamic = gdt == wl.F16
        scale0 = 2.0 ** 10 if dynamic else 1.0
        bucket = 24_000  # several buckets, parameters of several sizes in each
        z = ShardedZeroStep(SHAPES, stage, bucket, gdt, pdt, local=OracleShard, comm_dtype=cdt)
        cdt = z.comm_dtype
        numel = wl.numels(SHAPES)
        L = oracle.layout(numel, world, bucket, wl.ELEM_BYTES[gdt])
        assert z.np == L.np_total and len(z.buckets) == len(L.bucket_start) > 1
        assert z.offsets == [int(o) for o in L.param_offset]
        master0 = wl.master_init(z.offsets, numel, z.np, 0.02, wl.master_seed(40))
        z.init(master0, init_scale=scale0, dynamic=dynamic, growth_interval=3)

        n = z.shard_elems
        ref_master = bits(master0)[L.flat_of_shard()].copy()
        ref_m, ref_v = np.zeros_like(ref_master), np.zeros_like(ref_master)
        ref_params = oracle.encode(bits(master0), pdt)
        ref_params[~L.real_mask().astype(bool)] = 0
        sc = oracle.Scaler(scale=scale0, dynamic=dynamic, growth_interval=3)
        hp = Hparams(max_grad_norm=1.0 if stage != 3 else 0.05)
        o_hp = oracle.Hparams(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.max_grad_norm,
                              hp.grad_divisor)
        shard_flat = L.flat_of_shard()[rank * n:(rank + 1) * n]
        for step in range(6):
            sigma = 1e-3 * (scale0 if dynamic else 1.0)
            g_all = [wl.flat_grads(z.offsets, numel, z.np, sigma, wl.grad_seed(41, w, step), gdt)
                     for w in range(world)]
            if step == 2:  # one non-finite value on one rank: every rank skips
                g_all[1][z.offsets[2] + 5] = float("inf")
            outs = ([np.zeros(z.np, oracle.storage_dtype(cdt)) for _ in range(world)]
                    if stage == 1 else None)
            info = oracle.zero_step(numel, world, min(stage, 2), bucket, gdt, cdt, pdt,
                                    [bits(g) for g in g_all], ref_master, ref_m, ref_v, ref_params,
                                    o_hp, sc, allreduce_out=outs)
            mine = g_all[rank].clone()
            z.step(mine, hp)
            st = z.scaler_state()
            assert (st["scale"], st["counter"], st["t"]) == (sc.scale, sc.counter, sc.t), (step, st)
            assert st["skipped"] == info.skipped == (1 if step == 2 else 0)
            for got, ref in ((z.local.master, ref_master), (z.local.m, ref_m), (z.local.v, ref_v)):
                assert np.array_equal(bits(got)[:n].view(np.uint32),
                                      ref[rank * n:(rank + 1) * n].view(np.uint32)), step
            p = bits(z.local.params)
            if stage == 3:
                assert np.array_equal(p[:n], ref_params[shard_flat]), step
            else:
                assert np.array_equal(p[:z.np], ref_params), step

        if stage == 3:  # every bucket's parameters, all-gathered from the ranks' slices
            for b, (b0, bl) in enumerate(zip(L.bucket_start, L.bucket_len)):
                out = torch.empty(int(bl), dtype=TORCH_DTYPE[pdt])
                z.gather_bucket(b, out)
                assert np.array_equal(bits(out), ref_params[int(b0):int(b0) + int(bl)]), b

        # A checkpoint independent of W: every rank exports its elements, the
        # all-reduce of their bit patterns assembles the whole buffer, equal to
        # the oracle's state in parameter-major order.
        def shards_to_pm(x, lay):
            flat = np.zeros(lay.np_total, np.float32)
            flat[lay.flat_of_shard()] = x
            return np.concatenate([flat[o:o + k] for o, k in zip(lay.param_offset, numel)])

        def pm_to_shards(pm, lay):
            flat = np.zeros(lay.np_total, np.float32)
            at = 0
            for o, k in zip(lay.param_offset, numel):
                flat[o:o + k] = pm[at:at + k]
                at += k
            return flat[lay.flat_of_shard()].copy(), flat

        ex = z.export_params()
        for got, ref in zip(ex, (ref_master, ref_m, ref_v)):
            assert np.array_equal(bits(got).view(np.uint32), shards_to_pm(ref, L).view(np.uint32))
        # ... and restarts a job with another bucket size, which then steps
        # like the oracle restarted from the same state
        bucket2 = 50_000
        z2 = ShardedZeroStep(SHAPES, stage, bucket2, gdt, pdt, local=OracleShard, comm_dtype=cdt)
        z2.init(torch.zeros(z2.np), init_scale=scale0, dynamic=dynamic, growth_interval=3)
        z2.import_params(*ex, scaler=z.scaler_state())
        L2 = oracle.layout(numel, world, bucket2, wl.ELEM_BYTES[gdt])
        n2 = z2.shard_elems
        ref_master, mflat = pm_to_shards(bits(ex[0]), L2)
        ref_m, _ = pm_to_shards(bits(ex[1]), L2)
        ref_v, _ = pm_to_shards(bits(ex[2]), L2)
        ref_params = oracle.encode(mflat, pdt)
        ref_params[~L2.real_mask().astype(bool)] = 0
        shard_flat2 = L2.flat_of_shard()[rank * n2:(rank + 1) * n2]
        for step in range(6, 8):
            g_all = [wl.flat_grads(z2.offsets, numel, z2.np, 1e-3 * scale0, wl.grad_seed(41, w, step),
                                   gdt) for w in range(world)]
            outs = ([np.zeros(z2.np, oracle.storage_dtype(cdt)) for _ in range(world)]
                    if stage == 1 else None)
            oracle.zero_step(numel, world, min(stage, 2), bucket2, gdt, cdt, pdt,
                             [bits(g) for g in g_all], ref_master, ref_m, ref_v, ref_params, o_hp, sc,
                             allreduce_out=outs)
            z2.step(g_all[rank].clone(), hp)
            st = z2.scaler_state()
            assert (st["scale"], st["counter"], st["t"]) == (sc.scale, sc.counter, sc.t), (step, st)
            for got, ref in ((z2.local.master, ref_master), (z2.local.m, ref_m), (z2.local.v, ref_v)):
                assert np.array_equal(bits(got)[:n2].view(np.uint32),
                                      ref[rank * n2:(rank + 1) * n2].view(np.uint32)), step
            p = bits(z2.local.params)
            if stage == 3:
                assert np.array_equal(p[:n2], ref_params[shard_flat2]), step
            else:
                assert np.array_equal(p[:z2.np], ref_params), step
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception:
        q.put((rank, traceback.format_exc()))


@pytest.mark.parametrize("stage,gdt,cdt", [(2, 2, -1), (2, 1, -1), (1, 2, -1), (3, 2, -1), (3, 1, -1),
                                           (2, 2, 0), (1, 1, 0)])
def test_sharded_schedule_matches_oracle_two_ranks(stage, gdt, cdt):
    """cdt 0: fp32 collectives of 16-bit gradients (each rank widens its
    gradients, exactly, and the reduce-scatter or all-reduce runs in fp32)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, stage, gdt, q, cdt)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        r, msg = q.get(timeout=300)
        res[r] = msg
    for p in procs:
        p.join(timeout=60)
    for r in range(2):
        assert res[r] == "ok", f"rank {r}:\n{res[r]}"
    assert all(p.exitcode == 0 for p in procs)


def _worker_leaves(rank, world, port, q):
    """Both ranks step once; rank 1 then leaves between steps (its process
    ends, nothing of it in flight). Rank 0's next step must end with an
    error from its first collective, within the process group's timeout,
    not hang."""
    import time
    from datetime import timedelta
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        import torch.distributed as dist
        dist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=10))
        import workloads as wl
        from _oracle_shard import OracleShard
        from mixed_precision_gb300.engine import Hparams
        from mixed_precision_gb300.sharded import ShardedZeroStep

        z = ShardedZeroStep(SHAPES, 2, 24_000, wl.BF16, wl.BF16, local=OracleShard)
        numel = wl.numels(SHAPES)
        z.init(wl.master_init(z.offsets, numel, z.np, 0.02, wl.master_seed(42)))
        g = wl.flat_grads(z.offsets, numel, z.np, 1e-3, wl.grad_seed(43, rank), wl.BF16)
        z.step(g.clone(), Hparams())
        if rank == 1:
            q.put((rank, "left"))
            q.close()
            q.join_thread()  # the message is sent before the process ends
            os._exit(0)  # leaves between steps, no collective in flight
        t0 = time.monotonic()
        try:
            z.step(g.clone(), Hparams())
            q.put((rank, "no error"))
        except Exception as e:  # the collective reports the missing peer
            q.put((rank, f"error after {time.monotonic() - t0:.1f} s: {type(e).__name__}"))
        q.close()
        q.join_thread()
        os._exit(0)
    except Exception:
        q.put((rank, traceback.format_exc()))


def test_rank_leaving_ends_the_next_collective_with_an_error():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker_leaves, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
    assert res[1] == "left", res
    assert res[0].startswith("error after"), res
    assert float(res[0].split()[2]) < 30.0, res
