"""Benchmark of the ZeRO-1/2 gradient-and-optimizer step on GB300.

One "step" is one pass of the whole hot path over one batch of synthetic
gradients: the W-way reduce with overflow/norm partials, the finalize kernel
(norm, clip, loss-scale state machine) and the fused unscale/clip/AdamW/
cast-out kernel. Default workload: the Qwen3-0.6B-shaped parameter list
(596,049,920 elements, 310 tensors), W = 2 simulated ranks, ZeRO-2, bf16
gradients N(0, 1e-4), bucket 500 MB, clip 1.0. Inputs (2.4 GB of gradients,
7.2 GB of fp32 state) are larger than the 129 MB L2, so no flush is needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 (torchrun, one rank per GPU) runs N independent replicas of the same
workload (weak scaling: the simulated ranks already live inside each GPU).
Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ZeRO step params updated/s and achieved HBM GB/s (% of GB300 step roofline)"
DEFAULT_WORKLOAD = "qwen3_0.6b_bf16_w2"
L2_BYTES = 129 * 1000 * 1000
# DRAM bytes per real element of each dominant kernel, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum, one launch, one pass) on a
# profiling-sized slice of the workload, at the kernel's current grid; the
# bench line scales them by the workload's elements. Keyed by (kernel,
# workload); a workload without a capture of its kernel reports null.
NCU_TRAFFIC_PER_ELEM = {
    # update kernel, one block per tile (15,392 blocks), 8 Qwen3 layers,
    # 125,847,552 elements: (1.762588 + 1.701842) GB
    ("k_adamw_cast", "qwen3_0.6b_bf16_w2"): 27.529,
    # reduce kernel, W=2, 1,824 blocks, the same slice: (0.504079 + 0.214297) GB
    ("k_reduce_norm", "qwen3_0.6b_bf16_w2"): 5.708,
    # update kernel, one block per tile (28,680 blocks), 2 MoE layers,
    # 234,946,560 elements: (3.290513 + 3.229704) GB
    ("k_adamw_cast", "moe_3.9b_bf16_w4"): 27.752,
    # reduce kernel, W=4, 1,216 blocks, the same slice: (1.880805 + 0.448101) GB
    ("k_reduce_norm", "moe_3.9b_bf16_w4"): 9.912,
    # speculative single pass, W=2, 26 blocks per SM and resident block,
    # 8 Qwen3 layers: (2.014366 + 1.708428) GB
    ("k_spec_step", "qwen3_0.6b_bf16_w2"): 29.582,
    # speculative single pass, W=4, the same grid rule, 2 MoE layers:
    # (4.700327 + 3.243320) GB
    ("k_spec_step", "moe_3.9b_bf16_w4"): 33.810,
    # update kernel's per-tensor pointer instance, 2 MoE layers with each
    # rank's idle experts NULL: (3.051415 + 3.230056) GB
    ("k_adamw_cast_table", "moe_3.9b_bf16_w4"): 26.736,
    # the stage-1 single pass (all-reduce writes included), W=8, 2-byte
    # gradients, 8 Qwen3 layers: (3.524556 + 3.723003) GB
    ("k_spec_step_s1", "qwen3_0.6b_fp16_w8"): 57.590,
    # update kernel, one block per tile (19,763 blocks), the first 200 of the
    # 2000 ragged tensors, 160,922,893 elements: (2.254052 + 2.193213) GB
    ("k_adamw_cast", "ragged_2000"): 27.636,
    # fp16 W=8, 8 Qwen3 layers: the update (15,392 blocks), (1.762527 +
    # 1.701489) GB; the stage-1 reduce with its W all-reduce writes (1,216
    # blocks), (2.014353 + 1.962679) GB
    ("k_adamw_cast", "qwen3_0.6b_fp16_w8"): 27.526,
    ("k_reduce_norm_s1", "qwen3_0.6b_fp16_w8"): 31.602,
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=10,
                    help="end-to-end steps through the host-buffer entry point (0: skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--per-config-steps", type=int, default=20,
                    help="timed steps of each other named workload after the default line "
                         "(the MoE ~3.9B list; fp16 W=8 at stages 1 and 2); 0: skip")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--world", type=int, default=None, help="override the simulated world size")
    ap.add_argument("--bucket-bytes", type=int, default=None, help="override the bucket size")
    ap.add_argument("--stage", type=int, default=None, help="override the ZeRO stage (1, 2, 3)")
    ap.add_argument("--profile-range", action="store_true",
                    help="bracket the timed steps with cudaProfilerStart/Stop (for "
                         "nsys/ncu capture ranges on the CUDA profiler API)")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured into a CUDA graph and replayed (flat modes)")
    ap.add_argument("--clip", type=float, default=None,
                    help="override max_grad_norm (<= 0: no clipping)")
    ap.add_argument("--speculative", action="store_true",
                    help="time zero_step_speculative (single pass when clipping stays inactive)")
    ap.add_argument("--per-tensor-launch", action="store_true",
                    help="launch the step tensor by tensor (the hook-style baseline)")
    ap.add_argument("--tensors", action="store_true",
                    help="step from per-tensor gradient pointers (NULL for all-zero gradients)")
    ap.add_argument("--sharded", action="store_true",
                    help="one rank per GPU (torchrun, NCCL): the workload's world is the number "
                         "of GPUs, each GPU holds its own gradients and its shard of the state; "
                         "reduce-scatter, norm all-reduce and all-gather between the local "
                         "kernels (stages 2 and 3)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# Distributed plumbing (timing only: no collective touches the data path)
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """Largest value over all ranks (the slowest rank sets the job's time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: float, n_ranks: int, seconds: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest time."""
    return units_per_rank * n_ranks / seconds


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return self
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# Shared helpers
# ---------------------------------------------------------------------------

def hbm_peak():
    """(GB/s, source): the measured copy bandwidth, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def workload_of(args):
    """The named workload with the command line's overrides."""
    import workloads as wl
    over = {}
    if getattr(args, "world", None):
        over["world"] = args.world
    if getattr(args, "bucket_bytes", None):
        over["bucket_bytes"] = args.bucket_bytes
    if getattr(args, "stage", None):
        over["stage"] = args.stage
    if getattr(args, "clip", None) is not None:
        over["max_grad_norm"] = args.clip
    return wl.workload(args.workload, **over)


def config_of(w, scaling_note=None) -> dict:
    import workloads as wl
    cfg = {"workload": w.name, "n_params": w.n_real, "tensors": len(w.shapes),
           "world_simulated": w.world, "zero_stage": w.stage,
           "grad_dtype": wl.DTYPE_NAME[w.grad_dtype], "param_dtype": wl.DTYPE_NAME[w.param_dtype],
           "comm_dtype": wl.DTYPE_NAME[w.comm_dtype], "bucket_bytes": w.bucket_bytes,
           "clip": w.max_grad_norm, "grad_sigma": w.grad_sigma,
           "l2": "inputs larger than L2 (no flush)", "parallelism": "replicas"}
    if scaling_note:
        cfg["note"] = scaling_note
    return cfg


def sample_shapes(shapes, target_elems: int):
    """A bounded sample of a workload: its tensors in order, skipping any tensor
    larger than the target, until the target element count is reached."""
    import workloads as wl
    out, total = [], 0
    for s in shapes:
        n = wl.numels([s])[0]
        if n > target_elems:
            continue
        out.append(s)
        total += n
        if total >= target_elems:
            break
    return out, total


def _oracle_setup(w, target_elems: int):
    """Inputs and state for the host oracle's ZeRO step on a sample of the
    workload; returns (one step as a callable, sample elements, sample text)."""
    import numpy as np
    import torch

    import oracle
    import workloads as wl

    shapes, n_sample = sample_shapes(w.shapes, target_elems)
    numel = wl.numels(shapes)
    L = oracle.layout(numel, w.world, w.bucket_bytes, wl.ELEM_BYTES[w.grad_dtype])

    def bits(t):
        return t.numpy() if t.dtype == torch.float32 else t.view(torch.int16).numpy().view(np.uint16)

    grads = [bits(wl.flat_grads(L.param_offset, numel, L.np_total, w.grad_sigma,
                                wl.grad_seed(w.index, r), w.grad_dtype)) for r in range(w.world)]
    ms = bits(wl.master_init(L.param_offset, numel, L.np_total, w.master_sigma,
                             wl.master_seed(w.index)))[L.flat_of_shard()].copy()
    m, v = np.zeros_like(ms), np.zeros_like(ms)
    params = np.zeros(L.np_total, oracle.storage_dtype(w.param_dtype))
    outs = ([np.zeros(L.np_total, oracle.storage_dtype(w.comm_dtype)) for _ in range(w.world)]
            if w.stage == 1 else None)
    hp = oracle.Hparams(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_grad_norm, 0.0)
    sc = oracle.Scaler(scale=w.init_scale, dynamic=w.dynamic, growth_interval=w.growth_interval)

    def one():
        oracle.zero_step(numel, w.world, w.stage, w.bucket_bytes, w.grad_dtype, w.comm_dtype,
                         w.param_dtype, grads, ms, m, v, params, hp, sc, allreduce_out=outs)

    desc = (f"{len(shapes)} of the workload's {len(w.shapes)} tensors ({n_sample} elements, "
            f"tensors larger than {target_elems} skipped), W={w.world}, ZeRO-{w.stage}")
    return one, n_sample, desc


def time_oracle(w, target_elems: int, seconds: float, min_steps: int = 1, warmup: int = 0,
                steps: int | None = None):
    """Run the host oracle's ZeRO step on a sample of the workload.

    Returns (params per second, steps timed, sample elements, sample description).
    Single-threaded: the oracle is plain sequential host code.
    """
    one, n_sample, desc = _oracle_setup(w, target_elems)
    for _ in range(warmup):
        one()
    t0 = time.perf_counter()
    done = 0
    while True:
        one()
        done += 1
        el = time.perf_counter() - t0
        if steps is not None:
            if done >= steps:
                break
        elif done >= min_steps and el >= seconds:
            break
    el = time.perf_counter() - t0
    return n_sample * done / el, done, n_sample, f"{desc}, {done} full oracle steps"


def time_oracle_threads(w, target_elems: int, seconds: float, threads: int):
    """The same oracle step on all host cores: `threads` host threads each
    step their own copy of the sample (the oracle itself stays sequential;
    its ctypes calls release the interpreter lock). Returns (aggregate params
    per second, sample description)."""
    import concurrent.futures

    setups = [_oracle_setup(w, target_elems) for _ in range(threads)]
    n_sample, desc = setups[0][1], setups[0][2]
    for one, _, _ in setups:  # first touch of every copy's buffers
        one()

    def loop(one):
        done, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < seconds or done == 0:
            one()
            done += 1
        return done, time.perf_counter() - t0

    with concurrent.futures.ThreadPoolExecutor(threads) as ex:
        res = list(ex.map(loop, [s[0] for s in setups]))
    total = sum(d for d, _ in res)
    wall = max(t for _, t in res)
    return n_sample * total / wall, (f"{threads} threads, each stepping its own copy of {desc}; "
                                     f"{total} full oracle steps in all")


def timed_steps(z, do_step, K: int, W: int, local: int, dist=None, device=None,
                profile_range: bool = False) -> dict:
    """W untimed warm-up steps, then K steps bracketed by a barrier and
    synchronize() on both sides and timed with CUDA events on the launching
    stream, with nothing else enqueued between the steps' kernels (an event
    between two kernels would keep the second from starting while the first
    finishes). Then K more steps in which the library records four events
    around its own launches (zero_set_step_events), for the per-kernel
    times. Returns the first region (max over ranks), per-step durations and
    per-kernel intervals from the second, and the clocks sampled over both."""
    import torch

    from mixed_precision_gb300 import _abi as abi

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for row in ev:  # events are created on first record
        for e in row:
            e.record()
    for _ in range(W):
        do_step()
    torch.cuda.synchronize()
    barrier(dist, device)

    sampler = ClockSampler(local).start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if profile_range:
        torch.cuda.cudart().cudaProfilerStart()
    t_start.record()
    for k in range(K):
        do_step()
    t_end.record()
    if profile_range:
        torch.cuda.cudart().cudaProfilerStop()
    torch.cuda.synchronize()
    local_ms = t_start.elapsed_time(t_end)
    for k in range(K):  # the per-kernel times
        abi.zero_set_step_events(z.handle, [e.cuda_event for e in ev[k]])
        do_step()
    torch.cuda.synchronize()
    abi.zero_set_step_events(z.handle, None)
    clocks = sampler.stop()
    barrier(dist, device)
    return {"total_ms": max_over_ranks(dist, local_ms, device),
            "steps_ms": sorted(ev[k][0].elapsed_time(ev[k][3]) for k in range(K)),
            "k1": [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)],
            "k2": [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)],
            "k3": [ev[k][2].elapsed_time(ev[k][3]) for k in range(K)],
            "clocks": clocks}


# ---------------------------------------------------------------------------
# Our arm: the CUDA library through its C ABI
# ---------------------------------------------------------------------------

def run_ours(args) -> dict | None:
    import torch

    import workloads as wl
    from mixed_precision_gb300 import _abi as abi
    from mixed_precision_gb300.engine import Hparams, ZeroStep

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    w = workload_of(args)
    K, W = args.steps, args.warmup
    if W < 3:
        raise SystemExit("--warmup must be at least 3")

    z = ZeroStep(w.shapes, w.world, w.stage, w.bucket_bytes, w.grad_dtype, w.param_dtype,
                 w.comm_dtype)
    z.allocate(speculative=args.speculative)
    info = z.info
    numel = wl.numels(w.shapes)
    master0 = wl.master_init(z.offsets, numel, z.np, w.master_sigma, wl.master_seed(w.index),
                             device=device)
    z.init(master0, init_scale=w.init_scale, dynamic=w.dynamic, growth_interval=w.growth_interval)
    torch.cuda.synchronize()
    del master0
    grads = [wl.flat_grads(z.offsets, numel, z.np, w.grad_sigma,
                           wl.grad_seed(w.index, r + 1000 * rank), w.grad_dtype, device=device,
                           zero_params=wl.zero_params(w, r))
             for r in range(w.world)]
    per_tensor = None
    if args.tensors:
        per_tensor = []
        for r in range(w.world):
            zero = set(wl.zero_params(w, r))
            per_tensor.append([None if p in zero else grads[r][off:off + n]
                               for p, (off, n) in enumerate(zip(z.offsets, numel))])

    def do_step():
        if per_tensor is not None and args.speculative:
            z.step_speculative_tensors(per_tensor, hp)
        elif per_tensor is not None:
            z.step_tensors(per_tensor, hp)
        elif args.per_tensor_launch:
            z.step_per_tensor_launch(grads, hp)
        elif args.speculative:
            z.step_speculative(grads, hp)
        else:
            z.step(grads, hp)
    hp = Hparams(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                 max_grad_norm=w.max_grad_norm)

    tm = timed_steps(z, do_step, K, W, local, dist, device, args.profile_range)
    total_ms, steps_ms, k1, k2, k3, clocks = (tm["total_ms"], tm["steps_ms"], tm["k1"], tm["k2"],
                                              tm["k3"], tm["clocks"])
    st = z.scaler_state()
    assert st["overflow"] == 0 and st["steps"] == 2 * K + W, st  # timed, then kernel-timed
    # the speculative step commits on the fast path unless clipping is active
    fast_path = st["fast_path"] if args.speculative else None

    # The same step captured once into a CUDA graph and replayed K times.
    graph = None
    if args.graph and per_tensor is None and not args.per_tensor_launch:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                do_step()
        torch.cuda.current_stream().wait_stream(side)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        r0.record()
        for _ in range(K):
            g.replay()
        r1.record()
        torch.cuda.synchronize()
        st_g = z.scaler_state()
        assert st_g["overflow"] == 0 and st_g["steps"] == 2 * K + W + 3 + K, st_g
        graph = {"ms_per_step": r0.elapsed_time(r1) / K, "steps": K,
                 "value": job_value(info.n_real, world, r0.elapsed_time(r1) / 1e3 / K)}
        del g

    # A skipped step: +inf in one element, the update kernel returns at once.
    saved = grads[0][z.offsets[0]].clone()
    grads[0][z.offsets[0]] = float("inf")
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(3):
        do_step()
    s1.record()
    torch.cuda.synchronize()
    skip_ms = s0.elapsed_time(s1) / 3
    assert z.scaler_state()["skipped"] == 1
    grads[0][z.offsets[0]] = saved
    torch.cuda.synchronize()

    # K4: the cast-out parameters copied into per-tensor storage (one replica),
    # what a framework's parameter tensors would receive after the step.
    gather_params = None
    if not args.tensors:
        pt = [torch.empty(max(n, 8), dtype=z.params_flat.dtype, device=device) for n in numel]
        views = [[t[:n] if n else t for t, n in zip(pt, numel)]]
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(2):
            z.gather(views)
        g0.record()
        for _ in range(10):
            z.gather(views)
        g1.record()
        torch.cuda.synchronize()
        ms = g0.elapsed_time(g1) / 10
        pbytes = wl.ELEM_BYTES[w.param_dtype]
        gather_params = {"replicas": 1, "ms": ms, "gbs": 2 * pbytes * info.n_real / (ms / 1e3) / 1e9,
                         "bytes_per_param": 2 * pbytes}
        del pt, views

    # Gradient accumulation (the step before the reduce): every rank's
    # micro-step gradients added into its fp32 main gradients.
    accumulate = None
    if not args.tensors:
        stream = torch.cuda.current_stream().cuda_stream
        mains = [torch.empty(z.np, dtype=torch.float32, device=device) for _ in range(w.world)]
        mptr, gptr = [t.data_ptr() for t in mains], [g.data_ptr() for g in grads]
        abi.zero_accumulate(z.handle, gptr, w.grad_dtype, mptr, True, stream)
        abi.zero_accumulate(z.handle, gptr, w.grad_dtype, mptr, False, stream)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for _ in range(10):
            abi.zero_accumulate(z.handle, gptr, w.grad_dtype, mptr, False, stream)
        a1.record()
        torch.cuda.synchronize()
        ms = a0.elapsed_time(a1) / 10
        per = w.world * (wl.ELEM_BYTES[w.grad_dtype] + 8)
        accumulate = {"ms": ms, "gbs": per * info.n_real / (ms / 1e3) / 1e9, "bytes_per_param": per}
        del mains

    # Checkpoint in parameter-major order (independent of W, stage and bucket
    # size): export master/m/v, then import them back (the import also
    # recasts the parameters). Only where the three host-side-sized buffers
    # stay small next to the workload.
    checkpoint = None
    if info.n_real * 12 <= 16e9:
        stream = torch.cuda.current_stream().cuda_stream
        pm = [torch.empty(info.n_real, dtype=torch.float32, device=device) for _ in range(3)]
        ptrs = [t.data_ptr() for t in pm]
        abi.zero_state_export_params(z.handle, *ptrs, stream)
        abi.zero_state_import_params(z.handle, *ptrs, stream)
        c0, c1, c2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        c0.record()
        for _ in range(5):
            abi.zero_state_export_params(z.handle, *ptrs, stream)
        c1.record()
        for _ in range(5):
            abi.zero_state_import_params(z.handle, *ptrs, stream)
        c2.record()
        torch.cuda.synchronize()
        ex, im = c0.elapsed_time(c1) / 5, c1.elapsed_time(c2) / 5
        pbytes = wl.ELEM_BYTES[w.param_dtype]
        checkpoint = {"export_ms": ex, "export_gbs": 24 * info.n_real / (ex / 1e3) / 1e9,
                      "import_ms": im,
                      "import_gbs": (24 + 4 + pbytes) * info.n_real / (im / 1e3) / 1e9}
        del pm

    # ZeRO-3: the per-bucket all-gather of the sharded parameters into a flat
    # working buffer (what a forward pass would prefetch bucket by bucket).
    gather = None
    if w.stage == 3:
        stream = torch.cuda.current_stream().cuda_stream
        blen = max(abi.zero_bucket_range(z.handle, b)[1] for b in range(info.n_buckets))
        work = torch.empty(blen, dtype=z.params_flat.dtype, device=device)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        for _ in range(2):
            for b in range(info.n_buckets):
                abi.zero_gather_bucket(z.handle, b, work.data_ptr(), stream)
        g0.record()
        for _ in range(reps):
            for b in range(info.n_buckets):
                abi.zero_gather_bucket(z.handle, b, work.data_ptr(), stream)
        g1.record()
        torch.cuda.synchronize()
        ms = g0.elapsed_time(g1) / reps
        pbytes = wl.ELEM_BYTES[w.param_dtype]
        gather = {"buckets": info.n_buckets, "ms_all_buckets": ms,
                  "gbs": 2 * pbytes * info.n_real / (ms / 1e3) / 1e9,
                  "bytes_per_param": 2 * pbytes}
        del work

    # End to end through the host-buffer entry point: pinned host gradients are
    # copied in every step and the step's scaler state is read back.
    E = args.e2e_steps
    e2e = None
    if E > 0:
        host = [g.cpu().pin_memory() for g in grads]
        # two device gradient sets in turn: each step's copies overlap the
        # previous step's kernels, so the host link never waits for the GPU
        dev_sets = [grads, [torch.empty_like(g) for g in grads]]
        blobs = torch.zeros((E + 1, abi.ZERO_STATE_BLOB_BYTES), dtype=torch.uint8).pin_memory()
        stream = torch.cuda.current_stream().cuda_stream
        for d in dev_sets:
            z.step_host(host, d, hp)
        z.scaler_state()
        torch.cuda.synchronize()
        barrier(dist, device)
        t0 = time.perf_counter()
        for k in range(E):
            z.step_host(host, dev_sets[k % 2], hp)
            # the step's result, read back to the host asynchronously
            abi.zero_loss_scale_state_async(z.handle, blobs[k].data_ptr(), stream)
        torch.cuda.synchronize()
        e2e_s = max_over_ranks(dist, time.perf_counter() - t0, device)
        reads = [abi.zero_state_blob_decode(blobs[k].data_ptr()) for k in range(E)]
        assert all(r.overflow == 0 for r in reads)
        assert [r.steps for r in reads] == list(range(reads[0].steps, reads[0].steps + E))
        del host, dev_sets
        e2e = {"value": job_value(info.n_real, world, e2e_s / E), "unit": "params/s",
               "h2d_bytes_per_step": w.world * z.np * wl.ELEM_BYTES[w.grad_dtype],
               "d2h_bytes_per_step": int(info.state_blob_used),
               "note": "two device gradient sets in turn: each step's host-to-device copies "
                       "overlap the previous step's kernels; the step result is read back "
                       "asynchronously into pinned memory"}

    N = info.n_real
    peak, peak_src = hbm_peak()
    step_s = total_ms / 1e3 / K
    G = wl.ELEM_BYTES[w.grad_dtype]
    C = wl.ELEM_BYTES[w.comm_dtype]
    P = wl.ELEM_BYTES[w.param_dtype]
    k1_bytes = N * (w.world * G + (w.world * C if w.stage == 1 else C))
    k3_bytes = N * (C + 24 + P)
    if args.tensors:  # the update's per-tensor instance skips the idle tiles' gradient reads
        idle = set.intersection(*[set(wl.zero_params(w, r)) for r in range(w.world)])
        k3_bytes -= C * sum(wl.numels(w.shapes)[p] for p in idle)
    k1_ms, k2_ms, k3_ms = statistics.mean(k1), statistics.mean(k2), statistics.mean(k3)
    if args.speculative and fast_path:
        # events: [single pass] [its finalize] [guarded fallback kernels + restore];
        # in stage 1 the pass also writes the W all-reduce outputs
        spec_bytes = N * (info.step_bytes_per_elem + (w.world * C if w.stage == 1 else 0))
        dom = ("k_spec_step", spec_bytes, k1_ms)
        kernels = {"k_spec_step": k1_ms, "between": k2_ms, "guarded_fallback": k3_ms,
                   "k_spec_step_gbs": spec_bytes / (k1_ms / 1e3) / 1e9}
    else:
        dom = ("k_adamw_cast", k3_bytes, k3_ms) if k3_ms >= k1_ms else \
            ("k_reduce_norm", k1_bytes, k1_ms)
        # "k_finalize": the interval between the reduce and the update (the
        # finalize runs inside the reduce's last block, or as its own kernel
        # with the register-staged reduce and per-tensor launches). A
        # speculative step whose last finalize predicted clipping launches
        # these two kernels itself, and the events bracket them the same way.
        kernels = {"k_reduce_norm": k1_ms, "k_finalize": k2_ms, "k_adamw_cast": k3_ms,
                   "k_reduce_norm_gbs": k1_bytes / (k1_ms / 1e3) / 1e9,
                   "k_adamw_cast_gbs": k3_bytes / (k3_ms / 1e3) / 1e9}
    achieved = dom[1] / (dom[2] / 1e3) / 1e9
    # the capture of the instance that ran: the stage-1 single pass, or the
    # per-tensor pointer update, has a key of its own
    kname = dom[0]
    if dom[0] in ("k_spec_step", "k_reduce_norm") and w.stage == 1:
        kname += "_s1"
    elif dom[0] == "k_adamw_cast" and args.tensors:
        kname += "_table"
    tr = NCU_TRAFFIC_PER_ELEM.get((kname, w.name))
    sb = stage_bytes(w)
    # the stage's own bytes: the ledger, plus the all-reduce writes in stage 1
    step_gbs = sb["own"] * N / step_s / 1e9
    impl_bytes = sb["own"] if (args.speculative and fast_path) else sb["impl"]
    out = {
        "metric": METRIC,
        "value": job_value(N, world, step_s),
        "unit": "params/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": total_ms / K,
        "step_ms_median": steps_ms[K // 2],
        "step_ms_min": steps_ms[0],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": config_of(w, "per-tensor gradient pointers, NULL for all-zero gradients"
                            if args.tensors else ("one reduce and one update launch per tensor"
                                                  if args.per_tensor_launch else
                                                  ("speculative single pass; e2e through the "
                                                   "two-pass host entry point"
                                                   if args.speculative else None))),
        "hbm_gbs_step": step_gbs,
        "step_roofline": {"bytes_per_param": sb["own"], "ledger_bytes_per_param": sb["ledger"],
                          "peak_gbs": peak, "frac": step_gbs / peak, "peak_source": peak_src,
                          # bytes the kernels must move per param: the stage's own, plus
                          # (two-pass) the reduced gradient written and read back
                          "impl_bytes_per_param": impl_bytes,
                          "impl_ceiling": sb["own"] / impl_bytes},
        "roofline": {"bound": "hbm", "kernel": dom[0], "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "traffic": (tr * N if tr is not None else None),
                     "algorithmic_bytes_per_launch": dom[1], "peak_source": peak_src},
        "kernels_ms": kernels,
        "fast_path": fast_path,
        "skip_step_ms": skip_ms,
        "graph": graph,
        "zero3_gather": gather,
        "gather_params": gather_params,
        "accumulate": accumulate,
        "checkpoint": checkpoint,
        "e2e": e2e,
        # two-pass: reduce (its last block finalizes) + update; speculative:
        # single pass (finalizes) + guarded reduce + guarded update (which also
        # carries the parameter restore), or, once the device has predicted
        # clipping, the two-pass launches
        "gpu_launches": K * ((2 * sum(1 for n in numel if n > 0) + 1) if args.per_tensor_launch
                             else (3 if (args.speculative and fast_path) else 2)),
        "clocks": clocks,
    }
    z.close()
    if dist is not None:
        dist.destroy_process_group()
    return out if rank == 0 else None


# The other named workloads the step is quoted on, timed after the default
# line in the same run: the ~3.9B MoE list (W=4, ZeRO-2) and the Qwen3 list
# with fp16 dynamic scaling at W=8, ZeRO-1 against ZeRO-2.
PER_CONFIG = [
    ("moe_3.9b_bf16_w4", {"stage": 2}),
    ("qwen3_0.6b_fp16_w8", {"stage": 1}),
    ("qwen3_0.6b_fp16_w8", {"stage": 2}),
    # the speculative step where clipping stays off: one pass, the step's
    # whole ledger (the default line's workload clips every step)
    ("qwen3_0.6b_bf16_w2", {"max_grad_norm": 0.0, "speculative": True}),
    ("moe_3.9b_bf16_w4", {"max_grad_norm": 0.0, "speculative": True}),
    # ZeRO-1 at fp16 W=8, clip 1.0 (inactive there): the single pass also
    # writes the W all-reduce outputs
    ("qwen3_0.6b_fp16_w8", {"stage": 1, "speculative": True}),
    # the layout sweep's 2000 ragged tensors (1.69G elements): the flat step at
    # W = 2 and 8, and at W = 8 the same step launched tensor by tensor
    ("ragged_2000", {"world": 2}),
    ("ragged_2000", {"world": 8}),
    ("ragged_2000", {"world": 8, "per_tensor_launch": True}),
    # the MoE list as its gradients arrive: each rank's idle experts (14 of 16
    # per layer) passed as NULL pointers
    ("moe_3.9b_bf16_w4", {"stage": 2, "tensors": True}),
]


def stage_bytes(w) -> dict:
    """Bytes per real element of one step of workload w.

    ledger: the step's byte roofline, W*G gradient reads + 24 B of fp32
    master/m/v read and written + P B of parameter writes. own: what the
    stage itself must move -- stage 1 also writes the all-reduce result into
    all W outputs (W*C more). impl: what the two-pass kernels move -- the
    reduced gradient is stored (C, or W*C in stage 1) and read back (C).
    """
    import workloads as wl
    G, C, P = (wl.ELEM_BYTES[w.grad_dtype], wl.ELEM_BYTES[w.comm_dtype],
               wl.ELEM_BYTES[w.param_dtype])
    ledger = w.world * G + 24 + P
    own = ledger + (w.world * C if w.stage == 1 else 0)
    impl = ledger + (w.world * C if w.stage == 1 else C) + C
    return {"ledger": ledger, "own": own, "impl": impl,
            "k1": w.world * G + (w.world * C if w.stage == 1 else C), "k3": C + 24 + P}


def time_config(name: str, over: dict, steps: int, warmup: int, local: int) -> dict:
    """One named workload through zero_step (or, with over["speculative"],
    zero_step_speculative): its own buffers, seeded inputs, warm-up, K timed
    steps with per-kernel events and sampled clocks. Frees every buffer
    before it returns."""
    import torch

    import workloads as wl
    from mixed_precision_gb300.engine import Hparams, ZeroStep

    device = torch.device("cuda", local)
    over = dict(over)
    speculative = over.pop("speculative", False)
    per_tensor_launch = over.pop("per_tensor_launch", False)
    tensors = over.pop("tensors", False)
    w = wl.workload(name, **over)
    z = ZeroStep(w.shapes, w.world, w.stage, w.bucket_bytes, w.grad_dtype, w.param_dtype,
                 w.comm_dtype)
    z.allocate(speculative=speculative)
    numel = wl.numels(w.shapes)
    master0 = wl.master_init(z.offsets, numel, z.np, w.master_sigma, wl.master_seed(w.index),
                             device=device)
    z.init(master0, init_scale=w.init_scale, dynamic=w.dynamic, growth_interval=w.growth_interval)
    torch.cuda.synchronize()
    del master0
    grads = [wl.flat_grads(z.offsets, numel, z.np, w.grad_sigma, wl.grad_seed(w.index, r),
                           w.grad_dtype, device=device, zero_params=wl.zero_params(w, r))
             for r in range(w.world)]
    hp = Hparams(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                 max_grad_norm=w.max_grad_norm)
    sparse_read = None
    if tensors:
        # per-tensor pointers, NULL for a rank's all-zero gradients (the
        # experts its tokens did not reach): those reads are skipped
        per, live_elems = [], 0
        for r in range(w.world):
            zero = set(wl.zero_params(w, r))
            per.append([None if p in zero else grads[r][off:off + n]
                        for p, (off, n) in enumerate(zip(z.offsets, numel))])
            live_elems += sum(n for p, n in enumerate(numel) if p not in zero)
        sparse_read = live_elems * wl.ELEM_BYTES[w.grad_dtype] / w.n_real  # B/param read
        # parameters NULL on every rank: the update does not read their
        # reduced gradient back (it is +0.0)
        idle = set.intersection(*[set(wl.zero_params(w, r)) for r in range(w.world)])
        idle_frac = sum(numel[p] for p in idle) / w.n_real
        step = lambda: z.step_tensors(per, hp)  # noqa: E731
    elif speculative:
        step = lambda: z.step_speculative(grads, hp)  # noqa: E731
    elif per_tensor_launch:
        step = lambda: z.step_per_tensor_launch(grads, hp)  # noqa: E731
    else:
        step = lambda: z.step(grads, hp)  # noqa: E731
    tm = timed_steps(z, step, steps, warmup, local)
    st = z.scaler_state()
    assert st["overflow"] == 0 and st["steps"] == 2 * steps + warmup, st
    N = w.n_real
    peak, peak_src = hbm_peak()
    b = stage_bytes(w)
    step_s = tm["total_ms"] / 1e3 / steps
    k1_ms, k3_ms = statistics.mean(tm["k1"]), statistics.mean(tm["k3"])
    if speculative:
        # events: [single pass, its finalize in its last block] [between]
        # [guarded fallback kernels: no-ops when the step committed]
        assert st["fast_path"] == 1, st
        one_pass = b["own"]  # the ledger, and in stage 1 the W all-reduce writes
        out = {
            "config": config_of(w, "speculative single pass; clipping inactive, so every step "
                                   "commits in one pass"),
            "steps": steps, "warmup": warmup,
            "ms_per_step": tm["total_ms"] / steps,
            "step_ms_median": tm["steps_ms"][steps // 2],
            "value": N / step_s, "unit": "params/s",
            "step_roofline": {"bytes_per_param": b["own"], "ledger_bytes_per_param": b["ledger"],
                              "hbm_gbs": b["own"] * N / step_s / 1e9, "peak_gbs": peak,
                              "frac": b["own"] * N / step_s / 1e9 / peak, "peak_source": peak_src,
                              "impl_bytes_per_param": one_pass, "impl_ceiling": 1.0},
            "kernels_ms": {"k_spec_step": k1_ms, "between": statistics.mean(tm["k2"]),
                           "guarded_fallback": k3_ms,
                           "k_spec_step_gbs": one_pass * N / (k1_ms / 1e3) / 1e9},
            "fast_path": st["fast_path"],
            "clocks": tm["clocks"],
        }
        achieved = one_pass * N / (k1_ms / 1e3) / 1e9
        tr = NCU_TRAFFIC_PER_ELEM.get(("k_spec_step" + ("_s1" if w.stage == 1 else ""), w.name))
        out["roofline"] = {"bound": "hbm", "kernel": "k_spec_step", "achieved": achieved,
                           "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                           "traffic": tr * N if tr is not None else None,
                           "algorithmic_bytes_per_launch": one_pass * N, "peak_source": peak_src}
        z.close()
        del grads, z
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        return out
    note = None
    if per_tensor_launch:
        note = "per-tensor launches: two kernels per parameter and the finalize"
    elif tensors:
        note = ("per-tensor gradient pointers, NULL where a rank's gradient is all zero; the "
                "ledger counts those reads, sparse_bytes_per_param does not")
    out = {
        "config": config_of(w, note),
        "steps": steps, "warmup": warmup,
        "ms_per_step": tm["total_ms"] / steps,
        "step_ms_median": tm["steps_ms"][steps // 2],
        "value": N / step_s, "unit": "params/s",
        "step_roofline": {"bytes_per_param": b["own"], "ledger_bytes_per_param": b["ledger"],
                          "hbm_gbs": b["own"] * N / step_s / 1e9, "peak_gbs": peak,
                          "frac": b["own"] * N / step_s / 1e9 / peak, "peak_source": peak_src,
                          "impl_bytes_per_param": b["impl"],
                          "impl_ceiling": b["own"] / b["impl"]},
        "kernels_ms": {"k_reduce_norm": k1_ms, "k_finalize": statistics.mean(tm["k2"]),
                       "k_adamw_cast": k3_ms,
                       "k_reduce_norm_gbs": b["k1"] * N / (k1_ms / 1e3) / 1e9,
                       "k_adamw_cast_gbs": b["k3"] * N / (k3_ms / 1e3) / 1e9},
        "clip_coef_last": st["clip_coef"],
        "scale": st["scale"],
        "clocks": tm["clocks"],
    }
    if sparse_read is not None:
        # the bytes the step must move when the NULL gradients are not read
        sb = sparse_read + (b["own"] - w.world * wl.ELEM_BYTES[w.grad_dtype])
        out["step_roofline"]["sparse_bytes_per_param"] = sb
        out["step_roofline"]["sparse_frac"] = sb * N / step_s / 1e9 / peak
        out["kernels_ms"]["k_reduce_norm_sparse_gbs"] = (
            (sparse_read + b["k1"] - w.world * wl.ELEM_BYTES[w.grad_dtype]) * N / (k1_ms / 1e3) / 1e9)
    k3_b = b["k3"]
    if tensors:  # the update's per-tensor instance skips the idle tiles' gradient reads
        k3_b -= wl.ELEM_BYTES[w.comm_dtype] * idle_frac
        out["kernels_ms"]["k_adamw_cast_gbs"] = k3_b * N / (k3_ms / 1e3) / 1e9
    dom, dom_ms, dom_b = (("k_adamw_cast", k3_ms, k3_b) if k3_ms >= k1_ms
                          else ("k_reduce_norm", k1_ms, b["k1"]))
    achieved = dom_b * N / (dom_ms / 1e3) / 1e9
    suffix = "_table" if tensors else ("_s1" if dom == "k_reduce_norm" and w.stage == 1 else "")
    tr = NCU_TRAFFIC_PER_ELEM.get((dom + suffix, w.name))
    out["roofline"] = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                       "unit": "GB/s", "frac": achieved / peak,
                       "traffic": tr * N if tr is not None else None,
                       "algorithmic_bytes_per_launch": dom_b * N, "peak_source": peak_src}
    z.close()
    del grads, z
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def per_config(steps: int, warmup: int, local: int) -> dict:
    """Every workload of PER_CONFIG, one after the other."""
    out = {}
    for name, over in PER_CONFIG:
        if over.get("speculative") and over.get("stage") == 1:
            key = name + "_stage1_speculative"
        elif over.get("speculative"):
            key = name + "_speculative_clip0"
        elif over.get("tensors"):
            key = name + "_tensors_idle_experts_null"
        elif name == "ragged_2000":
            key = f"{name}_w{over['world']}" + ("_per_tensor_launch" if over.get("per_tensor_launch")
                                                 else "")
        else:
            key = name + "".join(f"_{k}{v}" for k, v in over.items())
        out[key] = time_config(name, over, steps, warmup, local)
    return out


def local_buckets(z, rank: int) -> int:
    """Buckets whose slice for `rank` holds a real element (each is one
    update launch of the sharded step)."""
    from mixed_precision_gb300 import _abi as abi
    n = 0
    for b in range(z.info.n_buckets):
        f0, _, ln = abi.zero_shard_range(z.handle, b, rank)
        if any(min(o + k, f0 + ln) > max(o, f0) for o, k in zip(z.offsets, z.numels) if k > 0):
            n += 1
    return n


def run_sharded(args) -> dict | None:
    """The sharded step across N GPUs (one process each): the workload's
    parameter list with W = N, each rank's own seeded gradients, timed over
    the whole step (collectives included) with CUDA events on the launching
    stream, max over ranks. The model is fixed, so its shards shrink as N
    grows: strong scaling."""
    import socket

    import torch
    import torch.distributed as tdist

    import workloads as wl
    from mixed_precision_gb300.engine import Hparams
    from mixed_precision_gb300.sharded import ShardedZeroStep

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if not tdist.is_initialized():
        if "MASTER_PORT" not in os.environ:  # a single process without torchrun
            with socket.socket() as s:
                s.bind(("127.0.0.1", 0))
                os.environ["MASTER_PORT"] = str(s.getsockname()[1])
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        tdist.init_process_group("nccl", rank=rank, world_size=world, device_id=device)
    w = dataclasses_replace(workload_of(args), world=world)
    if w.stage == 1:
        raise SystemExit("--sharded times stages 2 and 3 (stage 1 all-reduces the gradients in place)")
    K, Wm = args.steps, args.warmup
    if Wm < 3:
        raise SystemExit("--warmup must be at least 3")
    z = ShardedZeroStep(w.shapes, w.stage, w.bucket_bytes, w.grad_dtype, w.param_dtype,
                        device=device)
    numel = wl.numels(w.shapes)
    master0 = wl.master_init(z.offsets, numel, z.np, w.master_sigma, wl.master_seed(w.index),
                             device=device)
    z.init(master0, init_scale=w.init_scale, dynamic=w.dynamic, growth_interval=w.growth_interval)
    del master0
    grads = wl.flat_grads(z.offsets, numel, z.np, w.grad_sigma, wl.grad_seed(w.index, rank),
                          w.grad_dtype, device=device, zero_params=wl.zero_params(w, rank))
    hp = Hparams(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                 max_grad_norm=w.max_grad_norm)
    for _ in range(Wm):
        z.step(grads, hp)
    torch.cuda.synchronize()
    barrier(tdist if world > 1 else None, device)
    sampler = ClockSampler(local).start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record()
    for _ in range(K):
        z.step(grads, hp)
    t1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    dist = tdist if world > 1 else None
    barrier(dist, device)
    total_ms = max_over_ranks(dist, t0.elapsed_time(t1), device)
    st = z.scaler_state()
    assert st["overflow"] == 0 and st["steps"] == K + Wm, st

    # this rank's update kernel alone (the dominant local kernel)
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    u0.record()
    for _ in range(10):
        z.local.update(None)
    u1.record()
    torch.cuda.synchronize()
    upd_ms = u0.elapsed_time(u1) / 10
    # end to end: each step's gradients copied in from pinned host memory, the
    # scaler state read back after the loop
    from mixed_precision_gb300 import _abi as abi
    host = grads.cpu().pin_memory()
    E = max(1, min(args.e2e_steps, 10))
    blobs = torch.zeros((E, abi.ZERO_STATE_BLOB_BYTES), dtype=torch.uint8).pin_memory()
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    barrier(dist, device)
    e0 = time.perf_counter()
    for k in range(E):
        grads.copy_(host, non_blocking=True)
        z.step(grads, hp)
        abi.zero_loss_scale_state_async(z.handle, blobs[k].data_ptr(), stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(dist, time.perf_counter() - e0, device)
    assert all(abi.zero_state_blob_decode(blobs[k].data_ptr()).overflow == 0 for k in range(E))

    N = w.n_real
    G, C, P = (wl.ELEM_BYTES[w.grad_dtype], wl.ELEM_BYTES[w.comm_dtype],
               wl.ELEM_BYTES[w.param_dtype])
    peak, peak_src = hbm_peak()
    upd_bytes = (C + 24 + P) * z.info.n_real / world
    achieved = upd_bytes / (upd_ms / 1e3) / 1e9
    step_s = total_ms / 1e3 / K
    out = {
        "metric": METRIC, "value": N / step_s, "unit": "params/s", "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(config_of(w), parallelism=f"zero{w.stage}_dp{world}",
                       note="one rank per GPU: per-bucket reduce-scatter, 16-byte norm "
                            "all-reduce and per-bucket all-gather (NCCL) around the local "
                            "kernels"),
        "roofline": {"bound": "hbm", "kernel": "k_adamw_cast (this rank's shard)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "algorithmic_bytes_per_launch": upd_bytes,
                     "peak_source": peak_src},
        "e2e": {"value": N / (e2e_s / E), "unit": "params/s",
                "h2d_bytes_per_step": z.np * G, "d2h_bytes_per_step": int(z.info.state_blob_used),
                "note": "per rank: its gradients copied in from pinned host memory each step, "
                        "the step's scaler state read back asynchronously"},
        # per step: the shard norm, the finalize and the update -- one launch
        # per bucket that holds some of this rank's elements when the
        # all-gathers overlap it (stages 1/2), one in stage 3 (the collectives
        # are NCCL's kernels)
        "gpu_launches": K * (2 + (1 if w.stage == 3 else local_buckets(z, rank))),
        "clocks": clocks,
    }
    z.close()
    if world > 1:
        tdist.destroy_process_group()
    return out if rank == 0 else None


def dataclasses_replace(w, **kw):
    import dataclasses
    return dataclasses.replace(w, **kw)


# ---------------------------------------------------------------------------
# Reference arm: the host oracle (a deliberately slow program)
# ---------------------------------------------------------------------------

def cpu_baseline(w, seconds: float) -> dict:
    rate, done, n, desc = time_oracle(w, 20_000_000, seconds)
    out = {"value": rate, "unit": "params/s", "cores": 1, "kind": "oracle", "sample": desc}
    cores = os.cpu_count() or 1
    if cores > 1:
        rate_mt, desc_mt = time_oracle_threads(w, 4_000_000, seconds / 2, cores)
        out["all_cores"] = {"value": rate_mt, "unit": "params/s", "cores": cores, "sample": desc_mt}
    return out


def run_reference(args) -> dict | None:
    import workloads as wl
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    w = workload_of(args)
    # size each step's sample so the whole run stays within about two minutes
    rate0, _, _, _ = time_oracle(w, 1_000_000, 0.0, min_steps=1)
    per_step = max(1_000_000, int(rate0 * 120.0 / max(1, args.steps + args.warmup)))
    per_step = min(per_step, 20_000_000)
    rate, done, n, desc = time_oracle(w, per_step, 0.0, warmup=args.warmup, steps=args.steps)
    cpu = {"value": rate, "unit": "params/s", "cores": 1, "kind": "oracle", "sample": desc}
    return {"impl": "reference", "metric": METRIC, "value": rate, "unit": "params/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": n / rate * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_of(w),
            "cpu_baseline": cpu,
            "e2e": {"value": rate, "unit": "params/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        out = run_reference(args)
    elif args.sharded:
        out = run_sharded(args)
    else:
        out = run_ours(args)
        rank, world, local = dist_env()
        if out is not None and world == 1 and args.per_config_steps > 0:
            out["per_config"] = per_config(args.per_config_steps, max(3, args.warmup), local)
        if out is not None and world == 1 and not args.no_cpu_baseline:
            import workloads as wl
            out["cpu_baseline"] = cpu_baseline(workload_of(args), args.cpu_seconds)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
