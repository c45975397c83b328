"""Workload definitions and seeded synthetic inputs for the ZeRO-1/2 step.

This module is shared by the oracle side (tests) and the CUDA side (tests,
smoke check, benchmark). It holds parameter-shape lists, seeds and random
draws only -- none of the step's arithmetic (no reduction, no scaling, no
optimizer math). Low-precision draws are rounded by torch's own dtype cast.

No model weights or datasets are used: the parameter lists are shape-only
stand-ins for the models the pages train (Qwen3-0.6B in "nano-deepspeed
(Teaching Edition)", section "9. Experimental Results"; the Phi-tiny-MoE-style
expert model of "nanoMegatron", section "Model"), and every value is drawn
from a seeded normal distribution.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

F32, F16, BF16 = 0, 1, 2
TORCH_DTYPE = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}
ELEM_BYTES = {F32: 4, F16: 2, BF16: 2}
DTYPE_NAME = {F32: "f32", F16: "f16", BF16: "bf16"}


# ---------------------------------------------------------------------------
# Parameter-shape lists
# ---------------------------------------------------------------------------

def tiny_shapes():
    """Three parameters: [256,256], [256], [1024,256] (327,936 elements)."""
    return [(256, 256), (256,), (1024, 256)]


def qwen3_0_6b_shapes(vocab=151936, hidden=1024, layers=28, q_dim=2048, kv_dim=1024,
                      ffn=3072, head_dim=128):
    """Qwen3-0.6B-shaped list (tied embedding): 310 tensors, 596,049,920 elements.

    Order per layer: q, k, v, o, q_norm, k_norm, gate, up, down, input norm,
    post-attention norm; then the final norm.
    """
    shapes = [(vocab, hidden)]
    for _ in range(layers):
        shapes += [(q_dim, hidden), (kv_dim, hidden), (kv_dim, hidden), (hidden, q_dim),
                   (head_dim,), (head_dim,), (ffn, hidden), (ffn, hidden), (hidden, ffn),
                   (hidden,), (hidden,)]
    shapes.append((hidden,))
    return shapes


def moe_3_9b_shapes(vocab=32064, hidden=2048, layers=32, experts=16, ffn=1024):
    """MoE list: embedding + untied head, per layer q/k/v/o, a router and 16
    SwiGLU experts (w1, w3 [ffn, hidden], w2 [hidden, ffn]): 1698 tensors,
    3,890,479,104 elements. Returns (shapes, expert_index) where expert_index[i]
    is (layer, expert) for expert tensors and None otherwise."""
    shapes, tag = [(vocab, hidden)], [None]
    for layer in range(layers):
        for _ in range(4):
            shapes.append((hidden, hidden))
            tag.append(None)
        shapes.append((experts, hidden))
        tag.append(None)
        for e in range(experts):
            for s in [(ffn, hidden), (ffn, hidden), (hidden, ffn)]:
                shapes.append(s)
                tag.append((layer, e))
    shapes.append((vocab, hidden))
    tag.append(None)
    return shapes, tag


def ragged_shapes(n=2000, lo=1e2, hi=1e7, seed=0x5A5A):
    """n one-dimensional tensors, sizes log-uniform in [lo, hi] (seeded)."""
    rng = np.random.default_rng(seed)
    sizes = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n)).astype(np.int64)
    return [(int(s),) for s in sizes]


def numels(shapes):
    return [int(np.prod(s)) if len(s) else 1 for s in shapes]


# ---------------------------------------------------------------------------
# Named configurations
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    shapes: list
    world: int
    stage: int
    grad_dtype: int
    param_dtype: int
    comm_dtype: int
    bucket_bytes: int
    grad_sigma: float
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    max_grad_norm: float = 1.0
    init_scale: float = 1.0
    dynamic: bool = False
    growth_interval: int = 1000
    master_sigma: float = 0.02
    index: int = 0  # seeds are derived from it

    @property
    def n_real(self) -> int:
        return sum(numels(self.shapes))


MB = 1000 * 1000


def workload(name: str, **over) -> Workload:
    """The named workloads. Keyword arguments override fields."""
    if name == "tiny":
        w = Workload("tiny", tiny_shapes(), 2, 2, F16, F16, F16, 500 * MB, 1e-3,
                     init_scale=2.0 ** 16, dynamic=True, index=1)
    elif name == "qwen3_0.6b_bf16_w2":
        w = Workload(name, qwen3_0_6b_shapes(), 2, 2, BF16, BF16, BF16, 500 * MB, 1e-4, index=2)
    elif name == "qwen3_0.6b_fp16_w8":
        w = Workload(name, qwen3_0_6b_shapes(), 8, 2, F16, F16, F16, 500 * MB, 1e-4,
                     init_scale=2.0 ** 16, dynamic=True, index=3)
    elif name == "qwen3_layers8_bf16_w2":
        # 8 Qwen3-0.6B decoder layers, no embedding: 125.8M elements, about
        # 2.5 GB on the device; a profiling-sized case of the same kernels.
        w = Workload(name, qwen3_0_6b_shapes(layers=8)[1:-1], 2, 2, BF16, BF16, BF16, 500 * MB,
                     1e-4, index=6)
    elif name == "qwen3_layers8_fp16_w8":
        # the same 8 layers with the fp16 W=8 list's dtypes and loss scaling
        w = Workload(name, qwen3_0_6b_shapes(layers=8)[1:-1], 8, 2, F16, F16, F16, 500 * MB, 1e-4,
                     init_scale=2.0 ** 16, dynamic=True, index=9)
    elif name == "moe_layers2_bf16_w4":
        # 2 layers of the MoE list (attention, router, 16 experts each), no
        # embedding or head: 235M elements, about 5.6 GB on the device; a
        # profiling-sized case of the same kernels with the same expert mix.
        w = Workload(name, moe_3_9b_shapes(layers=2)[0][1:-1], 4, 2, BF16, BF16, BF16, 500 * MB,
                     1e-4, index=7)
    elif name == "moe_3.9b_bf16_w4":
        w = Workload(name, moe_3_9b_shapes()[0], 4, 2, BF16, BF16, BF16, 500 * MB, 1e-4, index=4)
    elif name == "ragged_200_slice":
        # the first 200 tensors of the 2000-tensor list: 160.9M elements, about
        # 2.9 GB on the device at W=2; a profiling-sized case of the same kernels
        w = Workload(name, ragged_shapes()[:200], 2, 2, BF16, BF16, BF16, 128 * MB, 1e-3, index=8)
    elif name == "ragged_2000":
        w = Workload(name, ragged_shapes(), 2, 2, BF16, BF16, BF16, 128 * MB, 1e-3, index=5)
    else:
        raise KeyError(name)
    return dataclasses.replace(w, **over)


# ---------------------------------------------------------------------------
# Seeds and draws
# ---------------------------------------------------------------------------

def grad_seed(index: int, rank: int, step: int = 0) -> int:
    return 0x5EED0000 + 100 * index + rank + (step << 20)


def master_seed(index: int) -> int:
    return 0xA11CE + index


def normal(n: int, sigma: float, seed: int, dtype: int, device="cpu") -> torch.Tensor:
    """n draws of N(0, sigma^2) (sigma is the standard deviation), rounded to dtype."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
    x.mul_(sigma)
    return x.to(TORCH_DTYPE[dtype])


def flat_grads(param_offset, numel, np_total: int, sigma: float, seed: int, dtype: int,
               device="cpu", pad_fill: float | None = float("nan"), zero_params=()) -> torch.Tensor:
    """One rank's gradients in a flat layout: each parameter's draw at its offset.

    Padding elements get pad_fill (NaN by default, so a step that reads padding
    shows it). Parameters listed in zero_params are all-zero.
    """
    n_real = int(sum(numel))
    vals = normal(n_real, sigma, seed, dtype, device)
    out = torch.empty(np_total, dtype=TORCH_DTYPE[dtype], device=device)
    if pad_fill is None:
        out.zero_()
    else:
        out.fill_(pad_fill)
    at = 0
    zero = set(zero_params)
    for p, (off, n) in enumerate(zip(param_offset, numel)):
        off, n = int(off), int(n)
        if p in zero:
            out[off:off + n].zero_()
        else:
            out[off:off + n].copy_(vals[at:at + n])
        at += n
    return out


def master_init(param_offset, numel, np_total: int, sigma: float, seed: int,
                device="cpu") -> torch.Tensor:
    """fp32 master weights N(0, sigma^2) at each parameter's flat offset; padding 0."""
    return flat_grads(param_offset, numel, np_total, sigma, seed, F32, device, pad_fill=0.0)


def moe_zero_experts(tags, rank: int, seed: int, experts=16, active=2):
    """Parameter indices whose gradients are all-zero for this rank: per layer,
    all but `active` seeded experts (top-2 of 16 leaves 7/8 of expert grads zero)."""
    rng = np.random.default_rng(seed + 7919 * rank)
    layers = sorted({t[0] for t in tags if t is not None})
    live = {layer: set(rng.choice(experts, size=active, replace=False).tolist()) for layer in layers}
    return [i for i, t in enumerate(tags) if t is not None and t[1] not in live[t[0]]]


def inject_position(numel, param_offset, world: int, seed: int):
    """A seeded (rank, flat index) of a real element, for +inf injection."""
    rng = np.random.default_rng(seed)
    rank = int(rng.integers(0, world))
    p = int(rng.integers(0, len(numel)))
    while int(numel[p]) == 0:
        p = (p + 1) % len(numel)
    k = int(rng.integers(0, int(numel[p])))
    return rank, int(param_offset[p]) + k


def zero_params(w: Workload, rank: int):
    """Parameters whose gradients are all zero on this rank: for the MoE
    workload, the experts that rank's tokens did not route to (14 of 16 per
    layer); none otherwise."""
    if w.name.startswith("moe_"):
        layers = 2 if w.name == "moe_layers2_bf16_w4" else 32
        _, tags = moe_3_9b_shapes(layers=layers)
        if layers == 2:
            tags = tags[1:-1]
        return moe_zero_experts(tags, rank, grad_seed(w.index, 0))
    return []
