"""Seeded random configurations against the oracle (GB300).

Each case draws a parameter list (ragged sizes from 1 to 60K or, in a
quarter of the cases, 400K elements, empty tensors included), a world size,
a ZeRO stage, gradient / parameter / communication dtypes, a bucket size,
hyperparameters and a sequence of three entry points (flat buffers, per-tensor pointers with NULL for all-zero
gradients, tensor-by-tensor launches, host gradients, the speculative step),
then steps it three times, some steps with an injected non-finite gradient,
and checks every step against the oracle with the parity harness's bars:
reduced values, overflow flag, loss scale, counter and t bit-exact; the norm
and clip coefficient within 1e-6; fp32 state within 1e-5 of the largest
magnitude held; parameters within 1 ulp. The point is the interactions that
the targeted tests take one at a time.
"""
import numpy as np
import pytest

import workloads as wl
from _parity import Pair
from mixed_precision_gb300.engine import Hparams

pytestmark = pytest.mark.gpu

N_CASES = 96


def draw(i: int) -> dict:
    rng = np.random.default_rng(1000 + i)
    W = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16]))
    stage = int(rng.choice([1, 2, 3]))
    gdt = int(rng.choice([wl.BF16, wl.F16, wl.F32]))
    pdt = int(rng.choice([wl.BF16, wl.F16]))
    cdt = -1
    if gdt != wl.F32 and rng.random() < 0.3:
        cdt = wl.F32  # fp32 collectives of 16-bit gradients
    n_t = int(rng.integers(3, 40))
    top = 400_000 if rng.random() < 0.25 else 60_000  # some lists span many tiles per tensor
    sizes = np.exp(rng.uniform(0.0, np.log(top), size=n_t)).astype(int).tolist()
    if rng.random() < 0.5:
        sizes[int(rng.integers(n_t))] = 0
    shapes = [(int(s),) for s in sizes]
    bucket = int(rng.choice([4096, 40_000, 300_000, 2_000_000]))
    dynamic = gdt == wl.F16 and rng.random() < 0.7
    init_scale = float(2.0 ** int(rng.integers(4, 14))) if dynamic else 1.0
    clip = float(rng.choice([0.0, 1e-3, 1.0]))
    hp = Hparams(lr=float(rng.choice([1e-4, 1e-3])), weight_decay=float(rng.choice([0.0, 0.1])),
                 max_grad_norm=clip)
    modes = ["flat", "tensors", "per_tensor_launch", "host", "speculative"]
    if stage != 1:
        modes += ["speculative_tensors"]
    plan = [str(rng.choice(modes)) for _ in range(3)]
    inject = [bool(rng.random() < 0.25) for _ in range(3)]
    zero_params = [int(p) for p in rng.choice(n_t, size=n_t // 4, replace=False)]
    return dict(W=W, stage=stage, gdt=gdt, pdt=pdt, cdt=cdt, shapes=shapes, bucket=bucket,
                dynamic=dynamic, init_scale=init_scale, hp=hp, plan=plan, inject=inject,
                zero_params=zero_params, seed=1000 + i)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_config_matches_oracle(i):
    c = draw(i)
    desc = {k: v for k, v in c.items() if k not in ("shapes", "hp")}
    desc["tensors"] = len(c["shapes"])
    speculative = any(m.startswith("speculative") for m in c["plan"])
    pr = Pair(c["shapes"], c["W"], c["stage"], c["bucket"], c["gdt"], c["pdt"], comm_dtype=c["cdt"],
              init_scale=c["init_scale"], dynamic=c["dynamic"], growth_interval=2,
              index=c["seed"] % 997, speculative=speculative)
    rng = np.random.default_rng(c["seed"] + 1)
    sigma = 1e-3 * c["init_scale"]
    for step, (mode, inj) in enumerate(zip(c["plan"], c["inject"])):
        g = pr.grads(step, sigma, zero_params=c["zero_params"])
        live = [p for p, n in enumerate(pr.numel) if n > 0 and p not in c["zero_params"]]
        if inj and live:
            p = live[int(rng.integers(len(live)))]
            r = int(rng.integers(c["W"]))
            g[r][pr.offsets[p] + int(rng.integers(pr.numel[p]))] = float("inf")
        st, info, gc = pr.step(g, c["hp"], mode=mode)
        try:
            pr.check(st, info, gc)
        except AssertionError as e:
            raise AssertionError(f"case {desc}, step {step} ({mode}): {e}") from e
        if inj and live:
            assert info.skipped == 1 and st["skipped"] == 1, desc
