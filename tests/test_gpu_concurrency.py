"""Two layouts stepping at the same time on two streams share nothing: each
keeps its own device state (scaler, finalize counter, partials), so the
results equal those of each layout stepped alone, bit for bit."""
import pytest
import torch

import workloads as wl
from mixed_precision_gb300 import _abi as abi
from mixed_precision_gb300.engine import Hparams, ZeroStep

pytestmark = pytest.mark.gpu


def _shapes(k):
    return wl.qwen3_0_6b_shapes(vocab=800 + 100 * k, hidden=128, layers=2, q_dim=256, kv_dim=128,
                                ffn=384, head_dim=32)


def _make(k, spec):
    sh = _shapes(k)
    z = ZeroStep(sh, 2 + k, 2, 40_000, wl.BF16, wl.BF16)
    z.allocate(speculative=spec)
    z.init(wl.master_init(z.offsets, z.numels, z.np, 0.02, wl.master_seed(50 + k), device="cuda"),
           init_scale=8.0, dynamic=True, growth_interval=3)
    grads = [[wl.flat_grads(z.offsets, z.numels, z.np, 1e-3, wl.grad_seed(60 + k, r, s), wl.BF16,
                            device="cuda") for r in range(2 + k)] for s in range(4)]
    return z, grads


def _real(z):
    """Real elements of the rank-major state (the alternate set's padding is
    never written)."""
    mask = torch.zeros(max(z.np, 8), dtype=torch.bool, device="cuda")
    for b in range(z.info.n_buckets):
        for r in range(z.world):
            f0, s0, ln = abi.zero_shard_range(z.handle, b, r)
            for off, n in zip(z.offsets, z.numels):
                lo, hi = max(off, f0), min(off + n, f0 + ln)
                if lo < hi:
                    mask[s0 + lo - f0:s0 + hi - f0] = True
    return mask


def _run(z, grads, spec, stream=None):
    for s, g in enumerate(grads):
        hp = Hparams(max_grad_norm=1e-4 if s == 2 else 1.0)
        if spec:
            z.step_speculative(g, hp, stream=stream)
        else:
            z.step(g, hp, stream=stream)


@pytest.mark.parametrize("spec", [False, True])
def test_two_layouts_on_two_streams(spec):
    alone = []
    for k in range(2):
        z, g = _make(k, spec)
        _run(z, g, spec)
        torch.cuda.synchronize()
        mask = _real(z)
        alone.append(([t[mask].clone() for t in z.current_state()], z.params_flat.clone(),
                      z.scaler_state()))
        z.close()
    pair = [_make(k, spec) for k in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    torch.cuda.synchronize()
    for (z, g), s in zip(pair, streams):
        with torch.cuda.stream(s):
            _run(z, g, spec, stream=s)
    torch.cuda.synchronize()
    for (z, _), (state, params, sc) in zip(pair, alone):
        assert z.scaler_state() == sc
        mask = _real(z)
        for x, y in zip(z.current_state(), state):
            assert torch.equal(x[mask].view(torch.int32), y.view(torch.int32))
        assert torch.equal(z.params_flat.view(torch.int16), params.view(torch.int16))
        z.close()
