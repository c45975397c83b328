"""Guard bands around every buffer the kernels write (compute-sanitizer is
closed on this pool, so out-of-bounds writes are caught this way instead).

Each caller-owned output buffer sits between two 4 KiB guard regions filled
with a fixed byte pattern; the padding of the flat buffers holds NaN
gradients. After steps in every stage, the per-tensor and host entry points,
gathers, exports, imports and accumulation, every guard byte must still hold
its pattern.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from mixed_precision_gb300 import _abi as abi
from mixed_precision_gb300.engine import Hparams, ZeroStep

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A device buffer of `n` elements with GUARD bytes of pattern on each side."""

    def __init__(self, n, dtype):
        esz = torch.empty(0, dtype=dtype).element_size()
        self.raw = torch.full((2 * GUARD + max(n, 8) * esz,), PATTERN, dtype=torch.uint8,
                              device="cuda")
        self.t = self.raw[GUARD:GUARD + max(n, 8) * esz].view(dtype)
        self.nbytes = max(n, 8) * esz

    def intact(self):
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


@pytest.mark.parametrize("stage", [1, 2, 3])
def test_no_write_outside_buffers(stage):
    rng = np.random.default_rng(stage)
    shapes = [(int(x),) for x in rng.integers(1, 20000, size=12)] + [(3,), (0,), (8191,), (8193,)]
    W = 3
    z = ZeroStep(shapes, W, stage, 40_000, wl.BF16, wl.BF16)
    n = z.np
    f32, bf16 = torch.float32, torch.bfloat16
    bufs = {k: Guarded(n, f32) for k in ("master", "m", "v")}
    bufs["params"] = Guarded(n, bf16)
    bufs["scratch"] = Guarded(n, bf16)
    outs = [Guarded(n, bf16) for _ in range(W)]
    z.bind(bufs["master"].t, bufs["m"].t, bufs["v"].t, bufs["params"].t,
           bufs["scratch"].t if stage != 1 else None)
    if stage == 1:
        z.allreduce_out = [o.t for o in outs]
    numel = wl.numels(shapes)
    master0 = Guarded(n, f32)
    master0.t[:n].copy_(wl.master_init(z.offsets, numel, n, 0.02, 1, device="cuda"))
    z.init(master0.t, init_scale=8.0, dynamic=True)
    hp = Hparams()
    stream = torch.cuda.current_stream().cuda_stream
    for step in range(3):
        grads = [wl.flat_grads(z.offsets, numel, n, 1e-3, wl.grad_seed(170, r, step), wl.BF16,
                               device="cuda") for r in range(W)]
        if step == 0:
            z.step(grads, hp)
        elif step == 1:
            per = [[grads[r][off:off + k] if k else None for off, k in zip(z.offsets, numel)]
                   for r in range(W)]
            z.step_tensors(per, hp)
        else:
            z.step_host([g.cpu().pin_memory() for g in grads], grads, hp)
    z.step_per_tensor_launch(grads, hp)
    # gathers, exports, imports, accumulation
    reps = [[Guarded(k, bf16) for k in numel] for _ in range(2)]
    z.gather([[g.t[:k] if k else g.t for g, k in zip(row, numel)] for row in reps])
    flat_exp = [Guarded(n, f32) for _ in range(3)]
    abi.zero_state_export(z.handle, *[b.t.data_ptr() for b in flat_exp], stream)
    abi.zero_state_import(z.handle, *[b.t.data_ptr() for b in flat_exp], stream)
    pm = [Guarded(sum(numel), f32) for _ in range(3)]
    abi.zero_state_export_params(z.handle, *[b.t.data_ptr() for b in pm], stream)
    abi.zero_state_import_params(z.handle, *[b.t.data_ptr() for b in pm], stream)
    mains = [Guarded(n, f32) for _ in range(W)]
    abi.zero_accumulate(z.handle, [g.data_ptr() for g in grads], wl.BF16,
                        [b.t.data_ptr() for b in mains], True, stream)
    bucket_dst = Guarded(n, bf16)
    if stage == 3:
        for b in range(z.info.n_buckets):
            abi.zero_gather_bucket(z.handle, b, bucket_dst.t.data_ptr(), stream)
    red = Guarded(n, bf16)
    nsq = Guarded(1, torch.float64)
    ovf = Guarded(1, torch.int32)
    abi.zero_reduce_norm_noalloc([g.data_ptr() for g in grads], n, wl.BF16, -1, red.t.data_ptr(),
                                 nsq.t.data_ptr(), ovf.t.data_ptr(), stream)
    torch.cuda.synchronize()
    assert z.scaler_state()["steps"] == 4
    everything = list(bufs.values()) + outs + [master0] + [g for row in reps for g in row] + \
        flat_exp + pm + mains + [bucket_dst, red, nsq, ovf]
    bad = [i for i, g in enumerate(everything) if not g.intact()]
    assert not bad, bad
    z.close()
