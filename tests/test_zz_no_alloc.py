"""The allocation-free reduce/norm entry point against the regular step.

zero_reduce_norm_noalloc serves callers that cannot allocate device memory
(for instance while a CUDA graph is being captured elsewhere in the process,
or when every byte of device memory was handed out at start-up): it keeps its
scratch in a fixed array inside the library. This test calls it through the C
ABI twice in a row, on different inputs, and checks each result against what
zero_step computed on the same gradients: the reduced values bit for bit, the
overflow flag exactly, and the squared norm within the relative tolerance the
parity tests use for the norm (1e-6 on its square root).

Kept in a file of its own that pytest collects last, so a run that stops at
the first failure has already run every other test.
"""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from _parity import to_np
from mixed_precision_gb300 import ZeroError
from mixed_precision_gb300 import _abi as abi
from mixed_precision_gb300.engine import Hparams, ZeroStep

pytestmark = pytest.mark.gpu


def test_noalloc_matches_step_on_two_calls():
    shapes = wl.qwen3_0_6b_shapes(vocab=1000, hidden=128, layers=2, q_dim=256, kv_dim=128,
                                  ffn=384, head_dim=32)
    W = 4
    z = ZeroStep(shapes, W, 2, 80_000, wl.BF16, wl.BF16)
    z.allocate()
    numel = wl.numels(shapes)
    z.init(wl.master_init(z.offsets, numel, z.np, 0.02, wl.master_seed(7), device="cuda"))
    perm = np.empty(z.np, np.int64)  # flat index of every rank-major shard position
    for b in range(z.info.n_buckets):
        for r in range(W):
            f0, s0, ln = abi.zero_shard_range(z.handle, b, r)
            perm[s0:s0 + ln] = np.arange(f0, f0 + ln)
    real = np.zeros(z.np, bool)
    for off, n in zip(z.offsets, numel):
        real[off:off + n] = True

    reduced = torch.empty(z.np, dtype=torch.bfloat16, device="cuda")
    norm_sq = torch.empty(1, dtype=torch.float64, device="cuda")
    ovf = torch.empty(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    # Sizes beyond the fixed scratch are refused before any device work.
    with pytest.raises(ZeroError) as e:
        abi.zero_reduce_norm_noalloc([reduced.data_ptr()] * W, (1 << 32) + 1, wl.BF16, -1, 0,
                                     norm_sq.data_ptr(), ovf.data_ptr(), stream)
    assert e.value.code == abi.ZERO_ERR_INVALID

    for call in range(2):
        # padding zero-filled: the no-alloc entry point reduces the plain range
        grads = [wl.flat_grads(z.offsets, numel, z.np, 1e-3, wl.grad_seed(70, r, call), wl.BF16,
                               device="cuda", pad_fill=0.0) for r in range(W)]
        if call == 1:
            grads[2][z.offsets[3] + 5] = float("inf")
        z.step(grads, Hparams())
        st = z.scaler_state()
        abi.zero_reduce_norm_noalloc([g.data_ptr() for g in grads], z.np, wl.BF16, -1,
                                     reduced.data_ptr(), norm_sq.data_ptr(), ovf.data_ptr(), stream)
        torch.cuda.synchronize()
        assert int(ovf.item()) == st["overflow"] == call
        got_sq, ref_sq = float(norm_sq.item()), st["norm_sq_raw"]
        if call == 0:
            assert abs(math.sqrt(got_sq) - math.sqrt(ref_sq)) <= 1e-6 * math.sqrt(ref_sq)
        else:
            assert math.isinf(got_sq) and math.isinf(ref_sq)
        got = to_np(reduced)
        exp = np.zeros(z.np, np.uint16)
        exp[perm] = to_np(z.scratch)[:z.np]
        assert np.array_equal(got[real], exp[real])
        assert np.all(got[~real] == 0)
    z.close()
