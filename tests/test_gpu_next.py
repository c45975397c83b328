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
