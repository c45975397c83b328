"""The allocation-free reduce/norm entry point against the regular step and
against the oracle.

zero_reduce_norm_noalloc serves callers that cannot allocate device memory
(for instance while a CUDA graph is being captured elsewhere in the process,
or when every byte of device memory was handed out at start-up): it keeps its
scratch in a fixed array inside the library. The first test calls it through
the C ABI twice in a row, on different inputs, and checks each result against
what zero_step computed on the same gradients: the reduced values bit for
bit, the overflow flag exactly, and the squared norm within the relative
tolerance the parity tests use for the norm (1e-6 on its square root). The
others check it against the oracle's reduce and overflow/sum of squares over
the same plain range, across world sizes, dtypes and ragged lengths.

Kept in a file of its own that pytest collects last, so a run that stops at
the first failure has already run every other test.
"""
import math

import numpy as np
import pytest
import torch

import oracle
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


def _draw(n, dtype, seed, sigma=1e-3):
    """n seeded N(0, sigma) values in dtype, on the CPU (flat, no layout)."""
    return wl.normal(n, sigma, seed, dtype)


def _call(grads_dev, n, gdt, cdt, reduced):
    norm_sq = torch.empty(1, dtype=torch.float64, device="cuda")
    ovf = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    abi.zero_reduce_norm_noalloc([g.data_ptr() for g in grads_dev], n, gdt, cdt,
                                 reduced.data_ptr() if reduced is not None else 0,
                                 norm_sq.data_ptr(), ovf.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return float(norm_sq.item()), int(ovf.item())


def _check_against_oracle(grads_cpu, n, gdt, cdt, with_out=True):
    """One call on [0, n) against the oracle's reduce and overflow/sum of
    squares over the same plain range (no padding mask): reduced values bit
    for bit, the flag exactly, the norm within 1e-6 (on its square root).
    The element after the range stays as it was."""
    cdt_eff = gdt if cdt < 0 else cdt
    dev = [g.cuda() for g in grads_cpu]
    guard_val = 0x5A5A
    bits_t = torch.int32 if cdt_eff == wl.F32 else torch.int16
    reduced = None
    if with_out:
        reduced = torch.empty(n + 8, dtype=wl.TORCH_DTYPE[cdt_eff], device="cuda")
        reduced.view(bits_t).fill_(guard_val)
    got_sq, got_ovf = _call(dev, n, gdt, cdt, reduced)
    host = [to_np(g[:n]) for g in grads_cpu]
    exp = oracle.reduce(host, gdt, cdt_eff, 0, n, None)
    exp_ovf, exp_sq = oracle.overflow_sumsq(exp, cdt_eff, None)
    assert got_ovf == exp_ovf
    if exp_ovf:
        assert not math.isfinite(got_sq)
    else:
        assert abs(math.sqrt(got_sq) - math.sqrt(exp_sq)) <= 1e-6 * max(math.sqrt(exp_sq), 1e-300)
    if with_out:
        raw = reduced.view(bits_t).cpu().numpy()
        exp_bits = exp.view(np.int32) if cdt_eff == wl.F32 else exp.view(np.int16)
        assert np.array_equal(raw[:n], exp_bits)
        assert np.all(raw[n:] == guard_val)  # nothing written past n
    return exp_ovf, exp_sq


@pytest.mark.parametrize("W", [1, 3, 8])
@pytest.mark.parametrize("gdt,cdt", [(wl.BF16, -1), (wl.F16, -1), (wl.BF16, wl.F32),
                                     (wl.F16, wl.F32), (wl.F32, wl.F32)])
@pytest.mark.parametrize("n", [1, 7, 65_535, 65_537, 3 * 65_536 + 5])
def test_noalloc_matches_oracle(W, gdt, cdt, n):
    grads = [_draw(n + 16, gdt, wl.grad_seed(71, r, n)) for r in range(W)]
    _check_against_oracle(grads, n, gdt, cdt)


def test_noalloc_fp16_overflow_only_after_the_sum():
    """Finite fp16 inputs whose fp16 sum exceeds 65504: the flag is set with an
    fp16 communication dtype and not with fp32 (the reduced value decides)."""
    n, W = 3 * 65_536 + 5, 3
    grads = [_draw(n + 16, wl.F16, wl.grad_seed(72, r)) for r in range(W)]
    for g in grads:
        g[65_536 + 17] = 40000.0
    ovf16, _ = _check_against_oracle(grads, n, wl.F16, -1)
    ovf32, _ = _check_against_oracle(grads, n, wl.F16, wl.F32)
    assert ovf16 == 1 and ovf32 == 0


def test_noalloc_without_reduced_output():
    n, W = 65_537, 3
    grads = [_draw(n + 16, wl.BF16, wl.grad_seed(73, r)) for r in range(W)]
    _check_against_oracle(grads, n, wl.BF16, -1, with_out=False)


def test_noalloc_more_chunks_than_blocks():
    """700 chunks of 65,536 elements and a 13-element tail: far more chunks than
    the grid's blocks, so blocks loop over chunks and the last block sums more
    partials than there are blocks. Then a ragged n (not a multiple of 8) on
    the same buffers, leaving the element after it untouched."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = 700 * 65_536 + 13
    assert (n + 65_535) // 65_536 > 4 * sms
    grads = [_draw(n + 16, wl.BF16, wl.grad_seed(74, r)) for r in range(2)]
    _check_against_oracle(grads, n, wl.BF16, -1)
    _check_against_oracle(grads, n - 5, wl.BF16, -1)
