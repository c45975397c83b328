"""Pins of the host oracle against what the pages and the mathematics fix.

Each test pins one step of the oracle to something other than the oracle
itself: the pages' printed example values (tests/golden/), closed forms,
invariants, brute force on tiny inputs, or torch's own CPU dtype casts (a
library routine). CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as wl

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Bit-level casts (cast-out / all-gather step, reduced communication values)
# ---------------------------------------------------------------------------

def _torch_bits(x32: np.ndarray, dtype) -> np.ndarray:
    return torch.from_numpy(x32).to(dtype).view(torch.int16).numpy().view(np.uint16)


def _compare_encode(orc, bits: np.ndarray, dt):
    x = bits.view(np.float32)
    ours = orc.encode(x, dt)
    ref = _torch_bits(x, wl.TORCH_DTYPE[dt])
    diff = ours != ref
    if diff.any():
        # Only NaN encodings may differ, and both must be NaN.
        exp_all = 0x7F80 if dt == wl.BF16 else 0x7C00
        man = 0x007F if dt == wl.BF16 else 0x03FF
        nan_in = np.isnan(x[diff])
        ours_nan = ((ours[diff] & exp_all) == exp_all) & ((ours[diff] & man) != 0)
        ref_nan = ((ref[diff] & exp_all) == exp_all) & ((ref[diff] & man) != 0)
        assert nan_in.all() and ours_nan.all() and ref_nan.all()


@pytest.mark.parametrize("dt", [wl.BF16, wl.F16])
def test_encode_matches_torch_cast(orc, dt):
    """RNE fp32 -> bf16/fp16 against torch's CPU cast (NaN: both NaN).

    Default: every 2^16 high half with the low halves that decide rounding
    (0, 1, just below/at/above the tie for both formats, all ones), plus a
    prime-stride sweep of all 2^32 patterns. ZERO_EXHAUSTIVE=1 checks all 2^32
    patterns (a few minutes)."""
    if os.environ.get("ZERO_EXHAUSTIVE") == "1":
        chunk = 1 << 26
        for start in range(0, 1 << 32, chunk):
            _compare_encode(orc, np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32), dt)
        return
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x2000, 0x3000, 0x7FFF, 0x8000, 0x8001,
                     0x9000, 0xEFFF, 0xF000, 0xF001, 0xFFFF], dtype=np.uint32)
    _compare_encode(orc, (hi[:, None] | lows[None, :]).ravel(), dt)
    _compare_encode(orc, (np.arange(0, 1 << 32, 4099, dtype=np.uint64)).astype(np.uint32), dt)


@pytest.mark.parametrize("dt", [wl.BF16, wl.F16])
def test_decode_matches_torch_exhaustive(orc, dt):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = orc.decode(bits, dt)
    ref = torch.from_numpy(bits.view(np.int16)).view(wl.TORCH_DTYPE[dt]).float().numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    same = (ours.view(np.uint32) == ref.view(np.uint32)) | both_nan
    assert same.all()


def test_encode_fp16_boundaries(orc):
    """Hand-checked binary16 facts: largest finite, the overflow tie, the
    smallest subnormal and its round-to-zero tie."""
    x = np.array([65504.0, 65519.996, 65520.0, 2.0 ** -24, 2.0 ** -25, 1.5 * 2.0 ** -25],
                 dtype=np.float32)
    assert orc.encode(x, wl.F16).tolist() == [0x7BFF, 0x7BFF, 0x7C00, 0x0001, 0x0000, 0x0001]


# ---------------------------------------------------------------------------
# a1: layout
# ---------------------------------------------------------------------------

def _check_layout(L, numel, world, cap):
    off, pb = L.param_offset, L.param_bucket
    bs, bl = L.bucket_start, L.bucket_len
    # buckets tile [0, np) contiguously, each padded to a multiple of W*128
    assert bs[0] == 0
    assert np.all(bs[1:] == bs[:-1] + bl[:-1])
    assert bs[-1] + bl[-1] == L.np_total
    assert np.all(bl % (world * 128) == 0)
    # parameters in order, 64-aligned, non-overlapping, inside their bucket
    assert np.all(off % 64 == 0)
    ends = off + numel
    assert np.all(off[1:] >= ends[:-1])
    for p in range(len(numel)):
        b = pb[p]
        assert bs[b] <= off[p] and ends[p] <= bs[b] + bl[b]
        if p:
            assert pb[p] in (pb[p - 1], pb[p - 1] + 1)
    # greedy bucket rule: a bucket holding >= 2 params spans <= cap; the first
    # param of a new bucket would have pushed the previous bucket past cap
    for b in range(len(bs)):
        members = np.nonzero(pb == b)[0]
        if len(members) >= 2:
            assert ends[members[-1]] - bs[b] <= cap
        if b > 0 and len(members):
            first = members[0]
            prev_start = bs[b - 1]
            would_be = -(-ends[first - 1] // 64) * 64 + numel[first] - prev_start
            assert would_be > cap
    # padding is minimal: each bucket length is the smallest multiple of W*128
    for b in range(len(bs)):
        members = np.nonzero(pb == b)[0]
        span = (ends[members[-1]] - bs[b]) if len(members) else 0
        assert bl[b] == -(-span // (world * 128)) * (world * 128)
    # every real index lies in exactly one (bucket, rank) shard, equal shard lengths
    owner = np.full(L.np_total, -1, dtype=np.int64)
    for b, r, f0, s0, ln in L.shard_ranges():
        assert ln == bl[b] // world
        assert np.all(owner[f0:f0 + ln] == -1)
        owner[f0:f0 + ln] = r
    assert np.all(owner >= 0)
    perm = L.flat_of_shard()
    assert np.array_equal(np.sort(perm), np.arange(L.np_total))


def test_layout_bruteforce_tiny(orc):
    rng = np.random.default_rng(7)
    for _ in range(300):
        n = int(rng.integers(1, 9))
        numel = rng.integers(0, 700, size=n)
        world = int(rng.integers(1, 9))
        grad_bytes = int(rng.choice([2, 4]))
        bucket_bytes = int(rng.choice([2, 64, 500, 1024, 4096, 1 << 20]))
        L = orc.layout(numel, world, bucket_bytes, grad_bytes)
        _check_layout(L, numel, world, bucket_bytes // grad_bytes)


def test_layout_known_small_case(orc):
    """Worked by hand: sizes 100, 30, 200 with W=2, cap 256 elements (512 B of bf16).
    p0 at 0; p1 at 128 (span 158 <= 256); p2 would end at 192+200 > 256, so a new
    bucket: bucket 0 = [0, 256) (158 padded to 256), p2 at 256, bucket 1 = [256, 512)."""
    L = orc.layout([100, 30, 200], 2, 512, 2)
    assert L.param_offset.tolist() == [0, 128, 256]
    assert L.bucket_start.tolist() == [0, 256]
    assert L.bucket_len.tolist() == [256, 256]
    assert list(L.shard_ranges()) == [(0, 0, 0, 0, 128), (1, 0, 256, 128, 128),
                                      (0, 1, 128, 256, 128), (1, 1, 384, 384, 128)]


def test_layout_bucket_boundary_is_strict(orc):
    """A bucket closes only when the next parameter would take its span past
    the cap: a parameter ending exactly at the cap stays in the bucket.
    Cap 256 elements (512 B of bf16), W=2: sizes 128 + 128 end at 256 -> one
    bucket [0, 256); sizes 128 + 129 would end at 257 -> the second parameter
    opens bucket 1 at 256 (129 elements padded to 2 * 128)."""
    L = orc.layout([128, 128], 2, 512, 2)
    assert L.param_offset.tolist() == [0, 128]
    assert L.bucket_start.tolist() == [0] and L.bucket_len.tolist() == [256]
    L = orc.layout([128, 129], 2, 512, 2)
    assert L.param_offset.tolist() == [0, 256]
    assert L.bucket_start.tolist() == [0, 256] and L.bucket_len.tolist() == [256, 256]


def test_layout_workload_sizes(orc):
    for name, n_real in [("tiny", 327936), ("qwen3_0.6b_bf16_w2", 596049920),
                         ("moe_3.9b_bf16_w4", 3890479104)]:
        w = wl.workload(name)
        numel = np.array(wl.numels(w.shapes), dtype=np.int64)
        assert numel.sum() == n_real
        L = orc.layout(numel, w.world, w.bucket_bytes, wl.ELEM_BYTES[w.grad_dtype])
        assert L.np_total >= n_real
        assert L.np_total % (w.world * 128) == 0


# ---------------------------------------------------------------------------
# a2: reduce
# ---------------------------------------------------------------------------

def test_reduce_rank_order_and_rounding(orc):
    """(1 + 2^-24) + 2^-24 rounds to 1 twice (ties to even) in fp32; the
    rank order is what the definition fixes, so the result is exactly 1.0."""
    g = [np.array([1.0], np.float32), np.array([2.0 ** -24], np.float32),
         np.array([2.0 ** -24], np.float32)]
    assert orc.reduce(g, wl.F32, wl.F32)[0] == np.float32(1.0)
    g2 = [g[1], g[2], g[0]]
    assert orc.reduce(g2, wl.F32, wl.F32)[0] == np.float32(1.0 + 2.0 ** -23)


def test_reduce_world1_is_identity(orc):
    rng = np.random.default_rng(3)
    for dt in (wl.BF16, wl.F16):
        bits = rng.integers(0, 1 << 16, size=5000).astype(np.uint16)
        out = orc.reduce([bits], dt, dt)
        fin = np.isfinite(orc.decode(bits, dt))
        assert np.array_equal(out[fin], bits[fin])


def test_reduce_exact_small_integers(orc):
    """Integer-valued gradients sum exactly; 3 ranks of bf16."""
    a = np.arange(-50, 50, dtype=np.float32)
    g = [orc.encode(a, wl.BF16), orc.encode(2 * a, wl.BF16), orc.encode(-a + 1, wl.BF16)]
    out = orc.decode(orc.reduce(g, wl.BF16, wl.BF16), wl.BF16)
    assert np.array_equal(out, 2 * a + 1)


def test_reduce_fp16_overflow_after_sum(orc):
    g = [orc.encode(np.array([40000.0, 1.0], np.float32), wl.F16)] * 2
    r = orc.reduce(g, wl.F16, wl.F16)
    ovf, _ = orc.overflow_sumsq(r, wl.F16)
    assert r[0] == 0x7C00 and ovf == 1
    r32 = orc.reduce(g, wl.F16, wl.F32)
    assert r32[0] == np.float32(80000.0)
    assert orc.overflow_sumsq(r32, wl.F32)[0] == 0


def test_reduce_skips_padding(orc):
    g = [np.array([1.0, np.nan, 2.0], np.float32)] * 2
    mask = np.array([1, 0, 1], np.uint8)
    r = orc.reduce(g, wl.F32, wl.F32, real_mask=mask)
    assert r.tolist() == [2.0, 0.0, 4.0]
    assert orc.overflow_sumsq(r, wl.F32, mask) == (0, 20.0)


# ---------------------------------------------------------------------------
# a4/a5: norm, clip, loss scale
# ---------------------------------------------------------------------------

def test_norm_and_clip_closed_form(orc):
    """All N reduced values equal a: norm = |a| sqrt(N) / (S D)."""
    n, a, S, W = 4096, 3.0, 8.0, 4
    hp = orc.Hparams(max_grad_norm=1.0)
    sc = orc.Scaler(scale=S)
    r = np.full(n, a, np.float32)
    ovf, ss = orc.overflow_sumsq(r, wl.F32)
    info = orc.finalize(ss, ovf, W, hp, sc)
    norm = a * math.sqrt(n) / (S * W)
    assert info.grad_norm == pytest.approx(norm, rel=1e-15)
    assert info.clip_coef == pytest.approx(1.0 / (norm + 1e-6), rel=1e-15)
    assert info.gscale == pytest.approx(info.clip_coef / (S * W), rel=1e-15)
    # below the threshold the coefficient is exactly 1; switched off also 1
    info2 = orc.finalize(ss, 0, W, orc.Hparams(max_grad_norm=100.0), orc.Scaler(scale=S))
    assert info2.clip_coef == 1.0
    info3 = orc.finalize(ss, 0, W, orc.Hparams(max_grad_norm=0.0), orc.Scaler(scale=S))
    assert info3.clip_coef == 1.0
    # divisor 1 is the plain sum
    info4 = orc.finalize(ss, 0, W, orc.Hparams(max_grad_norm=0.0, grad_divisor=1.0),
                         orc.Scaler(scale=S))
    assert info4.grad_norm == pytest.approx(a * math.sqrt(n) / S, rel=1e-15)


def _run_scaler(orc, ovf_seq, **kw):
    sc = orc.Scaler(dynamic=True, **kw)
    traj = []
    for o in ovf_seq:
        scale_used = sc.scale
        info = orc.finalize(1.0, o, 2, orc.Hparams(), sc)
        traj.append((scale_used, sc.t, info.skipped, sc.scale, sc.counter))
    return traj


def test_scaler_tiny_trajectory(orc):
    """Four steps from 2^16, an overflow at step 3: scales used 2^16, 2^16, 2^16
    (skipped), 2^15; Adam t after each step 1, 2, 2, 3."""
    traj = _run_scaler(orc, [0, 0, 1, 0], scale=2.0 ** 16)
    assert [t[0] for t in traj] == [2.0 ** 16, 2.0 ** 16, 2.0 ** 16, 2.0 ** 15]
    assert [t[1] for t in traj] == [1, 2, 2, 3]
    assert [t[2] for t in traj] == [0, 0, 1, 0]
    assert traj[-1][3] == 2.0 ** 15


def test_scaler_periodic_overflow_never_grows(orc):
    """Overflow at steps 50/100/150/200 with N = 1000: four halvings from 2^16."""
    seq = [1 if (s % 50 == 0) else 0 for s in range(1, 201)]
    traj = _run_scaler(orc, seq, scale=2.0 ** 16, growth_interval=1000)
    assert traj[-1][3] == 2.0 ** 12
    assert max(t[3] for t in traj) == 2.0 ** 16
    assert traj[-1][1] == 196


def test_scaler_growth_after_n_clean(orc):
    seq = [1] + [0] * 25
    traj = _run_scaler(orc, seq, scale=2.0 ** 10, growth_interval=10)
    scales_after = [t[3] for t in traj]
    assert scales_after[0] == 2.0 ** 9
    assert scales_after[1:10] == [2.0 ** 9] * 9
    assert scales_after[10] == 2.0 ** 10       # 10th clean step after the overflow
    assert scales_after[20] == 2.0 ** 11
    assert traj[10][4] == 0 and traj[11][4] == 1


def test_scaler_overflow_resets_clean_count(orc):
    """Seven clean steps, an overflow, then clean steps with N = 10: the
    overflow resets the clean count, so growth comes on the 10th clean step
    after it (not the 3rd, which a kept count of 7 would give)."""
    seq = [0] * 7 + [1] + [0] * 12
    traj = _run_scaler(orc, seq, scale=2.0 ** 10, growth_interval=10)
    after = [t[3] for t in traj]
    assert after[6] == 2.0 ** 10 and traj[6][4] == 7
    assert after[7] == 2.0 ** 9 and traj[7][4] == 0
    assert after[8:17] == [2.0 ** 9] * 9
    assert after[17] == 2.0 ** 10 and traj[17][4] == 0


def test_scaler_static_never_grows(orc):
    """Static loss scaling: the scale stays put however many clean steps pass."""
    sc = orc.Scaler(scale=4.0, dynamic=False, growth_interval=2)
    for _ in range(7):
        orc.finalize(1.0, 0, 2, orc.Hparams(), sc)
    assert sc.scale == 4.0 and sc.t == 7


def test_scaler_min_scale_and_static(orc):
    traj = _run_scaler(orc, [1, 1, 1], scale=2.0, min_scale=1.0)
    assert [t[3] for t in traj] == [1.0, 1.0, 1.0]
    sc = orc.Scaler(scale=1.0, dynamic=False)
    for o in [1, 0, 1]:
        orc.finalize(1.0, o, 2, orc.Hparams(), sc)
    assert sc.scale == 1.0 and sc.t == 1


# ---------------------------------------------------------------------------
# a6: AdamW
# ---------------------------------------------------------------------------

def _adamw_once(orc, g, p, m, v, hp, t0=0):
    info = orc.Info(0, 0, 0.0, 0.0, 1.0, 1.0, 1 - hp.beta1 ** (t0 + 1), 1 - hp.beta2 ** (t0 + 1))
    orc.adamw(g.astype(np.float32), wl.F32, hp, info, p, m, v)


def test_adamw_first_step_closed_form(orc):
    """From m = v = 0 at t = 1: m1 = (1-b1) g, v1 = (1-b2) g^2 and
    p1 = p0 (1 - lr wd) - lr g / (|g| + eps)."""
    rng = np.random.default_rng(11)
    g = rng.normal(0, 1e-2, 1000).astype(np.float32)
    p0 = rng.normal(0, 0.02, 1000).astype(np.float32)
    hp = orc.Hparams(lr=1e-3, weight_decay=0.01, eps=1e-8)
    p, m, v = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    _adamw_once(orc, g, p, m, v, hp)
    g64 = g.astype(np.float64)
    np.testing.assert_allclose(m, 0.1 * g64, rtol=2e-7)
    np.testing.assert_allclose(v, 0.001 * g64 ** 2, rtol=2e-7)
    expect = p0.astype(np.float64) * (1 - 1e-5) - 1e-3 * g64 / (np.abs(g64) + 1e-8)
    np.testing.assert_allclose(p, expect, rtol=1e-6, atol=1e-12)
    # Second step with the same gradient: bias correction makes m_hat = g and
    # v_hat = g^2 again, so the same closed form holds from p1.
    p1 = p.copy()
    info = orc.Info(0, 0, 0.0, 0.0, 1.0, 1.0, 1 - 0.9 ** 2, 1 - 0.999 ** 2)
    orc.adamw(g, wl.F32, hp, info, p, m, v)
    expect2 = p1.astype(np.float64) * (1 - 1e-5) - 1e-3 * g64 / (np.abs(g64) + 1e-8)
    np.testing.assert_allclose(p, expect2, rtol=1e-6, atol=1e-12)
    np.testing.assert_allclose(m, 0.19 * g64, rtol=4e-7)
    np.testing.assert_allclose(v, 0.001999 * g64 ** 2, rtol=4e-7)


def test_adamw_skipped_step_touches_nothing(orc):
    """A skipped step (overflow) leaves master, m and v bit for bit, even when
    the update is called with it."""
    rng = np.random.default_rng(31)
    g = rng.standard_normal(64).astype(np.float32)
    p = rng.standard_normal(64).astype(np.float32)
    m = (0.1 * rng.standard_normal(64)).astype(np.float32)
    v = (0.01 * rng.random(64)).astype(np.float32)
    p0, m0, v0 = p.copy(), m.copy(), v.copy()
    info = orc.Info(1, 1, float("inf"), float("inf"), 0.0, 0.0, 0.0, 0.0)
    orc.adamw(g, wl.F32, orc.Hparams(), info, p, m, v)
    assert np.array_equal(p.view(np.uint32), p0.view(np.uint32))
    assert np.array_equal(m.view(np.uint32), m0.view(np.uint32))
    assert np.array_equal(v.view(np.uint32), v0.view(np.uint32))


def test_adam_constant_gradient_moves_lr_per_step(orc):
    """Bias-corrected Adam under a constant gradient g: m_t = (1 - b1^t) g and
    v_t = (1 - b2^t) g^2, so the corrected moments are exactly g and g^2 and
    every step moves the parameter by lr * g / (|g| + eps) (weight decay off).
    Runs the composed step (finalize's t and bias corrections, then the update)
    for six steps; a correction from the wrong beta or the wrong t moves by a
    different amount."""
    n = 64
    g = np.tile(np.array([0.5, -0.25, 1.0, -2.0], np.float32), n // 4)
    grads = [orc.encode(g, wl.BF16)]
    p0 = np.linspace(-1.0, 1.0, n).astype(np.float32)
    master, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    params = np.zeros(n, np.uint16)
    hp = orc.Hparams(lr=1e-3, weight_decay=0.0, max_grad_norm=0.0)
    sc = orc.Scaler()
    step = hp.lr * g.astype(np.float64) / (np.abs(g.astype(np.float64)) + hp.eps)
    for k in range(1, 7):
        orc.ddp_step(grads, wl.BF16, wl.BF16, wl.BF16, master, m, v, params, hp, sc)
        expect = p0.astype(np.float64) - k * step
        # fp32 storage of master/m/v: a few ulps of |p| per step at most
        tol = k * 4 * np.spacing(np.abs(expect).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(master - expect) <= tol), (k, np.abs(master - expect).max())
    assert sc.t == 6


def test_adamw_zero_grad_pure_decay(orc):
    p0 = np.random.default_rng(5).normal(0, 1, 257).astype(np.float32)
    p, m, v = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    hp = orc.Hparams(lr=0.5, weight_decay=0.1)
    _adamw_once(orc, np.zeros_like(p0), p, m, v, hp)
    assert np.all(m == 0) and np.all(v == 0)
    assert np.array_equal(p, (p0.astype(np.float64) * (1 - 0.05)).astype(np.float32))


def test_adamw_gscale_applies_unscale(orc):
    """gscale multiplies the reduced value: r = 2^16 g with gscale 2^-16 is the
    same update as r = g with gscale 1 (both exact powers of two)."""
    rng = np.random.default_rng(9)
    g = rng.normal(0, 1e-3, 300).astype(np.float32)
    hp = orc.Hparams()
    p0 = rng.normal(0, 0.02, 300).astype(np.float32)
    a = [p0.copy(), np.zeros_like(p0), np.zeros_like(p0)]
    b = [p0.copy(), np.zeros_like(p0), np.zeros_like(p0)]
    i1 = orc.Info(0, 0, 0.0, 0.0, 1.0, 1.0, 0.1, 0.001)
    i2 = orc.Info(0, 0, 0.0, 0.0, 1.0, 2.0 ** -16, 0.1, 0.001)
    orc.adamw(g, wl.F32, hp, i1, *a)
    orc.adamw((g * 2.0 ** 16).astype(np.float32), wl.F32, hp, i2, *b)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ---------------------------------------------------------------------------
# Composed steps
# ---------------------------------------------------------------------------

def test_sharded_sgd_golden(orc):
    """The page's sharded-SGD example through the oracle's reduce, shard
    ranges and gather order, with a plain SGD update applied in the test."""
    gd = _gold("sharded_sgd.json")
    params = np.array(gd["parameters"], np.float32)
    grads = [np.array(g, np.float32) for g in gd["gradients"]]
    W = len(grads)
    L = orc.layout([params.size], W, 1 << 20, 4)
    mask = L.real_mask()
    flat_g = []
    for g in grads:
        f = np.zeros(L.np_total, np.float32)
        f[:params.size] = g
        flat_g.append(f)
    info = orc.finalize(1.0, 0, W, orc.Hparams(max_grad_norm=0.0), orc.Scaler())
    gathered = np.zeros(L.np_total, np.float32)
    pflat = np.zeros(L.np_total, np.float32)
    pflat[:params.size] = params
    for b, r, f0, s0, ln in L.shard_ranges():
        red = orc.decode(orc.reduce(flat_g, wl.F32, wl.F32, f0, f0 + ln, mask), wl.F32)
        gathered[f0:f0 + ln] = pflat[f0:f0 + ln] - np.float32(gd["lr"]) * (red * np.float32(info.gscale))
    np.testing.assert_allclose(gathered[:params.size], gd["expected_updated"], rtol=1e-6)


def test_token_weighted_divisor_golden(orc):
    """grad_divisor is a plain scalar: replica mean (D = W) reproduces the
    page's wrong 0.5; caller-weighted gradients with D = 1 give 0.75."""
    gd = _gold("token_weighted.json")
    lr, start = gd["lr"], gd["start"]
    means, tokens = gd["local_means"], gd["valid_tokens"]
    W = len(means)

    def sgd(grads, divisor):
        info = orc.finalize(1.0, 0, W, orc.Hparams(max_grad_norm=0.0, grad_divisor=divisor),
                            orc.Scaler())
        red = orc.reduce([np.array([g], np.float32) for g in grads], wl.F32, wl.F32)
        return start - lr * float(red[0]) * info.gscale

    assert sgd(means, 0.0) == pytest.approx(gd["expected_after_replica_mean"])
    weighted = [m * t / sum(tokens) for m, t in zip(means, tokens)]
    assert sgd(weighted, 1.0) == pytest.approx(gd["expected_after_token_weighted"])


def _random_problem(orc, rng, numel, W, gdt, bucket_bytes, sigma=1e-3):
    L = orc.layout(numel, W, bucket_bytes, wl.ELEM_BYTES[gdt])
    n = int(np.sum(numel))
    per_param = [rng.normal(0, sigma, n).astype(np.float32) for _ in range(W)]
    per_param = [orc.encode(x, gdt) for x in per_param]
    flat = []
    for x in per_param:
        f = np.full(L.np_total, 0x7FFF if gdt != wl.F32 else 0, dtype=x.dtype)  # NaN padding
        if gdt == wl.F32:
            f[:] = np.float32(np.nan)
        at = 0
        for off, k in zip(L.param_offset, numel):
            f[off:off + k] = x[at:at + k]
            at += k
        flat.append(f)
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    return L, per_param, flat, p0


def _to_shards(L, numel, x_param_major, fill=0.0):
    flat = np.full(L.np_total, fill, np.float32)
    at = 0
    for off, k in zip(L.param_offset, numel):
        flat[off:off + k] = x_param_major[at:at + k]
        at += k
    return flat[L.flat_of_shard()].copy()


def _from_shards(L, numel, shards):
    flat = np.empty(L.np_total, np.float32)
    flat[L.flat_of_shard()] = shards
    return np.concatenate([flat[off:off + k] for off, k in zip(L.param_offset, numel)])


@pytest.mark.parametrize("W,stage,gdt,cdt,bucket", [
    (1, 2, wl.BF16, wl.BF16, 1 << 20), (2, 2, wl.BF16, wl.BF16, 4096), (3, 1, wl.F16, wl.F16, 2048),
    (4, 2, wl.F16, wl.F32, 8192), (8, 2, wl.BF16, wl.BF16, 1000), (5, 1, wl.F32, wl.BF16, 3000)])
def test_partitioned_equals_unpartitioned(orc, W, stage, gdt, cdt, bucket):
    """ZeRO changes memory, not the algorithm: the partitioned step equals the
    DDP step. With clipping off the fp32 state is bit-identical; with clipping
    on, the two norms differ only in fp64 summation order."""
    rng = np.random.default_rng(100 + W)
    numel = rng.integers(1, 900, size=9)
    L, per_param, flat, p0 = _random_problem(orc, rng, numel, W, gdt, bucket)
    for clip in (0.0, 1e-6):
        hp = orc.Hparams(max_grad_norm=clip)
        sc_d, sc_z = orc.Scaler(scale=4.0), orc.Scaler(scale=4.0)
        md, mm, vd = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
        pd = np.zeros(p0.size, np.uint16)
        ms, ms_m, ms_v = _to_shards(L, numel, p0), np.zeros(L.np_total, np.float32), \
            np.zeros(L.np_total, np.float32)
        pz = np.zeros(L.np_total, np.uint16)
        outs = [np.zeros(L.np_total, orc.storage_dtype(cdt)) for _ in range(W)] if stage == 1 else None
        for step in range(3):
            i_d = orc.ddp_step(per_param, gdt, cdt, wl.BF16, md, mm, vd, pd, hp, sc_d)
            i_z = orc.zero_step(numel, W, stage, bucket, gdt, cdt, wl.BF16, flat, ms, ms_m, ms_v,
                                pz, hp, sc_z, allreduce_out=outs)
            assert i_d.overflow == i_z.overflow == 0
            assert i_z.grad_norm == pytest.approx(i_d.grad_norm, rel=1e-14)
        zm, zmm, zv = (_from_shards(L, numel, a) for a in (ms, ms_m, ms_v))
        if clip == 0.0:
            assert np.array_equal(zm, md) and np.array_equal(zmm, mm) and np.array_equal(zv, vd)
        else:
            for a, b in ((zm, md), (zmm, mm), (zv, vd)):
                ulps = np.abs(a.view(np.int32).astype(np.int64) - b.view(np.int32).astype(np.int64))
                assert ulps.max() <= 1
        gathered = np.concatenate([pz[off:off + k] for off, k in zip(L.param_offset, numel)])
        if clip == 0.0:
            assert np.array_equal(gathered, pd)
        mask = L.real_mask()
        assert np.all(pz[mask == 0] == 0)
        if stage == 1:
            ref = orc.reduce(flat, gdt, cdt, real_mask=mask)
            for o in outs:
                assert np.array_equal(o, ref)


def test_zero_stage1_equals_stage2(orc):
    rng = np.random.default_rng(77)
    numel = rng.integers(1, 2000, size=7)
    W = 4
    L, _, flat, p0 = _random_problem(orc, rng, numel, W, wl.F16, 4096)
    res = []
    for stage in (1, 2):
        ms = _to_shards(L, numel, p0)
        m, v = np.zeros_like(ms), np.zeros_like(ms)
        pz = np.zeros(L.np_total, np.uint16)
        outs = [np.zeros(L.np_total, np.uint16) for _ in range(W)]
        sc = orc.Scaler(scale=1024.0, dynamic=True)
        info = orc.zero_step(numel, W, stage, 4096, wl.F16, wl.F16, wl.F16, flat, ms, m, v, pz,
                             orc.Hparams(), sc, allreduce_out=outs)
        res.append((ms, m, v, pz, info.grad_norm))
    for a, b in zip(res[0][:4], res[1][:4]):
        assert np.array_equal(a, b)
    assert res[0][4] == res[1][4]


def test_overflow_anywhere_skips_step(orc):
    """+inf or NaN at the first or last real element of a shard, in any rank,
    sets the flag and leaves master/m/v/params/t untouched; NaN padding does not."""
    rng = np.random.default_rng(21)
    numel = np.array([300, 64, 513])
    W = 3
    L, _, flat, p0 = _random_problem(orc, rng, numel, W, wl.BF16, 1024)
    mask = L.real_mask()
    positions = []
    for _, _, f0, _, ln in L.shard_ranges():
        real = np.nonzero(mask[f0:f0 + ln])[0]
        if len(real):
            positions += [f0 + real[0], f0 + real[-1]]
    for pos in positions:
        for rank in (0, W - 1):
            for bad in (np.inf, -np.inf, np.nan):
                g = [f.copy() for f in flat]
                g[rank][pos] = orc.encode(np.array([bad], np.float32), wl.BF16)[0]
                ms = _to_shards(L, numel, p0)
                m, v = np.zeros_like(ms), np.zeros_like(ms)
                pz = np.full(L.np_total, 7, np.uint16)
                sc = orc.Scaler(scale=8.0, dynamic=True, t=5)
                info = orc.zero_step(numel, W, 2, 1024, wl.BF16, wl.BF16, wl.BF16, g, ms, m, v,
                                     pz, orc.Hparams(), sc)
                assert info.overflow == 1 and info.skipped == 1
                assert sc.t == 5 and sc.scale == 4.0
                assert np.array_equal(ms, _to_shards(L, numel, p0))
                assert not m.any() and not v.any() and np.all(pz == 7)
    # clean inputs (NaN only in padding) do not overflow
    ms = _to_shards(L, numel, p0)
    info = orc.zero_step(numel, W, 2, 1024, wl.BF16, wl.BF16, wl.BF16, flat, ms,
                         np.zeros_like(ms), np.zeros_like(ms), np.zeros(L.np_total, np.uint16),
                         orc.Hparams(), orc.Scaler())
    assert info.overflow == 0


# ---------------------------------------------------------------------------
# Gradient accumulation (the step before the reduce)
# ---------------------------------------------------------------------------

def test_accumulate_exact_and_ordered(orc):
    """Integer micro-gradients sum exactly; `first` restarts the window; the
    fp32 adds run in micro-step order (1 + 2^-24 + 2^-24 stays 1)."""
    main = np.full(4, 123.0, np.float32)
    steps = [np.array([1, -2, 3, 2.0 ** -24], np.float32), np.array([4, 5, -6, 2.0 ** -24], np.float32),
             np.array([-7, 8, 9, 0], np.float32)]
    orc.accumulate(orc.encode(steps[0], wl.BF16), wl.BF16, main, first=True)
    orc.accumulate(steps[1], wl.F32, main, first=False)
    orc.accumulate(steps[2], wl.F32, main, first=False)
    assert main[:3].tolist() == [-2.0, 11.0, 6.0]
    assert main[3] == np.float32(2.0 ** -24 + 2.0 ** -24)  # bf16 keeps 2^-24 exactly
    m2 = np.array([1.0], np.float32)
    orc.accumulate(np.array([2.0 ** -24], np.float32), wl.F32, m2, first=False)
    orc.accumulate(np.array([2.0 ** -24], np.float32), wl.F32, m2, first=False)
    assert m2[0] == 1.0


def test_accumulate_first_and_padding(orc):
    main = np.array([5.0, 7.0, 9.0], np.float32)
    mask = np.array([1, 0, 1], np.uint8)
    orc.accumulate(np.array([-0.0, 1.0, 2.0], np.float32), wl.F32, main, first=True, real_mask=mask)
    assert main.tolist() == [0.0, 7.0, 2.0]
    assert not np.signbit(main[0])  # +0 + -0 is +0
