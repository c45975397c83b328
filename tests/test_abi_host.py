"""Host-side checks of the C-ABI library (no GPU needed).

The library loads, exports every entry point include/zero.h declares, builds
the same layout as the oracle's independent layout code (bit-exact offsets,
buckets and shard ranges), reports the pages' byte ledger, and rejects bad
arguments before touching the device.
"""
import json
import os
import re
import subprocess

import numpy as np
import pytest

import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def zlib():
    from mixed_precision_gb300 import build
    build.build()
    import mixed_precision_gb300 as mp
    mp.lib()
    return mp


def _declared():
    text = open(os.path.join(ROOT, "include", "zero.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zero_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(zlib):
    names = _declared()
    assert len(names) >= 15
    lib_path = os.path.join(ROOT, "mixed_precision_gb300", "libzero_gb300.so")
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r" T (\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(zlib.lib(), n)


def _cfg(zlib, W, stage=2, bucket=500_000_000, g=wl.BF16, p=wl.BF16, c=-1):
    return zlib.zero_config(W, stage, bucket, g, p, c, 0)


def _compare_layout(zlib, orc, shapes, W, bucket, g):
    numel = wl.numels(shapes)
    h = zlib.zero_layout_create(shapes, _cfg(zlib, W, 2, bucket, g))
    try:
        info = zlib.zero_layout_query(h)
        L = orc.layout(numel, W, bucket, wl.ELEM_BYTES[g])
        assert info.n_padded == L.np_total and info.n_real == sum(numel)
        assert info.n_buckets == len(L.bucket_start)
        offs = [zlib.zero_param_offset(h, p) for p in range(len(shapes))]
        assert offs == L.param_offset.tolist()
        for b in range(info.n_buckets):
            assert zlib.zero_bucket_range(h, b) == (L.bucket_start[b], L.bucket_len[b])
        ranges = {(b, r): (f0, s0, ln) for b, r, f0, s0, ln in L.shard_ranges()}
        for b in range(info.n_buckets):
            for r in range(W):
                assert zlib.zero_shard_range(h, b, r) == ranges[(b, r)]
        return info
    finally:
        zlib.zero_layout_destroy(h)


def test_layout_matches_oracle_random(zlib, orc):
    rng = np.random.default_rng(1234)
    for _ in range(150):
        n = int(rng.integers(1, 12))
        shapes = [tuple(int(x) for x in rng.integers(0, 40, size=int(rng.integers(0, 3))))
                  for _ in range(n)]
        W = int(rng.integers(1, 9))
        g = int(rng.choice([wl.F32, wl.F16, wl.BF16]))
        bucket = int(rng.choice([4, 100, 1000, 5000, 1 << 20]))
        _compare_layout(zlib, orc, shapes, W, bucket, g)


@pytest.mark.parametrize("name,W,bucket", [("qwen3_0.6b_bf16_w2", 2, 500_000_000),
                                           ("qwen3_0.6b_bf16_w2", 8, 500_000_000),
                                           ("moe_3.9b_bf16_w4", 4, 500_000_000),
                                           ("ragged_2000", 8, 1_000_000),
                                           ("ragged_2000", 2, 1_000_000_000)])
def test_layout_matches_oracle_workloads(zlib, orc, name, W, bucket):
    w = wl.workload(name)
    info = _compare_layout(zlib, orc, w.shapes, W, bucket, w.grad_dtype)
    assert info.n_params == len(w.shapes)


def test_ledger_matches_page_table(zlib):
    gold = json.load(open(os.path.join(ROOT, "tests", "golden", "ledger.json")))
    for d, expect in gold["bf16_param_fp32_grad_stage1"].items():
        h = zlib.zero_layout_create([(1024,)], _cfg(zlib, int(d), 1, 1 << 20, wl.F32, wl.BF16))
        assert zlib.zero_layout_query(h).ledger_bytes_per_param == pytest.approx(expect)
        zlib.zero_layout_destroy(h)
    h = zlib.zero_layout_create([(1024,)], _cfg(zlib, 1, 2, 1 << 20, wl.F16, wl.F16))
    per_param = zlib.zero_layout_query(h).ledger_bytes_per_param
    assert per_param == pytest.approx(gold["fp16_param_fp16_grad_unsharded"])
    assert 70e9 * per_param / 1e9 == pytest.approx(gold["seventy_b_model_state_gb"])
    zlib.zero_layout_destroy(h)


def test_ledger_stage3_shards_everything(zlib):
    """ZeRO-3 shards all 16 bytes of fp16/bf16 mixed-precision state: 16/W per
    parameter ("3.7 ...", "ZeRO Stages Recap")."""
    for W in (1, 2, 4, 8):
        h = zlib.zero_layout_create([(1024,)], _cfg(zlib, W, 3, 1 << 20, wl.BF16, wl.BF16))
        assert zlib.zero_layout_query(h).ledger_bytes_per_param == pytest.approx(16.0 / W)
        zlib.zero_layout_destroy(h)


def test_step_bytes_formula(zlib):
    for W in (2, 4, 8):
        h = zlib.zero_layout_create([(4096,)], _cfg(zlib, W))
        assert zlib.zero_layout_query(h).step_bytes_per_elem == 2 * W + 26
        zlib.zero_layout_destroy(h)


def test_invalid_arguments(zlib):
    bad = [_cfg(zlib, 0), _cfg(zlib, 65), _cfg(zlib, 2, stage=4), _cfg(zlib, 2, bucket=0),
           _cfg(zlib, 2, g=7), _cfg(zlib, 2, p=wl.F32), _cfg(zlib, 2, c=9), _cfg(zlib, 2, bucket=1)]
    for cfg in bad:
        with pytest.raises(zlib.ZeroError) as e:
            zlib.zero_layout_create([(10,)], cfg)
        assert e.value.code == 1
    with pytest.raises(zlib.ZeroError):
        zlib.zero_layout_create([], _cfg(zlib, 2))
    with pytest.raises(zlib.ZeroError):
        zlib.zero_layout_create([(-1, 3)], _cfg(zlib, 2))
    h = zlib.zero_layout_create([(10,), (3, 3)], _cfg(zlib, 2))
    with pytest.raises(zlib.ZeroError) as e:
        zlib.zero_param_offset(h, 2)
    assert e.value.code == 1
    with pytest.raises(zlib.ZeroError):
        zlib.zero_shard_range(h, 0, 2)
    # bind: NULL and misaligned pointers are rejected before any device call
    with pytest.raises(zlib.ZeroError) as e:
        zlib.zero_state_bind(h, 0, 16, 32, 48, 64)
    assert e.value.code == 1
    with pytest.raises(zlib.ZeroError) as e:
        zlib.zero_state_bind(h, 8, 16, 32, 48, 64)
    assert e.value.code == 1
    with pytest.raises(zlib.ZeroError) as e:
        zlib.zero_state_bind(h, 16, 32, 48, 64, 0)  # stage 2 needs scratch
    assert e.value.code == 1
    # a step before bind is out of order
    hp = zlib.zero_hparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1.0, 0.0)
    with pytest.raises(zlib.ZeroError) as e:
        zlib.zero_step(h, [16, 32], None, hp, 0)
    assert e.value.code == 5
    # the speculative step's entry points are out of order before bind too
    with pytest.raises(zlib.ZeroError) as e:
        zlib.zero_state_bind_alternate(h, 16, 32, 48)
    assert e.value.code == 5
    with pytest.raises(zlib.ZeroError) as e:
        zlib.zero_step_speculative(h, [16, 32], hp, 0)
    assert e.value.code == 5
    zlib.zero_layout_destroy(h)


def test_size_limits(zlib):
    """The parameters' total is capped at ZERO_MAX_ELEMS (2^36) elements, per
    parameter and in all; below the cap, element offsets past 2^32 are exact."""
    cap = zlib.ZERO_MAX_ELEMS
    assert cap == 1 << 36
    for shapes in ([(cap + 1,)], [(1 << 20, (1 << 16) + 1)], [(cap // 2 + 1,), (cap // 2 + 1,)],
                   [(1 << 40, 1 << 40)]):
        with pytest.raises(zlib.ZeroError) as e:
            zlib.zero_layout_create(shapes, _cfg(zlib, 2))
        assert e.value.code == 1
    # 5 parameters, three of them past 2^31 elements and ending past 2^33
    big = [(3,), ((1 << 31) + 5,), (1 << 31, 3), (7,), ((1 << 31) + 64,)]
    h = zlib.zero_layout_create(big, _cfg(zlib, 2, bucket=1 << 33))
    info = zlib.zero_layout_query(h)
    n = [3, (1 << 31) + 5, 3 << 31, 7, (1 << 31) + 64]
    assert info.n_real == sum(n)
    # offsets: each parameter starts on the next multiple of 64 (one bucket
    # of 2^32 bf16 elements holds p0..p1; p2 opens the next, and so on)
    offs = [zlib.zero_param_offset(h, p) for p in range(5)]
    assert offs[0] == 0 and offs[1] == 64
    for p in range(1, 5):
        assert offs[p] % 64 == 0 and offs[p] >= offs[p - 1] + n[p - 1]
    assert offs[4] > 1 << 33
    # every rank's slice of every bucket is equal and tiles the bucket
    total = 0
    for b in range(info.n_buckets):
        b0, bl = zlib.zero_bucket_range(h, b)
        assert b0 == total and bl % (2 * 128) == 0
        for r in range(2):
            f0, s0, ln = zlib.zero_shard_range(h, b, r)
            assert (f0, ln) == (b0 + r * bl // 2, bl // 2)
        total += bl
    assert total == info.n_padded
    zlib.zero_layout_destroy(h)


def test_allocator_failure_is_oom(zlib):
    from mixed_precision_gb300 import _abi
    calls = []

    @_abi.ALLOC_FN
    def fail_alloc(n, ctx):
        calls.append(n)
        return None

    @_abi.FREE_FN
    def no_free(p, ctx):
        pass

    h = zlib.zero_layout_create([(1000,), (77,)], _cfg(zlib, 4))
    zlib.zero_layout_set_allocator(h, fail_alloc, no_free, 0)
    with pytest.raises(zlib.ZeroError) as e:
        zlib.zero_state_bind(h, 256, 512, 768, 1024, 1280)
    assert e.value.code == 3 and calls and calls[0] == zlib.zero_layout_query(h).device_bytes_owned
    zlib.zero_layout_destroy(h)


def test_last_error_is_set(zlib):
    with pytest.raises(zlib.ZeroError):
        zlib.zero_layout_create([(10,)], _cfg(zlib, 0))
    assert "world" in zlib.zero_last_error()


def test_dist_set_rank_partitions_the_tiles(zlib):
    """zero_dist_set_rank keeps exactly rank r's tiles: over all ranks the
    tables partition the full table. Rank out of range, a second call and a
    16-bit communication dtype other than the gradients' are refused."""
    from mixed_precision_gb300 import _abi
    shapes = [(1000,), (77,), (300, 41), (8200,), (0,), (5,), (20000,)]
    for W in (1, 2, 3, 5):
        full = zlib.zero_layout_create(shapes, _cfg(zlib, W, 2, 40_000))
        total = zlib.zero_layout_query(full).n_tiles
        zlib.zero_layout_destroy(full)
        per = []
        for r in range(W):
            h = zlib.zero_layout_create(shapes, _cfg(zlib, W, 2, 40_000))
            _abi.zero_dist_set_rank(h, r)
            info = zlib.zero_layout_query(h)
            per.append(info.n_tiles)
            # the buffers of one rank's shard
            assert info.state_bytes == info.shard_elems * 4
            assert info.scratch_bytes == info.shard_elems * 2
            assert info.params_bytes == info.n_padded * 2  # stage 2: the all-gathered buffer
            with pytest.raises(zlib.ZeroError) as e:
                _abi.zero_dist_set_rank(h, r)
            assert e.value.code == _abi.ZERO_ERR_STATE
            zlib.zero_layout_destroy(h)
        assert sum(per) == total and all(n > 0 for n in per)
    h = zlib.zero_layout_create(shapes, _cfg(zlib, 2))
    for bad in (-1, 2):
        with pytest.raises(zlib.ZeroError) as e:
            _abi.zero_dist_set_rank(h, bad)
        assert e.value.code == _abi.ZERO_ERR_INVALID
    zlib.zero_layout_destroy(h)
    # a 16-bit communication dtype other than the gradients' is refused; fp32 is not
    h = zlib.zero_layout_create(shapes, _cfg(zlib, 2, c=wl.F16))
    with pytest.raises(zlib.ZeroError) as e:
        _abi.zero_dist_set_rank(h, 0)
    assert e.value.code == _abi.ZERO_ERR_INVALID
    zlib.zero_layout_destroy(h)
    h = zlib.zero_layout_create(shapes, _cfg(zlib, 2, c=wl.F32))
    _abi.zero_dist_set_rank(h, 0)
    assert zlib.zero_layout_query(h).scratch_bytes == zlib.zero_layout_query(h).shard_elems * 4
    zlib.zero_layout_destroy(h)
