"""bench.py's GPU arm: a short run prints one JSON line with every key the
contract asks for (GB300)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_our_line_keys():
    res = subprocess.run([sys.executable, "bench.py", "--steps", "5", "--warmup", "3",
                          "--e2e-steps", "2", "--cpu-seconds", "1", "--per-config-steps", "3"],
                         cwd=ROOT,
                         capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
              "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["value"] > 0
    assert d["scaling"] == "weak" and d["gpu_launches"] == 2 * 5
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "hbm" and 0 < r["frac"] < 1.5
    for k in ("value", "unit", "cores", "kind", "sample"):
        assert k in d["cpu_baseline"], k
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in d["e2e"], k
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    for k in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert k in d["clocks"], k
    # the other named workloads, each with its own bytes per step
    pc = d["per_config"]
    assert set(pc) == {"moe_3.9b_bf16_w4_stage2", "qwen3_0.6b_fp16_w8_stage1",
                       "qwen3_0.6b_fp16_w8_stage2", "qwen3_0.6b_bf16_w2_speculative_clip0",
                       "moe_3.9b_bf16_w4_speculative_clip0", "ragged_2000_w2", "ragged_2000_w8",
                       "ragged_2000_w8_per_tensor_launch", "moe_3.9b_bf16_w4_tensors_idle_experts_null",
                       "qwen3_0.6b_fp16_w8_stage1_speculative"}
    for name, c in pc.items():
        assert c["steps"] == 3 and c["ms_per_step"] > 0 and 0 < c["step_roofline"]["frac"] < 1.5
        base = name.rsplit("_stage", 1)[0].split("_speculative")[0].split("_tensors")[0]
        if name.startswith("ragged_2000"):
            base = "ragged_2000"
            assert c["config"]["world_simulated"] == int(name.split("_w")[1][0])
        assert c["config"]["workload"] == base
        assert "roofline" in c
        for k in ("sm_mhz", "sm_max_mhz", "reasons"):
            assert k in c["clocks"], k
    for name in ("qwen3_0.6b_bf16_w2_speculative_clip0", "moe_3.9b_bf16_w4_speculative_clip0"):
        assert pc[name]["fast_path"] == 1 and pc[name]["config"]["clip"] == 0.0
    # ZeRO-1 through the single pass: clip 1.0 stays inactive, every step commits,
    # and its bytes count the all-reduce writes
    s1s = pc["qwen3_0.6b_fp16_w8_stage1_speculative"]
    assert s1s["fast_path"] == 1 and s1s["config"]["zero_stage"] == 1
    assert s1s["step_roofline"]["bytes_per_param"] == \
        pc["qwen3_0.6b_fp16_w8_stage1"]["step_roofline"]["bytes_per_param"]
    # the flat step against launching it tensor by tensor, same bytes
    assert "per-tensor" in pc["ragged_2000_w8_per_tensor_launch"]["config"]["note"]
    assert "note" not in pc["ragged_2000_w8"]["config"]
    # the MoE list with each rank's idle experts passed as NULL: fewer bytes to move
    sp = pc["moe_3.9b_bf16_w4_tensors_idle_experts_null"]["step_roofline"]
    assert sp["sparse_bytes_per_param"] < sp["bytes_per_param"] and 0 < sp["sparse_frac"] < 1.5
    s1 = pc["qwen3_0.6b_fp16_w8_stage1"]["step_roofline"]
    assert s1["bytes_per_param"] == s1["ledger_bytes_per_param"] + 8 * 2  # the W*C all-reduce writes


def test_sharded_line_keys():
    """bench.py --sharded, one process on one GPU (NCCL with one rank): the
    whole sharded step, collectives included, prints a complete line."""
    res = subprocess.run([sys.executable, "bench.py", "--sharded", "--steps", "3", "--warmup", "3",
                          "--e2e-steps", "2"], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
              "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["value"] > 0 and d["scaling"] == "strong"
    # per step: the shard norm, the finalize and one update per bucket (3 buckets
    # of the Qwen3 list at 500 MB), each bucket's all-gather beside the next update
    assert d["config"]["parallelism"] == "zero2_dp1" and d["gpu_launches"] == 3 * (2 + 3)
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
