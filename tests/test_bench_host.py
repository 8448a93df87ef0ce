"""bench.py host logic: the reference arm (one JSON line from rank 0, nothing from other
ranks) and the per-step launch count it claims."""
from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_fp32",
           "--steps", "2", "--warmup", "3", "--reference-tokens", "64"]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_line():
    r = _run({"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("tiny_fp32: T=256 d=128 E=8 top-2")
    assert d["config"]["tokens_per_step"] == 64
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["h2d_bytes_per_step"] == 0 == e2e["d2h_bytes_per_step"]


def test_reference_arm_other_ranks_do_no_work():
    r = _run({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_launch_count_claim_matches_the_launch_lists():
    """gpu_launches per step, as the committed ncu launch lists count them: 10 launches per
    DeepSeek-V2-Lite or Llama-4-Scout forward (router 3, dispatch 2, GEMMs 4, combine 1; the
    bf16 pair GEMM reads the bucket offsets itself), 9 per Qwen3-30B-A3B forward (its
    8192-entry dispatch count table takes a scan launch of its own; no shared expert) and 16
    per condensing Luffy-shaped forward (condensation 5: m-tiles, tile list, similarity GEMM
    with each row's earliest similar row, resolve, greedy scan with the condensed count; the
    dispatch forms the row statistics)."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from routing_expert_ffn_gb300 import inputs as gen
    assert bench.launches_per_step(gen.CONFIGS["dsv2_lite"], False) == 10
    assert bench.launches_per_step(gen.CONFIGS["llama4_scout_farskip"], False) == 10
    assert bench.launches_per_step(gen.CONFIGS["qwen3_30b_a3b"], False) == 9
    assert bench.launches_per_step(gen.CONFIGS["luffy_condense"], True) == 16
    # 64 tokens: the same tensor-core router as larger batches
    assert bench.launches_per_step(gen.CONFIGS["dsv2_lite_decode"], False) == 10
