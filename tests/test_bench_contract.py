"""Host-side arithmetic of bench.py: the algorithmic bytes behind the attention's roofline and the
rule that decides when its launches may be timed back to back (no GPU needed)."""
import pytest

import bench


def test_gqa_attention_bytes_per_launch():
    # 16 requests x (2048 records of 8 KV heads x (128 K + 128 V) bf16 = 4096 B, q of 32 heads x 128
    # bf16, fp32 output of 32 x 128, 2048 int32 slots)
    w = bench.WORKLOADS["gqa_b16_l32"]
    assert bench.record_bytes(w) == 4096
    assert bench.attn_bytes_per_launch(w) == 16 * (2048 * 4096 + 32 * 128 * 2 + 32 * 128 * 4 + 2048 * 4)
    assert bench.attn_bytes_per_launch(w) == 134_742_016


def test_latent_attention_bytes_per_launch():
    # 8 requests x (2048 records of a 576-value bf16 latent, q of 64 heads x 576, output 64 x 512 fp32)
    w = bench.WORKLOADS["mla_b8"]
    assert bench.record_bytes(w) == 1152
    assert bench.attn_bytes_per_launch(w) == 8 * (2048 * 1152 + 64 * 576 * 2 + 64 * 512 * 4 + 2048 * 4)


@pytest.mark.parametrize("name, exceeds", [("gqa_b16_l32", True), ("mla_b8", False), ("csa_b8", False),
                                           ("tiny", False), ("stress_b16_l4", False)])
def test_back_to_back_timing_only_above_l2(name, exceeds):
    # 32 GQA launches gather 4.3 GB per step; the single-layer latent workloads stay inside L2
    assert bench.steps_exceed_l2(bench.WORKLOADS[name]) is exceeds


def test_reference_arm_prints_its_line():
    """`bench.py --impl reference` times the CPU oracle and prints one JSON line with the keys the
    reference arm carries: impl, the same metric and unit, a cpu_baseline and a zero-copy e2e."""
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    import time

    env = dict(os.environ, HS_REF_STEP_SECONDS="0.05")
    t0 = time.time()
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2",
                          "--warmup", "3"], cwd=root, env=env, capture_output=True, text=True, timeout=600)
    wall = time.time() - t0
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "layer-steps/s"
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # the line claims only what ran: its steps took steps x ms_per_step inside the run's wall time, and
    # the rate extrapolated from the sampled pairs says so
    assert d["steps"] == 2 and d["steps"] * d["ms_per_step"] / 1e3 <= wall
    assert d["extrapolated"] is True and d["timed_work"]["pairs_per_step"] >= 1
    assert d["cpu_baseline"]["nproc"] >= 1 and d["cpu_baseline"]["cpu_model"]


@pytest.mark.parametrize("name, per_layer", [("gqa_b16_l32", 2), ("mla_b8", 3), ("csa_b8", 3), ("stress_b16_l4", 3),
                                             ("tiny", 2)])
def test_launches_per_layer(name, per_layer):
    # resolve (append fused) + attention; the 64-head shared-latent attention also launches its combine
    assert bench.launches_per_layer(bench.WORKLOADS[name]) == per_layer
    assert bench.launches_per_layer(bench.WORKLOADS[name], separate_append=True) == per_layer + 1
