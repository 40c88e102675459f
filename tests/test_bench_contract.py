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
