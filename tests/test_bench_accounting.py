"""The benchmark's own arithmetic on the CPU: the per-stage work of the
prefill step adds up to the pages' FLOP count, the roofline entry divides the
right numbers, and the launch counts match the kernels a step issues."""
import pytest

import bench
import workloads
from causal_gqa_attention_rmsnorm_gb300 import accounting as acc

PEAKS = {"bf16_tflops": 1958.8, "bf16_tflops_sustained": 1730.0, "hbm_gbs": 6761.6}


def test_stage_work_adds_up_to_the_block():
    s = workloads.CONFIGS["gqa_8k"]
    w = bench.prefill_stage_work(s)
    M = s.B * s.T
    gemm = sum(w[k][1] for k in ("qkv", "wo", "w13", "w2"))
    assert gemm == acc.gemm_flops(s.d, s.H, s.Hkv, s.dh, s.f, M)
    # 2 FLOPs per parameter per token, the weight matrices of the GQA block
    assert gemm == 2 * M * (s.d * (s.H + 2 * s.Hkv) * s.dh + s.H * s.dh * s.d + 3 * s.d * s.f)
    # exact causal pairs: 4·B·H·dh·T(T+1)/2 = 2.199e12 at B=4, T=8192
    assert w["attn"][1] == 4 * s.B * s.H * s.dh * s.T * (s.T + 1) // 2
    assert w["attn"][1] == pytest.approx(2.199e12, rel=1e-3)
    assert all(w[k][0] == "tensor" for k in ("qkv", "attn", "wo", "w13", "w2")) and w["rms"][0] == "hbm"


def test_roofline_entry_takes_the_longest_stage():
    s = workloads.CONFIGS["gqa_8k"]
    work = bench.prefill_stage_work(s)
    stages = {"rms": 0.05, "qkv": 1.0, "attn": 1.6, "wo": 0.8, "w13": 4.2, "w2": 2.2}
    r = bench.roofline_entry(stages, work, PEAKS, "measured", s.name)
    assert r["kernel"] == "w13" and r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    achieved = work["w13"][1] / (4.2e-3) / 1e12
    assert r["achieved"] == pytest.approx(achieved)
    assert r["frac"] == pytest.approx(achieved / 1958.8)
    assert r["frac_of_sustained"] == pytest.approx(achieved / 1730.0)
    assert r["peak"] == 1958.8 and r["ms"] == 4.2 and r["algorithmic"] == work["w13"][1]
    # the ncu traffic belongs to this workload's W1/W3 launch, and to nothing else
    assert r["traffic"] == bench.NCU_TRAFFIC[("gqa_8k", "w13")]
    assert bench.roofline_entry(stages, work, PEAKS, "measured", "other")["traffic"] is None


def test_roofline_entry_for_a_bandwidth_stage():
    work = {"a": ("hbm", 6.7616e9), "b": ("tensor", 1.0)}
    r = bench.roofline_entry({"a": 1.0, "b": 0.5}, work, PEAKS, "measured", "x")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(6761.6) and r["frac"] == pytest.approx(1.0)


def test_decode_launch_counts():
    # the decode attention and its merge, and the four few-token GEMMs (the QKV
    # one forms the row statistics) when the batch takes them; above that, row
    # statistics and four tile GEMMs
    assert bench.decode_launches(32) == 2 + 4
    assert bench.decode_launches(bench.FEW_TOKENS + 1) == 3 + 4


def test_prefill_launch_counts():
    # four GEMMs and the attention (the tile QKV GEMM forms the row
    # statistics); with few tokens the row-statistics kernel first
    assert bench.prefill_launches(4 * 8192) == 5
    assert bench.prefill_launches(bench.FEW_TOKENS) == 6
