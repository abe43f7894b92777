"""bench.py's host-side arithmetic, no GPU: the algorithmic bytes the roofline divides by, the per-phase byte
counts, the phase order of each model family, and the rule that a DRAM-traffic figure is reported only for the
kernel sources it was captured from."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth.configs import MOE_M, TWO_B  # noqa: E402


def test_algorithmic_bytes_of_the_bench_launch():
    # 1,024 tokens after a 128-token prompt: every weight once per token + 51,200 bytes of K/V per attended position
    assert TWO_B.weight_bytes_per_token() == 3_899_392_000
    kv = sum(51_200 * c for c in range(129, 1153))
    assert bench.algorithmic_bytes(TWO_B, 128, 1024) == 1024 * 3_899_392_000 + kv == 4_026_558_054_400


def test_moe_active_bytes_count_only_the_routed_experts():
    assert MOE_M.weight_bytes_per_token() == 1_246_232_576
    d, dh, F = MOE_M.d_model, MOE_M.head_dim, MOE_M.expert_ffn
    attn = 2 * ((MOE_M.n_heads + 2 * MOE_M.n_kv_heads) * dh * d + d * MOE_M.n_heads * dh)
    dense_parts = MOE_M.n_layers * (attn + 2 * MOE_M.n_experts * d) + 2 * MOE_M.vocab * d
    per_expert = 3 * F * d + 4 * (2 * F + d)  # FP8 codes + fp32 row scales
    assert MOE_M.weight_bytes_per_token() - dense_parts == MOE_M.n_layers * MOE_M.top_k * per_expert
    assert bench.algorithmic_bytes(MOE_M, 256, 512) == 650_968_563_712


def test_phase_bytes_add_up_to_a_layer():
    b = bench.phase_bytes(TWO_B, 145)
    layer = TWO_B.weight_bytes_per_token() - b["lm"]
    assert (b["qkv"] + b["wo"] + b["gu"] + b["down"]) * TWO_B.n_layers == layer
    assert b["att"] == 2 * 2 * TWO_B.n_kv_heads * TWO_B.head_dim * 145
    assert bench.phase_names(TWO_B) == ["qkv", "att", "wo", "gu", "down"]
    assert bench.phase_names(MOE_M) == ["qkv", "att", "wo", "router", "egu", "edown"]
    m = bench.phase_bytes(MOE_M, 300)
    layer_moe = (MOE_M.weight_bytes_per_token() - m["lm"]) // MOE_M.n_layers
    assert m["qkv"] + m["wo"] + m["router"] + m["egu"] + m["edown"] == layer_moe


def test_traffic_is_reported_only_for_matching_sources():
    import persistent_monokernel_decode_gb300 as kie
    digest = kie.source_digest()
    t = bench.profiled_traffic("llama2b_p128_n1024", digest)
    assert t is None or 0.99 < t / bench.algorithmic_bytes(TWO_B, 128, 1024) < 1.01
    assert bench.profiled_traffic("llama2b_p128_n1024", "0" * 16) is None
    assert bench.profiled_traffic("no_such_workload", digest) is None
