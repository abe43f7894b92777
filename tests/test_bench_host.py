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
    # the router is folded into the QKV and WO phases: five grid phases per MoE layer
    assert bench.phase_names(MOE_M) == ["qkv", "att", "wo", "egu", "edown"]
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


def _golden(name):
    vals = {}
    for line in open(os.path.join(ROOT, "tests", "golden", name)):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = (x.strip() for x in line.split("="))
            vals[k] = float(v)
    return vals


def test_roofline_arithmetic_reproduces_the_pages_worked_numbers():
    """The pages' own example of the bandwidth roofline (8 GPUs' aggregate bandwidth over a 2B model's ~4 GB of
    fp16 weights gives ~8,400 tok/s, of which ~3,000 tok/s is ~36 %) and of the launch tax (4.5 us x 10 kernels x
    25 layers per token caps decode near 890 tok/s; 3,000 tok/s leaves ~333 us per token), through the same
    roofline function the bench reports with."""
    g = _golden("roofline_arithmetic.txt")
    bytes_per_token = g["active_weight_gb"] * 1e9
    peak_gbs = g["aggregate_bandwidth_tbs"] * 1e3
    ceiling = peak_gbs * 1e9 / bytes_per_token
    assert abs(ceiling - g["ceiling_tok_s"]) / g["ceiling_tok_s"] < 0.01
    # one second of decode at the reported rate: the fraction of the ceiling is the MBU-style fraction
    _, frac = bench.roofline(bytes_per_token * g["target_tok_s"], 1.0, peak_gbs)
    assert abs(frac - g["fraction_of_ceiling"]) < 0.005
    tax = g["launch_us_per_kernel"] * g["kernels_per_layer"] * g["layers"]
    assert tax == g["launch_tax_us_per_token"]
    assert abs(1e6 / tax - g["launch_bound_tok_s"]) / g["launch_bound_tok_s"] < 0.01
    assert abs(1e6 / g["target_tok_s"] - g["budget_us_per_token"]) < 0.5
