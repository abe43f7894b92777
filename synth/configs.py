"""The synthetic workloads: model shapes, seeds and prompt/decode lengths.

Shapes follow the batch-1 decode workloads of the Kog monokernel pages ("2B demo vs frontier scale":
a 2B fp16 model, ~25 layers, batch 1), made concrete as Llama-style decoders. Weights are random
(no trained checkpoint is used); only byte counts and shapes matter for speed, and the oracle fixes
the values for parity.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    seed: int
    rope_theta: float = 10000.0
    rms_eps: float = 1e-5
    weight_std: float = 0.02
    gain_std: float = 0.0  # 0: RMSNorm gains exactly 1

    def weight_bytes_per_token(self) -> int:
        """fp16 bytes of every weight a decode step must stream (all projections + LM head)."""
        d, dh, F = self.d_model, self.head_dim, self.ffn_dim
        per_layer = (self.n_heads * dh + 2 * self.n_kv_heads * dh) * d + d * self.n_heads * dh + 3 * F * d
        return 2 * (self.n_layers * per_layer + self.vocab * d)

    def kv_bytes_per_token(self, c: int) -> int:
        """fp16 K and V bytes one decode step reads when it attends over c positions."""
        return 2 * 2 * self.n_layers * self.n_kv_heads * self.head_dim * c


@dataclass(frozen=True)
class MoEConfig(ModelConfig):
    """A sparse-MoE decoder: the FFN of every layer is n_experts SwiGLU experts of width expert_ffn with FP8
    E4M3 weights (per-output-row fp32 scales) and a top_k softmax router (fp16 weights [n_experts, d])."""
    n_experts: int = 0
    top_k: int = 0
    expert_ffn: int = 0

    def weight_bytes_per_token(self) -> int:
        """Active bytes a decode step must stream: attention and router (fp16), top_k experts (FP8 plus
        their row scales), embedding row excluded, LM head (fp16)."""
        d, dh, Fe = self.d_model, self.head_dim, self.expert_ffn
        attn = 2 * ((self.n_heads * dh + 2 * self.n_kv_heads * dh) * d + d * self.n_heads * dh)
        router = 2 * self.n_experts * d
        experts = self.top_k * (3 * Fe * d + 4 * (2 * Fe + d))
        return self.n_layers * (attn + router + experts) + 2 * self.vocab * d


@dataclass(frozen=True)
class Workload:
    name: str
    model: ModelConfig
    prompt_len: int
    decode_len: int
    max_seq: int = 0

    @property
    def capacity(self) -> int:
        return self.max_seq or (self.prompt_len + self.decode_len)


@dataclass(frozen=True)
class GemvShape:
    M: int
    K: int
    seed: int

    def bytes(self) -> int:
        return 2 * self.M * self.K + 2 * self.K + 4 * self.M


TINY = ModelConfig("tiny", n_layers=2, d_model=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=704,
                   vocab=4096, seed=0)
TWO_B = ModelConfig("llama2b", n_layers=25, d_model=2560, n_heads=20, n_kv_heads=4, head_dim=128,
                    ffn_dim=7680, vocab=32000, seed=1, gain_std=0.01)

# the sparse-MoE model (FP8 experts) and a tiny one of the same structure
MOE_M = MoEConfig("moe", n_layers=24, d_model=2048, n_heads=16, n_kv_heads=4, head_dim=128, ffn_dim=1024,
                  vocab=32000, seed=2, gain_std=0.01, n_experts=64, top_k=4, expert_ffn=1024)
MOE_TINY = MoEConfig("moe_tiny", n_layers=2, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=128,
                     vocab=4096, seed=3, gain_std=0.01, n_experts=8, top_k=4, expert_ffn=128)

TINY_DECODE = Workload("tiny_p16_n32", TINY, prompt_len=16, decode_len=32)
TWO_B_DECODE = Workload("llama2b_p128_n1024", TWO_B, prompt_len=128, decode_len=1024)
TWO_B_LONG = Workload("llama2b_p8192_n512", TWO_B, prompt_len=8192, decode_len=512)

GEMV_DIMS = (2048, 2560, 4096, 7680, 16384)
GEMV_SHAPES = tuple(GemvShape(M, K, 1000 + 5 * i + j) for i, M in enumerate(GEMV_DIMS)
                    for j, K in enumerate(GEMV_DIMS))

MOE_DECODE = Workload("moe_p256_n512", MOE_M, prompt_len=256, decode_len=512)

WORKLOADS = {w.name: w for w in (TINY_DECODE, TWO_B_DECODE, TWO_B_LONG, MOE_DECODE)}
