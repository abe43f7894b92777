"""Seeded synthetic inputs shared by the CPU oracle and the GPU library.

This module holds no part of the decoder's arithmetic. It draws random numbers (counter-based SplitMix64
plus Box-Muller, in ``synth.c``), rounds them to fp16, and lays them out as the weight tensors, prompts and
GEMV operands of the workloads in :mod:`synth.configs`. Both sides of every parity test take their inputs
from here and from nowhere else.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .configs import GemvShape, ModelConfig, MoEConfig, Workload  # noqa: F401  (re-export)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None

# Tensor ids of the weight streams (one independent stream per tensor).
TID_EMBED, TID_LM_HEAD, TID_FINAL_NORM, TID_PROMPT = 1, 2, 3, 0xFFFF
LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


TID_ROUTER_SLOT = len(LAYER_TENSORS)  # the router of layer l has layer tensor slot 9
EXPERT_KINDS = ("gate", "up", "down")


def layer_tid(layer: int, name: str) -> int:
    return 16 + 16 * layer + LAYER_TENSORS.index(name)


def expert_tid(layer: int, expert: int, kind: str) -> int:
    return 0x10000000 + (layer * 4096 + expert) * 4 + EXPERT_KINDS.index(kind)


def build_cmd() -> list[str]:
    return ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o", _LIB, _SRC, "-lm"]


def build(force: bool = False) -> None:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(build_cmd())


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u64, i64, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
        L.synth_normal_f16.argtypes = [u64, u64, i64, dbl, dbl, ctypes.c_void_p]
        L.synth_normal_f32.argtypes = [u64, u64, i64, dbl, dbl, ctypes.c_void_p]
        L.synth_tokens.argtypes = [u64, u64, i64, i64, ctypes.c_void_p]
        L.synth_draw.argtypes = [u64, u64, u64]
        L.synth_draw.restype = u64
        L.synth_splitmix64_next.argtypes = [ctypes.POINTER(u64)]
        L.synth_splitmix64_next.restype = u64
        L.synth_f32_to_f16.argtypes = [ctypes.c_float]
        L.synth_f32_to_f16.restype = ctypes.c_uint16
        L.synth_e4m3_rows.argtypes = [u64, u64, i64, i64, dbl, ctypes.c_void_p, ctypes.c_void_p]
        L.synth_f32_to_e4m3.argtypes = [ctypes.c_float]
        L.synth_f32_to_e4m3.restype = ctypes.c_uint8
        _lib = L
    return _lib


def normal_f16(seed: int, tensor_id: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """fp16 bit patterns (uint16) of mean + std * N(0, 1), rounded fp64 -> fp32 -> fp16 (RNE)."""
    out = np.empty(shape, dtype=np.uint16)
    lib().synth_normal_f16(seed, tensor_id, out.size, mean, std, out.ctypes.data)
    return out


def normal_f32(seed: int, tensor_id: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    lib().synth_normal_f32(seed, tensor_id, out.size, mean, std, out.ctypes.data)
    return out


def tokens(seed: int, n: int, vocab: int, tensor_id: int = TID_PROMPT) -> np.ndarray:
    """n token ids uniform over [0, vocab)."""
    out = np.empty(n, dtype=np.int32)
    lib().synth_tokens(seed, tensor_id, n, vocab, out.ctypes.data)
    return out


def model_weights(cfg: ModelConfig, ffn: bool = True) -> dict:
    """All weights of a Llama-style decoder as fp16 bit patterns, row-major [out, in] (without the dense FFN
    matrices when ffn is False).

    Projections, embedding and LM head are N(0, weight_std). RMSNorm gains are exactly 1 when gain_std
    is 0, else 1 + N(0, gain_std).
    """
    s, d, dh = cfg.seed, cfg.d_model, cfg.head_dim

    def w(tid, shape):
        return normal_f16(s, tid, shape, 0.0, cfg.weight_std)

    def gain(tid):
        if cfg.gain_std == 0.0:
            return np.full(d, 0x3C00, dtype=np.uint16)
        return normal_f16(s, tid, d, 1.0, cfg.gain_std)

    layers = []
    for l in range(cfg.n_layers):
        t = lambda name: layer_tid(l, name)  # noqa: E731
        layers.append({
            "attn_norm": gain(t("attn_norm")),
            "wq": w(t("wq"), (cfg.n_heads * dh, d)),
            "wk": w(t("wk"), (cfg.n_kv_heads * dh, d)),
            "wv": w(t("wv"), (cfg.n_kv_heads * dh, d)),
            "wo": w(t("wo"), (d, cfg.n_heads * dh)),
            "ffn_norm": gain(t("ffn_norm")),
        })
        if ffn:
            layers[-1].update({
                "w_gate": w(t("w_gate"), (cfg.ffn_dim, d)),
                "w_up": w(t("w_up"), (cfg.ffn_dim, d)),
                "w_down": w(t("w_down"), (d, cfg.ffn_dim)),
            })
    return {
        "embed": w(TID_EMBED, (cfg.vocab, d)),
        "lm_head": w(TID_LM_HEAD, (cfg.vocab, d)),
        "final_norm": gain(TID_FINAL_NORM),
        "layers": layers,
    }


def e4m3_rows(seed: int, tensor_id: int, rows: int, cols: int, std: float):
    """FP8 weight rows: (q uint8 [rows, cols] E4M3 codes, scale float32 [rows]); weight = E4M3(q) * scale."""
    q = np.empty((rows, cols), dtype=np.uint8)
    sc = np.empty(rows, dtype=np.float32)
    lib().synth_e4m3_rows(seed, tensor_id, rows, cols, std, q.ctypes.data, sc.ctypes.data)
    return q, sc


def moe_weights(cfg: MoEConfig) -> dict:
    """A sparse-MoE decoder's weights: attention, norms, embedding and LM head as in model_weights (fp16),
    per layer a router [n_experts, d] (fp16, N(0, weight_std)) and the experts' FP8 matrices with row scales,
    stacked over experts: gate_q/up_q [E, F_e, d], down_q [E, d, F_e] (uint8), gate_s/up_s [E, F_e],
    down_s [E, d] (float32); every expert weight is N(0, weight_std) before quantisation."""
    s, d, Fe, E = cfg.seed, cfg.d_model, cfg.expert_ffn, cfg.n_experts
    base = model_weights(cfg, ffn=False)
    for l, lay in enumerate(base["layers"]):
        lay["router"] = normal_f16(s, 16 + 16 * l + TID_ROUTER_SLOT, (E, d), 0.0, cfg.weight_std)
        for kind, (rows, cols) in (("gate", (Fe, d)), ("up", (Fe, d)), ("down", (d, Fe))):
            q = np.empty((E, rows, cols), dtype=np.uint8)
            sc = np.empty((E, rows), dtype=np.float32)
            for e in range(E):
                q[e], sc[e] = e4m3_rows(s, expert_tid(l, e, kind), rows, cols, cfg.weight_std)
            lay[kind + "_q"], lay[kind + "_s"] = q, sc
    return base


def prompt(wl: Workload) -> np.ndarray:
    return tokens(wl.model.seed, wl.prompt_len, wl.model.vocab)


def gemv_operands(shape: GemvShape):
    """W [M, K] fp16 ~ N(0, 1/sqrt(K)) and x [K] fp16 ~ N(0, 1), seeded per shape."""
    W = normal_f16(shape.seed, 1, (shape.M, shape.K), 0.0, 1.0 / np.sqrt(shape.K))
    x = normal_f16(shape.seed, 2, shape.K, 0.0, 1.0)
    return W, x


def as_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of fp16 bit patterns (numpy's own float16 conversion)."""
    return bits.view(np.float16).astype(np.float32)
