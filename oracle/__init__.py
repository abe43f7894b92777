"""ctypes wrapper of the CPU oracle (oracle.c). TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import this package. It never
imports the GPU library, and the GPU library never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, f) for f in ("oracle.c", "oracle_impl.h")]
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

P = ctypes.c_void_p


class OrcConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim",
                                             "ffn_dim", "vocab", "max_seq")] + \
               [("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float)]


class OrcWeights(ctypes.Structure):
    _fields_ = [(n, P) for n in ("embed", "lm_head", "final_norm", "attn_norm", "wq", "wk", "wv", "wo",
                                 "ffn_norm", "w_gate", "w_up", "w_down")]


def build_cmd() -> list[str]:
    return ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            "-o", _LIB, os.path.join(_HERE, "oracle.c"), "-lm"]


def build(force: bool = False) -> None:
    newest = max(os.path.getmtime(s) for s in _SRCS)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        subprocess.check_call(build_cmd())


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i, f, d = ctypes.c_int, ctypes.c_float, ctypes.c_double
        sig = {
            "orc_set_threads": ([i], None), "orc_get_threads": ([], i),
            "orc_half_to_double": ([ctypes.c_uint16], d), "orc_double_to_half": ([d], ctypes.c_uint16),
            "orc_argmax_f32": ([P, i], i), "orc_argmax_f64": ([P, i], i),
            "orc_rmsnorm_f32": ([P, P, i, f, P], None), "orc_rmsnorm_f64": ([P, P, i, d, P], None),
            "orc_gemv_f32": ([P, P, i, i, P], None), "orc_gemv_f64": ([P, P, i, i, P], None),
            "orc_rope_f32": ([P, i, i, d], None), "orc_rope_f64": ([P, i, i, d], None),
            "orc_silu_f32": ([f], f), "orc_silu_f64": ([d], d),
            "orc_attention_f32": ([P, P, P, i, i, P], None), "orc_attention_f64": ([P, P, P, i, i, P], None),
            "orc_create": ([ctypes.POINTER(OrcConfig), ctypes.POINTER(OrcWeights), i], P),
            "orc_destroy": ([P], None), "orc_pos": ([P], i), "orc_reset": ([P], None),
            "orc_forward": ([P, i, P], i), "orc_kv_row": ([P, i, i, i, i, P], None),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes, fn.restype = args, res
        _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def _real(precision):
    return np.float32 if precision == 32 else np.float64


def set_threads(n: int) -> None:
    lib().orc_set_threads(n)


def threads() -> int:
    return lib().orc_get_threads()


def half_to_double(bits: int) -> float:
    return lib().orc_half_to_double(bits)


def double_to_half(v: float) -> int:
    return lib().orc_double_to_half(v)


def rmsnorm(x, g_bits, eps, precision=32):
    x, px = _c(x, _real(precision))
    g, pg = _c(g_bits, np.uint16)
    out = np.empty_like(x)
    getattr(lib(), f"orc_rmsnorm_f{precision}")(px, pg, x.size, eps, out.ctypes.data)
    return out


def gemv(W_bits, x, precision=32):
    W, pW = _c(W_bits, np.uint16)
    x, px = _c(x, _real(precision))
    M, K = W.shape
    y = np.empty(M, dtype=_real(precision))
    getattr(lib(), f"orc_gemv_f{precision}")(pW, px, M, K, y.ctypes.data)
    return y


def rope(v, pos, theta=10000.0, precision=32):
    v = np.array(v, dtype=_real(precision), copy=True)
    getattr(lib(), f"orc_rope_f{precision}")(v.ctypes.data, v.size, pos, theta)
    return v


def silu(z, precision=32):
    return getattr(lib(), f"orc_silu_f{precision}")(z)


def attention(q, K_bits, V_bits, precision=32):
    q, pq = _c(q, _real(precision))
    K, pK = _c(K_bits, np.uint16)
    V, pV = _c(V_bits, np.uint16)
    c, dh = K.shape
    out = np.empty(dh, dtype=_real(precision))
    getattr(lib(), f"orc_attention_f{precision}")(pq, pK, pV, c, dh, out.ctypes.data)
    return out


def argmax(v) -> int:
    v = np.ascontiguousarray(v)
    if v.dtype == np.float64:
        return lib().orc_argmax_f64(v.ctypes.data, v.size)
    v = v.astype(np.float32, copy=False)
    return lib().orc_argmax_f32(v.ctypes.data, v.size)


class Model:
    """The oracle decoder over borrowed fp16 weights (dict from synth.model_weights)."""

    def __init__(self, cfg, weights: dict, max_seq: int, precision: int = 32):
        self.cfg, self.precision, self.max_seq = cfg, precision, max_seq
        self._keep = weights
        L = cfg.n_layers
        self._arrays = {}
        ptrs = {}
        for name in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down"):
            arr = (P * max(L, 1))(*[weights["layers"][l][name].ctypes.data for l in range(L)])
            self._arrays[name] = arr
            ptrs[name] = ctypes.cast(arr, P)
        self._w = OrcWeights(embed=weights["embed"].ctypes.data, lm_head=weights["lm_head"].ctypes.data,
                             final_norm=weights["final_norm"].ctypes.data, **ptrs)
        self._c = OrcConfig(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim,
                            cfg.ffn_dim, cfg.vocab, max_seq, cfg.rope_theta, cfg.rms_eps)
        self._h = lib().orc_create(ctypes.byref(self._c), ctypes.byref(self._w), precision)
        if not self._h:
            raise ValueError("oracle rejected the configuration")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().orc_destroy(h)
            self._h = None

    @property
    def pos(self) -> int:
        return lib().orc_pos(self._h)

    def reset(self) -> None:
        lib().orc_reset(self._h)

    def forward(self, token: int) -> np.ndarray:
        logits = np.empty(self.cfg.vocab, dtype=_real(self.precision))
        if lib().orc_forward(self._h, int(token), logits.ctypes.data) != 0:
            raise ValueError("oracle forward refused (cache full or token out of range)")
        return logits

    def prefill(self, tokens) -> np.ndarray:
        logits = None
        for t in tokens:
            logits = self.forward(t)
        return logits

    def kv_row(self, layer: int, kv: int, head: int, pos: int) -> np.ndarray:
        out = np.empty(self.cfg.head_dim, dtype=np.uint16)
        lib().orc_kv_row(self._h, layer, kv, head, pos, out.ctypes.data)
        return out


def generate(cfg, weights, prompt, n_new, max_seq=None, precision=32, keep_logits=True):
    """Greedy decode: returns (tokens [n_new], logits [(n_new + 1), V] or None).

    logits[0] are those of the last prompt position; tokens[i] = argmax(logits[i]); logits[i + 1] are
    those after the forward of tokens[i].
    """
    m = Model(cfg, weights, max_seq or (len(prompt) + n_new), precision)
    cur = m.prefill(prompt)
    toks = np.empty(n_new, dtype=np.int32)
    L = [cur] if keep_logits else None
    for i in range(n_new):
        toks[i] = argmax(cur)
        cur = m.forward(int(toks[i]))
        if keep_logits:
            L.append(cur)
    return toks, (np.stack(L) if keep_logits else None)
