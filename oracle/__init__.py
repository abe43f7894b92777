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


class OrcMoe(ctypes.Structure):
    _fields_ = [("n_experts", ctypes.c_int), ("top_k", ctypes.c_int), ("expert_ffn", ctypes.c_int)] + \
        [(n, P) for n in ("router", "gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s")]


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
            "orc_set_moe": ([P, ctypes.POINTER(OrcMoe)], i), "orc_moe_ffn": ([P, i, P, P], None),
            "orc_e4m3_to_double": ([ctypes.c_uint8], d),
            "orc_gemv_fp8_f32": ([P, P, P, i, i, P], None), "orc_gemv_fp8_f64": ([P, P, P, i, i, P], None),
            "orc_topk_softmax_f64": ([P, i, i, P, P], None), "orc_route_margin": ([P, i], d),
            "orc_route_ids": ([P, P, P], i),
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


def e4m3_to_double(code: int) -> float:
    return lib().orc_e4m3_to_double(code)


def gemv_fp8(q, scale, x, precision=64):
    """y = diag(scale) E4M3(q) x for codes q [M, K] (uint8) and row scales [M] (float32)."""
    q, pq = _c(q, np.uint8)
    sc, ps = _c(scale, np.float32)
    x, px = _c(x, _real(precision))
    M, K = q.shape
    y = np.empty(M, dtype=_real(precision))
    getattr(lib(), f"orc_gemv_fp8_f{precision}")(pq, ps, px, M, K, y.ctypes.data)
    return y


def topk_softmax(r, k):
    """(indices of the k largest of r, lowest index first on ties, in descending order; softmax over them)."""
    r, pr = _c(r, np.float64)
    idx = np.empty(k, dtype=np.int32)
    w = np.empty(k, dtype=np.float64)
    lib().orc_topk_softmax_f64(pr, r.size, k, idx.ctypes.data, w.ctypes.data)
    return idx, w


def argmax(v) -> int:
    v = np.ascontiguousarray(v)
    if v.dtype == np.float64:
        return lib().orc_argmax_f64(v.ctypes.data, v.size)
    v = v.astype(np.float32, copy=False)
    return lib().orc_argmax_f32(v.ctypes.data, v.size)


class Model:
    """The oracle decoder over borrowed weights (dict from synth.model_weights, or synth.moe_weights for a
    sparse-MoE config)."""

    def __init__(self, cfg, weights: dict, max_seq: int, precision: int = 32):
        self.cfg, self.precision, self.max_seq = cfg, precision, max_seq
        self._keep = weights
        L = cfg.n_layers
        self._arrays = {}
        ptrs = {}
        moe = getattr(cfg, "n_experts", 0) > 0
        for name in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down"):
            # a MoE model has no dense FFN matrices: null pointers, never read
            arr = (P * max(L, 1))(*[(None if moe and name in ("w_gate", "w_up", "w_down")
                                     else weights["layers"][l][name].ctypes.data) for l in range(L)])
            self._arrays[name] = arr
            ptrs[name] = ctypes.cast(arr, P)
        self._w = OrcWeights(embed=weights["embed"].ctypes.data, lm_head=weights["lm_head"].ctypes.data,
                             final_norm=weights["final_norm"].ctypes.data, **ptrs)
        self._c = OrcConfig(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim,
                            cfg.ffn_dim, cfg.vocab, max_seq, cfg.rope_theta, cfg.rms_eps)
        self._h = lib().orc_create(ctypes.byref(self._c), ctypes.byref(self._w), precision)
        if not self._h:
            raise ValueError("oracle rejected the configuration")
        if moe:
            mp = {}
            for name, key in (("router", "router"), ("gate_q", "gate_q"), ("up_q", "up_q"), ("down_q", "down_q"),
                              ("gate_s", "gate_s"), ("up_s", "up_s"), ("down_s", "down_s")):
                arrs = [np.ascontiguousarray(weights["layers"][l][key]) for l in range(L)]
                self._arrays["moe_" + name] = arrs
                tbl = (P * max(L, 1))(*[a.ctypes.data for a in arrs])
                self._arrays["moe_" + name + "_tbl"] = tbl
                mp[name] = ctypes.cast(tbl, P)
            self._moe = OrcMoe(cfg.n_experts, cfg.top_k, cfg.expert_ffn, **mp)
            if lib().orc_set_moe(self._h, ctypes.byref(self._moe)) != 0:
                raise ValueError("oracle rejected the MoE description")

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

    def forward(self, token: int, want_logits: bool = True):
        """One forward at the current position; its logits, or None when want_logits is False (the final norm
        and LM head are then skipped; cache and state are the same)."""
        logits = np.empty(self.cfg.vocab, dtype=_real(self.precision)) if want_logits else None
        if lib().orc_forward(self._h, int(token), logits.ctypes.data if want_logits else None) != 0:
            raise ValueError("oracle forward refused (cache full or token out of range)")
        return logits

    def prefill(self, tokens) -> np.ndarray:
        """Forward every prompt token; the logits of the last one (the others' LM heads are skipped)."""
        tokens = list(tokens)
        for t in tokens[:-1]:
            self.forward(t, want_logits=False)
        return self.forward(tokens[-1]) if tokens else None

    def route(self):
        """The routing of the last forward (sparse-MoE models): (ids [n_layers, top_k] in selection order,
        gaps [n_layers]: each layer's k-th selected router logit minus its best unselected one)."""
        L, k = self.cfg.n_layers, self.cfg.top_k
        ids = np.empty((L, k), dtype=np.int32)
        gaps = np.empty(L, dtype=np.float64)
        if lib().orc_route_ids(self._h, ids.ctypes.data, gaps.ctypes.data) != 0:
            raise ValueError("not a sparse-MoE model")
        return ids, gaps

    def moe_ffn(self, layer: int, u) -> np.ndarray:
        """The sparse-MoE FFN output of `layer` for a normalised input u."""
        u = np.ascontiguousarray(u, dtype=_real(self.precision))
        out = np.empty(self.cfg.d_model, dtype=_real(self.precision))
        lib().orc_moe_ffn(self._h, layer, u.ctypes.data, out.ctypes.data)
        return out

    def route_margin(self, reset: bool = True) -> float:
        """Smallest routing margin (top_k-th router logit minus the best unselected one) over the MoE layers
        evaluated since the last reset; +inf for a dense model or when every expert is selected."""
        return lib().orc_route_margin(self._h, int(reset))

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
