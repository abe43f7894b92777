"""Python binding of the GB300 persistent decode monokernel (C ABI in include/kie.h).

The binding only marshals arguments: every step of decode runs in the CUDA kernels of ``libkie.so``.
PyTorch is used for two things only, device memory (``torch.empty`` buffers handed to
``kie_create_with_buffers``) and the CUDA stream the library launches on. There is no CPU fallback: if
the extension is not built, or no GPU is present, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
_INCLUDE = os.path.join(_ROOT, "include")
_BUILD = os.path.join(_ROOT, "_build")
LIB_PATH = os.path.join(_HERE, "libkie.so")
SOURCES = ("kie_api.cu", "kie_decode.cu", "kie_gemv.cu", "kie_prefill.cu")
HEADERS = ("kie_layout.h", "kie_device.cuh", "kie_decode.cuh", "kie_prefill.cuh", "kie_tcgemm.cuh", "kie_tcattn.cuh")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

KIE_OK, KIE_ERR_INVALID, KIE_ERR_OOM, KIE_ERR_CAPACITY = 0, -1, -2, -3
KIE_ERR_CUDA, KIE_ERR_LAUNCH, KIE_ERR_TIMEOUT = -4, -5, -6
ERROR_NAMES = {0: "KIE_OK", -1: "KIE_ERR_INVALID", -2: "KIE_ERR_OOM", -3: "KIE_ERR_CAPACITY", -4: "KIE_ERR_CUDA",
               -5: "KIE_ERR_LAUNCH", -6: "KIE_ERR_TIMEOUT"}


# ---- build ------------------------------------------------------------------------------------------

def _nvcc() -> str:
    if os.environ.get("NVCC"):
        return os.environ["NVCC"]
    return "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc"


def compile_cmds() -> list[list[str]]:
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{_INCLUDE}", f"-I{_CSRC}"]
    return [[_nvcc(), *flags, "-c", os.path.join(_CSRC, s), "-o", os.path.join(_BUILD, s + ".o")] for s in SOURCES]


def link_cmd() -> list[str]:
    return [_nvcc(), *ARCH, "-shared", "-o", LIB_PATH, *[os.path.join(_BUILD, s + ".o") for s in SOURCES]]


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(_CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(_INCLUDE, "kie.h")]
    return any(os.path.getmtime(f) > t for f in deps)


# The sources a decode launch is built from: the kernel, its ring and GEMV consumer, the packed layout, and the
# host code that plans and launches it.
DECODE_SOURCES = ("kie_decode.cu", "kie_device.cuh", "kie_decode.cuh", "kie_layout.h", "kie_api.cu")


def source_digest(files=DECODE_SOURCES) -> str:
    """First 16 hex digits of a SHA-256 over the named CUDA sources (names and contents), by default those of
    the decode launch: it identifies the kernel build that a stored profile was taken from."""
    import hashlib
    h = hashlib.sha256()
    for f in sorted(files):
        h.update(f.encode())
        with open(os.path.join(_CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def build(force: bool = False) -> str:
    """Compile libkie.so in-tree for sm_103a (the translation units in parallel, then link)."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), compile_cmds()))
    for r in results:
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    r = subprocess.run(link_cmd(), capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc link failed:\n" + r.stdout + r.stderr)
    return LIB_PATH


# ---- C structs --------------------------------------------------------------------------------------

P = ctypes.c_void_p


class KieConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim",
                                             "ffn_dim", "vocab", "max_seq")] + \
               [("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float)]


class KieWeights(ctypes.Structure):
    _fields_ = [(n, P) for n in ("embed", "lm_head", "final_norm", "attn_norm", "wq", "wk", "wv", "wo",
                                 "ffn_norm", "w_gate", "w_up", "w_down")]


class KieMoeConfig(ctypes.Structure):
    _fields_ = [("n_experts", ctypes.c_int), ("top_k", ctypes.c_int)]


class KieMoeWeights(ctypes.Structure):
    _fields_ = [(n, P) for n in ("router", "gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s")]


class KieBufferSizes(ctypes.Structure):
    _fields_ = [("weights_bytes", ctypes.c_size_t), ("kv_bytes", ctypes.c_size_t),
                ("workspace_bytes", ctypes.c_size_t), ("n_cta", ctypes.c_int)]


class KieBarrierStats(ctypes.Structure):
    _fields_ = [("barriers", ctypes.c_int64), ("mean_wait_ns", ctypes.c_double),
                ("mean_latency_ns", ctypes.c_double), ("total_ns", ctypes.c_double)]


# Every entry point of include/kie.h with its ctypes signature.
SIGNATURES = {
    "kie_query_buffers": ([P, ctypes.c_int, P], ctypes.c_int),
    "kie_create": ([P, P, P, P], ctypes.c_int),
    "kie_create_with_buffers": ([P, P, P, P, ctypes.c_size_t, P, ctypes.c_size_t, P, ctypes.c_size_t, P], ctypes.c_int),
    "kie_prefill": ([P, P, ctypes.c_int], ctypes.c_int),
    "kie_decode": ([P, ctypes.c_int, P], ctypes.c_int),
    "kie_decode_async": ([P, ctypes.c_int, P], ctypes.c_int),
    "kie_sync": ([P], ctypes.c_int),
    "kie_decode_forced": ([P, ctypes.c_int, P, P, P], ctypes.c_int),
    "kie_decode_forced_routed": ([P, ctypes.c_int, P, P, P, P, P], ctypes.c_int),
    "kie_get_logits": ([P, P], ctypes.c_int),
    "kie_position": ([P], ctypes.c_int),
    "kie_reset": ([P], ctypes.c_int),
    "kie_set_timeout_ns": ([P, ctypes.c_uint64], ctypes.c_int),
    "kie_get_barrier_stats": ([P, P], ctypes.c_int),
    "kie_get_barrier_trace": ([P, ctypes.c_int, ctypes.c_int, P, P], ctypes.c_int),
    "kie_debug_skip_arrival": ([P, ctypes.c_int, ctypes.c_int], ctypes.c_int),
    "kie_n_cta": ([P], ctypes.c_int),
    "kie_profile_attention": ([P, ctypes.c_int, ctypes.c_int], ctypes.c_int),
    "kie_last_error": ([P], ctypes.c_char_p),
    "kie_destroy": ([P], None),
    "kie_gemv_packed_bytes": ([ctypes.c_int, ctypes.c_int], ctypes.c_size_t),
    "kie_gemv_pack": ([P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P], ctypes.c_int),
    "kie_gemv": ([P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P], ctypes.c_int),
    "kie_decode_noalloc": ([P, ctypes.c_int, P], ctypes.c_int),
    "kie_packed_offset": ([ctypes.c_int] * 5, ctypes.c_int64),
    "kie_rows_of_cta": ([ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P], ctypes.c_int),
    "kie_query_buffers_moe": ([P, P, ctypes.c_int, P], ctypes.c_int),
    "kie_create_moe": ([P, P, P, P, P, P], ctypes.c_int),
    "kie_create_moe_with_buffers": ([P, P, P, P, P, P, ctypes.c_size_t, P, ctypes.c_size_t, P, ctypes.c_size_t, P],
                                    ctypes.c_int),
    "kie_packed_offset_fp8": ([ctypes.c_int] * 5, ctypes.c_int64),
    "kie_tc_tile_offset": ([ctypes.c_int] * 4, ctypes.c_int64),
}

_lib = None


def lib():
    """The loaded libkie.so. Raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() (or "
                               "persistent_monokernel_decode_gb300.build()) first")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes, fn.restype = args, res
        _lib = L
    return _lib


class KieError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


def _check(rc: int, ctx=None):
    if rc != KIE_OK:
        raise KieError(rc, (lib().kie_last_error(ctx) or b"").decode())


# ---- thin wrappers with the C names --------------------------------------------------------------------

def make_config(model, max_seq: int) -> KieConfig:
    return KieConfig(model.n_layers, model.d_model, model.n_heads, model.n_kv_heads, model.head_dim,
                     model.ffn_dim, model.vocab, max_seq, model.rope_theta, model.rms_eps)


def make_moe_config(model) -> KieMoeConfig:
    return KieMoeConfig(model.n_experts, model.top_k)


def is_moe(model) -> bool:
    return getattr(model, "n_experts", 0) > 0


def kie_query_buffers(cfg: KieConfig, n_cta: int = 0, moe: KieMoeConfig = None) -> KieBufferSizes:
    out = KieBufferSizes()
    if moe is None:
        _check(lib().kie_query_buffers(ctypes.byref(cfg), n_cta, ctypes.byref(out)))
    else:
        _check(lib().kie_query_buffers_moe(ctypes.byref(cfg), ctypes.byref(moe), n_cta, ctypes.byref(out)))
    return out


def _pointer_table(keep: dict, name: str, arrays: list):
    keep[name] = arrays
    tbl = (P * max(len(arrays), 1))(*[a.ctypes.data for a in arrays])
    keep[name + "_tbl"] = tbl
    return ctypes.cast(tbl, P)


class _HostMoeWeights:
    """ctypes view of the sparse-MoE part of a weights dict (router fp16 bits, FP8 codes, fp32 row scales)."""

    def __init__(self, weights: dict, n_layers: int):
        self.keep = weights
        self.arrays = {}
        dtypes = {"router": np.uint16, "gate_q": np.uint8, "up_q": np.uint8, "down_q": np.uint8,
                  "gate_s": np.float32, "up_s": np.float32, "down_s": np.float32}
        ptrs = {name: _pointer_table(self.arrays, name,
                                     [np.ascontiguousarray(weights["layers"][l][name], dtype=dt) for l in range(n_layers)])
                for name, dt in dtypes.items()}
        self.struct = KieMoeWeights(**ptrs)


class _HostWeights:
    """ctypes view of a weights dict (fp16 bit arrays) that keeps every array alive. The dense FFN matrices are
    left NULL when ffn is False (sparse-MoE models)."""

    def __init__(self, weights: dict, n_layers: int, ffn: bool = True):
        self.keep = weights
        self.arrays = {}
        ptrs = {}
        names = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm") + (("w_gate", "w_up", "w_down") if ffn else ())
        for name in names:
            arrs = [np.ascontiguousarray(weights["layers"][l][name], dtype=np.uint16) for l in range(n_layers)]
            self.arrays[name] = arrs
            tbl = (P * max(n_layers, 1))(*[a.ctypes.data for a in arrs])
            self.arrays[name + "_tbl"] = tbl
            ptrs[name] = ctypes.cast(tbl, P)
        for name in ("embed", "lm_head", "final_norm"):
            self.arrays[name] = np.ascontiguousarray(weights[name], dtype=np.uint16)
        self.struct = KieWeights(embed=self.arrays["embed"].ctypes.data, lm_head=self.arrays["lm_head"].ctypes.data,
                                 final_norm=self.arrays["final_norm"].ctypes.data, **ptrs)


def _torch():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("persistent_monokernel_decode_gb300 needs a CUDA GPU; none is available")
    return torch


class Decoder:
    """One decode context (kie_ctx): repacked weights, KV cache and workspace in torch-allocated HBM."""

    def __init__(self, model, weights: dict, max_seq: int, stream=None):
        """model: a ModelConfig-like object; a sparse-MoE model (n_experts > 0, with top_k, and ffn_dim the expert
        width) takes the weights of synth.moe_weights (router, FP8 experts with row scales)."""
        torch = _torch()
        self.model, self.max_seq = model, max_seq
        self.cfg = make_config(model, max_seq)
        self.moe = make_moe_config(model) if is_moe(model) else None
        sizes = kie_query_buffers(self.cfg, 0, self.moe)
        dev = torch.device("cuda", torch.cuda.current_device())
        self._wbuf = torch.empty(sizes.weights_bytes, dtype=torch.uint8, device=dev)
        self._kvbuf = torch.empty(sizes.kv_bytes, dtype=torch.uint8, device=dev)
        self._wsbuf = torch.empty(sizes.workspace_bytes, dtype=torch.uint8, device=dev)
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        hw = _HostWeights(weights, model.n_layers, ffn=self.moe is None)
        ctx = P()
        bufs = (P(self.stream.cuda_stream), self._wbuf.data_ptr(), sizes.weights_bytes, self._kvbuf.data_ptr(),
                sizes.kv_bytes, self._wsbuf.data_ptr(), sizes.workspace_bytes, ctypes.byref(ctx))
        if self.moe is None:
            rc = lib().kie_create_with_buffers(ctypes.byref(self.cfg), ctypes.byref(hw.struct), *bufs)
        else:
            mw = _HostMoeWeights(weights, model.n_layers)
            rc = lib().kie_create_moe_with_buffers(ctypes.byref(self.cfg), ctypes.byref(self.moe),
                                                   ctypes.byref(hw.struct), ctypes.byref(mw.struct), *bufs)
        _check(rc, None)
        self.ctx = ctx
        self.n_cta = lib().kie_n_cta(ctx)

    def close(self):
        if getattr(self, "ctx", None):
            lib().kie_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, tokens) -> None:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        _check(lib().kie_prefill(self.ctx, t.ctypes.data, t.size), self.ctx)

    def decode(self, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.int32)
        _check(lib().kie_decode(self.ctx, n, out.ctypes.data), self.ctx)
        return out

    @staticmethod
    def _device_tokens(out_dev, n: int) -> int:
        """Address of out_dev after checking that it can take n int32 tokens written by the kernel: a contiguous
        int32 CUDA tensor of at least n elements (the kernel writes n values there, unchecked)."""
        torch = _torch()
        if not isinstance(out_dev, torch.Tensor) or not out_dev.is_cuda:
            raise ValueError("out_dev must be a CUDA tensor")
        if out_dev.dtype != torch.int32 or not out_dev.is_contiguous() or out_dev.numel() < n:
            raise ValueError(f"out_dev must be a contiguous int32 tensor of at least {n} elements "
                             f"(got {out_dev.dtype}, {out_dev.numel()} elements, contiguous={out_dev.is_contiguous()})")
        return out_dev.data_ptr()

    def decode_async(self, n: int, out_dev) -> None:
        """Enqueue n greedy tokens into the device int32 tensor out_dev; no synchronisation."""
        _check(lib().kie_decode_async(self.ctx, n, self._device_tokens(out_dev, n)), self.ctx)

    def decode_noalloc(self, n: int, out_dev) -> None:
        """n greedy tokens into the device int32 tensor out_dev, with no device allocation (static scratch)."""
        _check(lib().kie_decode_noalloc(self.ctx, n, self._device_tokens(out_dev, n)), self.ctx)

    def sync(self) -> None:
        _check(lib().kie_sync(self.ctx), self.ctx)

    def decode_forced(self, forced, want_logits: bool = True):
        f = np.ascontiguousarray(forced, dtype=np.int32)
        toks = np.empty(f.size, dtype=np.int32)
        logits = np.empty((f.size, self.model.vocab), dtype=np.float32) if want_logits else None
        _check(lib().kie_decode_forced(self.ctx, f.size, f.ctypes.data, toks.ctypes.data,
                                       logits.ctypes.data if want_logits else None), self.ctx)
        return toks, logits

    def decode_forced_routed(self, forced, forced_experts=None, want_logits: bool = True, want_experts: bool = True):
        """Teacher forcing of tokens and (sparse MoE) of expert selections: forced_experts [n, n_layers, top_k] or
        None. Returns (tokens [n], logits [n, V] or None, own selections [n, n_layers, top_k] or None). May start a
        sequence (then tokens[0] is -1)."""
        f = np.ascontiguousarray(forced, dtype=np.int32)
        n, L, k = f.size, self.model.n_layers, getattr(self.model, "top_k", 0)
        toks = np.empty(n, dtype=np.int32)
        logits = np.empty((n, self.model.vocab), dtype=np.float32) if want_logits else None
        fe = None
        if forced_experts is not None:
            fe = np.ascontiguousarray(forced_experts, dtype=np.int32)
            if fe.shape != (n, L, k):
                raise ValueError(f"forced_experts must have shape {(n, L, k)}, not {fe.shape}")
        own = np.empty((n, L, k), dtype=np.int32) if want_experts else None
        _check(lib().kie_decode_forced_routed(self.ctx, n, f.ctypes.data, None if fe is None else fe.ctypes.data,
                                              toks.ctypes.data, None if logits is None else logits.ctypes.data,
                                              None if own is None else own.ctypes.data), self.ctx)
        return toks, logits, own

    def logits(self) -> np.ndarray:
        out = np.empty(self.model.vocab, dtype=np.float32)
        _check(lib().kie_get_logits(self.ctx, out.ctypes.data), self.ctx)
        return out

    @property
    def position(self) -> int:
        return lib().kie_position(self.ctx)

    def reset(self) -> None:
        _check(lib().kie_reset(self.ctx), self.ctx)

    def set_timeout_ns(self, ns: int) -> None:
        _check(lib().kie_set_timeout_ns(self.ctx, ns), self.ctx)

    def barrier_stats(self) -> dict:
        st = KieBarrierStats()
        _check(lib().kie_get_barrier_stats(self.ctx, ctypes.byref(st)), self.ctx)
        return {"barriers": st.barriers, "mean_wait_ns": st.mean_wait_ns,
                "mean_latency_ns": st.mean_latency_ns, "total_ns": st.total_ns}

    def barrier_trace(self, first: int = 0, count: int = 4096):
        """(arrive_ns [m, n_cta] uint64, wait_ns [m, n_cta] uint32) for barriers first..first+m-1."""
        arrive = np.zeros((count, self.n_cta), dtype=np.uint64)
        wait = np.zeros((count, self.n_cta), dtype=np.uint32)
        m = lib().kie_get_barrier_trace(self.ctx, first, count, arrive.ctypes.data, wait.ctypes.data)
        if m < 0:
            _check(m, self.ctx)
        return arrive[:m], wait[:m]

    def profile_attention(self, c: int, n_layers: int) -> None:
        """The split-KV attention step alone for layers [0, n_layers) over c cached positions (profiling)."""
        _check(lib().kie_profile_attention(self.ctx, c, n_layers), self.ctx)

    def debug_skip_arrival(self, cta: int, barrier: int) -> None:
        _check(lib().kie_debug_skip_arrival(self.ctx, cta, barrier), self.ctx)


# ---- standalone GEMV ----------------------------------------------------------------------------------

def gemv_pack(W, n_cta: int = 0):
    """Pack a row-major fp16 CUDA tensor W [M, K] into the per-CTA tile layout (returns a new tensor)."""
    torch = _torch()
    M, K = W.shape
    packed = torch.empty(M * K, dtype=torch.int16, device=W.device)
    _check(lib().kie_gemv_pack(W.data_ptr(), M, K, n_cta, packed.data_ptr(),
                               P(torch.cuda.current_stream().cuda_stream)))
    return packed


def gemv(packed, x, M: int, K: int, n_cta: int = 0, y=None):
    """y = W x (fp32) from a packed fp16 W and an fp16 CUDA vector x, on the current stream."""
    torch = _torch()
    if y is None:
        y = torch.empty(M, dtype=torch.float32, device=x.device)
    _check(lib().kie_gemv(packed.data_ptr(), x.data_ptr(), y.data_ptr(), M, K, n_cta,
                          P(torch.cuda.current_stream().cuda_stream)))
    return y


def packed_offset(M: int, K: int, n_cta: int, r: int, c: int) -> int:
    return lib().kie_packed_offset(M, K, n_cta, r, c)


def tc_tile_offset(M: int, K: int, r: int, c: int) -> int:
    return lib().kie_tc_tile_offset(M, K, r, c)


def packed_offset_fp8(M: int, K: int, n_cta: int, r: int, c: int) -> int:
    return lib().kie_packed_offset_fp8(M, K, n_cta, r, c)


def rows_of_cta(M: int, n_cta: int, cta: int):
    r0, r1 = ctypes.c_int(), ctypes.c_int()
    _check(lib().kie_rows_of_cta(M, n_cta, cta, ctypes.byref(r0), ctypes.byref(r1)))
    return r0.value, r1.value
