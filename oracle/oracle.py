"""Python face of the CPU oracle (TEST INFRASTRUCTURE ONLY).

Only tests, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline and
reference legs may import this module.  It compiles and loads
``moe_oracle.c`` (plain C, fp64) with gcc and composes its primitives into
the layer.  It imports nothing from the CUDA package and the CUDA package
imports nothing from here.

Conversions to double (bf16, fp16 and fp32 to float64) are exact, so every
input reaches the C code bit-for-bit.

Layer (Swiftlet project pages, the Swiftlet README "How it works": k of E routed experts
plus a resident shared expert; the combine, SwiGLU and sigmoid gate follow the
Qwen3-Next / Qwen3.5-3.6 layer the pages name):
    logits = W_r x + b,  s = w_sg . x
    (idx, w) = top-k of logits, softmax over the k selected
    y = sum_r w_r * E_{idx_r}(x) + sigmoid(s) * E_shared(x)
    E(x) = W_d (silu(W_g x) * (W_u x))
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_OMP_PATH = os.path.join(_OUT_DIR, "liboracle_omp.so")
_lock = threading.Lock()
_lib = None
_lib_omp = None
_threads = 1

_D = ctypes.POINTER(ctypes.c_double)
_U32 = ctypes.POINTER(ctypes.c_uint32)
_I32 = ctypes.POINTER(ctypes.c_int32)


def _compile(path: str, extra, force: bool):
    if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        tmp = path + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-ffp-contract=off", *extra, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, path)
    return path


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/_build/liboracle.so (gcc, -O2, no
    fast-math), and the same source with OpenMP into liboracle_omp.so."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    _compile(_OMP_PATH, ["-fopenmp"], force)
    return _compile(_LIB_PATH, [], force)


def set_threads(n: int) -> None:
    """Run the oracle's loops over output rows on n threads (n > 1 loads the
    OpenMP build; every output is computed as in the plain build)."""
    global _threads
    _threads = max(1, int(n))
    if _threads > 1:
        lib().oracle_set_threads(_threads)


def lib():
    global _lib, _lib_omp
    with _lock:
        if _threads > 1:
            if _lib_omp is None:
                build()
                _lib_omp = _bind(ctypes.CDLL(_OMP_PATH))
            return _lib_omp
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(L):
    c_int = ctypes.c_int
    L.oracle_router.argtypes = [c_int, c_int, c_int, _D, _D, _D, _D, _D, _D]
    L.oracle_topk.argtypes = [c_int, c_int, _D, _I32, _D]
    L.oracle_dequant.argtypes = [c_int, c_int, c_int, c_int, _U32, _D, _D, _D]
    L.oracle_qmatvec.argtypes = [c_int, c_int, c_int, c_int, _U32, _D, _D, _D, _D]
    L.oracle_expert.argtypes = [c_int, c_int, c_int, c_int] + [_U32, _D, _D] * 3 + [_D, _D, _D]
    L.oracle_bucket.argtypes = [c_int, c_int, c_int, _I32, _I32, _I32, _I32, _I32]
    L.oracle_set_threads.argtypes = [c_int]
    for f in ("oracle_router", "oracle_topk", "oracle_dequant", "oracle_qmatvec",
              "oracle_expert", "oracle_bucket", "oracle_set_threads"):
        getattr(L, f).restype = None
    return L


# ---------------------------------------------------------------- marshalling

def _np(a):
    """torch tensor or array -> numpy (CPU); bf16 goes through fp32 (exact)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu()
            if a.dtype == torch.bfloat16:
                a = a.float()
            return a.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a)


def f64(a) -> np.ndarray:
    return np.ascontiguousarray(_np(a), dtype=np.float64)


def u32(a) -> np.ndarray:
    a = np.ascontiguousarray(_np(a))
    if a.dtype == np.int32:
        a = a.view(np.uint32)
    assert a.dtype == np.uint32
    return a


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


# ---------------------------------------------------------------- primitives

def router(x, w_router, bias=None, w_sg=None):
    """-> (logits [T,E], s [T]) in float64."""
    x, wr = f64(x), f64(w_router)
    T, H = x.shape
    E = wr.shape[0]
    logits = np.zeros((T, E))
    s = np.zeros(T)
    b = f64(bias) if bias is not None else None
    g = f64(w_sg) if w_sg is not None else None
    lib().oracle_router(T, H, E, _p(x, _D), _p(wr, _D), _p(b, _D) if b is not None else None,
                        _p(g, _D) if g is not None else None, _p(logits, _D), _p(s, _D))
    return logits, s


def topk(logits, k):
    """-> (idx [T,k] int32, w [T,k] float64) for logits [T,E] (or [E])."""
    lg = f64(logits)
    one = lg.ndim == 1
    lg = lg.reshape(-1, lg.shape[-1])
    T, E = lg.shape
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k))
    for t in range(T):
        row = np.ascontiguousarray(lg[t])
        lib().oracle_topk(E, k, _p(row, _D), _p(idx[t], _I32), _p(w[t], _D))
    return (idx[0], w[0]) if one else (idx, w)


def dequant(q, scale, bias, group, bits=4):
    q, s, b = u32(q), f64(scale), f64(bias)
    n_out, n_in = q.shape[0], q.shape[1] * (32 // bits)
    W = np.zeros((n_out, n_in))
    lib().oracle_dequant(n_out, n_in, group, bits, _p(q, _U32), _p(s, _D), _p(b, _D), _p(W, _D))
    return W


def qmatvec(q, scale, bias, group, v, bits=4):
    q, s, b, v = u32(q), f64(scale), f64(bias), f64(v)
    n_out, n_in = q.shape[0], q.shape[1] * (32 // bits)
    y = np.zeros(n_out)
    lib().oracle_qmatvec(n_out, n_in, group, bits, _p(q, _U32), _p(s, _D), _p(b, _D), _p(v, _D), _p(y, _D))
    return y


class ExpertView:
    """One expert's nine arrays, converted once to the oracle's types."""

    def __init__(self, mats: dict, e: int, prefix: str = ""):
        self.bits = int(mats.get("bits", 4))
        self.m = []
        for name in ("gate", "up", "down"):
            self.m += [u32(mats[prefix + "q_" + name][e]), f64(mats[prefix + "s_" + name][e]),
                       f64(mats[prefix + "b_" + name][e])]
        self.inter = self.m[0].shape[0]
        self.hidden = self.m[0].shape[1] * (32 // self.bits)


def expert(view: ExpertView, group: int, x):
    """E(x) for one token x [H] -> [H] float64."""
    x = f64(x).reshape(-1)
    H, I = view.hidden, view.inter
    y = np.zeros(H)
    work = np.zeros(3 * I)
    args = []
    for j, a in enumerate(view.m):
        args.append(_p(a, _U32 if j % 3 == 0 else _D))
    lib().oracle_expert(H, I, group, view.bits, *args, _p(x, _D), _p(y, _D), _p(work, _D))
    return y


def bucket(idx, n_experts):
    idx = np.ascontiguousarray(_np(idx), dtype=np.int32)
    T, k = idx.shape
    counts = np.zeros(n_experts, np.int32)
    offsets = np.zeros(n_experts + 1, np.int32)
    pt = np.zeros(T * k, np.int32)
    pr = np.zeros(T * k, np.int32)
    lib().oracle_bucket(T, k, n_experts, _p(idx, _I32), _p(counts, _I32), _p(offsets, _I32),
                        _p(pt, _I32), _p(pr, _I32))
    return counts, offsets, pt, pr


def sigmoid(v):
    return 1.0 / (1.0 + np.exp(-np.asarray(v, dtype=np.float64)))


# ---------------------------------------------------------------- the layer

class Layer:
    """Holds a layer's inputs in oracle form; experts are converted lazily."""

    def __init__(self, layer: dict, group: int, top_k: int):
        self.raw = layer
        self.group = group
        self.k = top_k
        self.w_router = f64(layer["w_router"])
        self.bias = f64(layer["router_bias"]) if layer.get("router_bias") is not None else None
        self.has_shared = "shared_q_gate" in layer
        self.w_sg = f64(layer["w_shared_gate"]) if self.has_shared else None
        self.shared = ExpertView(layer, 0, "shared_") if self.has_shared else None
        self._cache = {}

    def expert_view(self, e: int) -> ExpertView:
        v = self._cache.get(e)
        if v is None:
            v = ExpertView(self.raw, int(e))
            if len(self._cache) < 64:
                self._cache[e] = v
        return v

    def route(self, x):
        logits, s = router(x, self.w_router, self.bias, self.w_sg)
        idx, w = topk(logits, self.k)
        return logits, s, idx, w

    def forward(self, x, tokens=None):
        """-> dict(y [T,H] f64, idx, w, s, logits) for x [T,H]; `tokens`
        restricts the expert work to a subset of rows (others left at 0)."""
        x = f64(x)
        logits, s, idx, w = self.route(x)
        T, H = x.shape
        y = np.zeros((T, H))
        rows = range(T) if tokens is None else tokens
        for t in rows:
            acc = np.zeros(H)
            for r in range(self.k):
                acc += w[t, r] * expert(self.expert_view(idx[t, r]), self.group, x[t])
            if self.has_shared:
                acc += sigmoid(s[t]) * expert(self.shared, self.group, x[t])
            y[t] = acc
        return {"y": y, "idx": idx, "w": w, "s": s, "logits": logits}
