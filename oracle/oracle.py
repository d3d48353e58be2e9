"""Python face of the CPU oracle (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module. It builds ``liboracle.so`` from ``llama_ref.c``
with gcc and calls it through ctypes on numpy arrays. It imports nothing from
the CUDA package and the CUDA package imports nothing from it.

The arithmetic lives in ``llama_ref.c``; its header lists the definitions it
follows ("3 · L'interpréteur sur GPU", §3.2, the seven fused instructions, read
as the textbook Llama decoder).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "llama_ref.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

u16p = ctypes.POINTER(ctypes.c_uint16)
f64p = ctypes.POINTER(ctypes.c_double)
i32p = ctypes.POINTER(ctypes.c_int32)


class RefConfig(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("n_heads", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
        ("vocab", ctypes.c_int), ("tied", ctypes.c_int),
        ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double),
    ]


class RefWeights(ctypes.Structure):
    _fields_ = [
        ("embed", u16p), ("lm_head", u16p), ("final_norm", u16p),
        ("attn_norm", ctypes.POINTER(u16p)), ("wq", ctypes.POINTER(u16p)),
        ("wk", ctypes.POINTER(u16p)), ("wv", ctypes.POINTER(u16p)),
        ("wo", ctypes.POINTER(u16p)), ("mlp_norm", ctypes.POINTER(u16p)),
        ("wgate", ctypes.POINTER(u16p)), ("wup", ctypes.POINTER(u16p)),
        ("wdown", ctypes.POINTER(u16p)),
    ]


def build(force: bool = False) -> str:
    """Compile liboracle.so (plain C, portable flags, no -march)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                       os.path.getmtime(_SRC[:-2] + ".h"))):
            return _LIB_PATH
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True, cwd=_HERE)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        path = build()
        L = ctypes.CDLL(path)
        L.ref_bf16_to_f64.restype = ctypes.c_double
        L.ref_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.ref_f64_to_bf16.restype = ctypes.c_uint16
        L.ref_f64_to_bf16.argtypes = [ctypes.c_double]
        L.ref_rmsnorm.argtypes = [f64p, u16p, ctypes.c_int, ctypes.c_double, f64p]
        L.ref_rope.argtypes = [f64p, ctypes.c_int, ctypes.c_int, ctypes.c_double]
        L.ref_silu.restype = ctypes.c_double
        L.ref_silu.argtypes = [ctypes.c_double]
        L.ref_matvec.argtypes = [u16p, ctypes.c_int, ctypes.c_int, f64p, f64p, ctypes.c_int]
        L.ref_attend.argtypes = [f64p, u16p, u16p, ctypes.c_int, ctypes.c_int, ctypes.c_long,
                                 ctypes.c_double, f64p]
        L.ref_decode_step.restype = ctypes.c_int
        L.ref_decode_step.argtypes = [ctypes.POINTER(RefConfig), ctypes.POINTER(RefWeights),
                                      ctypes.POINTER(u16p), ctypes.POINTER(u16p),
                                      ctypes.c_int, ctypes.c_int, i32p, i32p, f64p, ctypes.c_int]
        L.ref_forward_full.restype = ctypes.c_int
        L.ref_forward_full.argtypes = [ctypes.POINTER(RefConfig), ctypes.POINTER(RefWeights),
                                       ctypes.c_int, i32p, f64p,
                                       ctypes.POINTER(u16p), ctypes.POINTER(u16p), ctypes.c_int]
        _lib = L
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ---------------------------------------------------------------- helpers

def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bits as uint16, got {a.dtype}")
    return a


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p16(a: np.ndarray):
    return a.ctypes.data_as(u16p)


def _p64(a: np.ndarray):
    return a.ctypes.data_as(f64p)


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(v) -> np.ndarray:
    L = lib()
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    flat_v, flat_o = v.reshape(-1), out.reshape(-1)
    for i in range(flat_v.size):
        flat_o[i] = L.ref_f64_to_bf16(float(flat_v[i]))
    return out


def rmsnorm(x, w_bits, eps: float) -> np.ndarray:
    x = _f64(x)
    w = _u16(w_bits)
    out = np.empty_like(x)
    lib().ref_rmsnorm(_p64(x), _p16(w), x.size, eps, _p64(out))
    return out


def rope(v, pos: int, theta: float) -> np.ndarray:
    v = _f64(v).copy()
    lib().ref_rope(_p64(v), v.size, int(pos), float(theta))
    return v


def silu(z: float) -> float:
    return lib().ref_silu(float(z))


def matvec(W_bits, x, nthreads: int = 1) -> np.ndarray:
    W = _u16(W_bits)
    x = _f64(x)
    rows, cols = W.shape
    y = np.empty(rows, dtype=np.float64)
    lib().ref_matvec(_p16(W), rows, cols, _p64(x), _p64(y), nthreads)
    return y


def attend(q, K_bits, V_bits, scale: float) -> np.ndarray:
    q = _f64(q)
    K = _u16(K_bits)
    V = _u16(V_bits)
    n, d = K.shape
    out = np.empty(d, dtype=np.float64)
    lib().ref_attend(_p64(q), _p16(K), _p16(V), n, d, d, float(scale), _p64(out))
    return out


# ---------------------------------------------------------------- model

class Model:
    """Holds a config dict and bf16 weights (numpy uint16) for the oracle.

    ``weights`` keys: embed, lm_head (None when tied), final_norm, and per-layer
    lists attn_norm, wq, wk, wv, wo, mlp_norm, wgate, wup, wdown.
    """

    def __init__(self, cfg: dict, weights: dict):
        self.cfg = dict(cfg)
        self.w = {k: (_u16(v) if isinstance(v, np.ndarray) else
                      ([_u16(x) for x in v] if isinstance(v, list) else v))
                  for k, v in weights.items()}
        c = self.cfg
        self._c = RefConfig(c["n_layers"], c["hidden"], c["n_heads"], c["n_kv_heads"],
                            c["head_dim"], c["ffn"], c["vocab"], int(bool(c["tied"])),
                            float(c["rms_eps"]), float(c["rope_theta"]))
        L = c["n_layers"]

        def arr(name):
            a = (u16p * L)()
            for i in range(L):
                a[i] = _p16(self.w[name][i])
            return a

        self._arrs = {n: arr(n) for n in ("attn_norm", "wq", "wk", "wv", "wo",
                                          "mlp_norm", "wgate", "wup", "wdown")}
        lm = self.w.get("lm_head")
        self._w = RefWeights(_p16(self.w["embed"]),
                             _p16(lm) if lm is not None else ctypes.cast(None, u16p),
                             _p16(self.w["final_norm"]),
                             *[self._arrs[n] for n in ("attn_norm", "wq", "wk", "wv", "wo",
                                                       "mlp_norm", "wgate", "wup", "wdown")])

    def decode_step(self, k_cache, v_cache, tokens, positions, nthreads: int | None = None):
        """One decode step; k_cache/v_cache: lists (per layer) of uint16 arrays
        [B][nkv][S][D], updated in place. Returns logits [B][V] float64."""
        c = self.cfg
        L = c["n_layers"]
        B = len(tokens)
        S = k_cache[0].shape[2]
        kp = (u16p * L)(*[_p16(_u16(k)) for k in k_cache])
        vp = (u16p * L)(*[_p16(_u16(v)) for v in v_cache])
        for k in list(k_cache) + list(v_cache):
            if not k.flags["C_CONTIGUOUS"] or k.dtype != np.uint16:
                raise TypeError("KV cache must be contiguous uint16")
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        pos = np.ascontiguousarray(positions, dtype=np.int32)
        out = np.empty((B, c["vocab"]), dtype=np.float64)
        rc = lib().ref_decode_step(ctypes.byref(self._c), ctypes.byref(self._w), kp, vp, B, S,
                                   tok.ctypes.data_as(i32p), pos.ctypes.data_as(i32p),
                                   _p64(out), nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle rejected the decode-step inputs")
        return out

    def forward_full(self, tokens, nthreads: int | None = None, want_kv: bool = False):
        """Full causal forward of one sequence at positions 0..n-1 (no cache).
        Returns logits [n][V] (and per-layer K, V [nkv][n][D] when want_kv)."""
        c = self.cfg
        L = c["n_layers"]
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        n = tok.size
        out = np.empty((n, c["vocab"]), dtype=np.float64)
        ks = [np.empty((c["n_kv_heads"], n, c["head_dim"]), np.uint16) for _ in range(L)]
        vs = [np.empty((c["n_kv_heads"], n, c["head_dim"]), np.uint16) for _ in range(L)]
        kp = (u16p * L)(*[_p16(k) for k in ks])
        vp = (u16p * L)(*[_p16(v) for v in vs])
        rc = lib().ref_forward_full(ctypes.byref(self._c), ctypes.byref(self._w), n,
                                    tok.ctypes.data_as(i32p), _p64(out), kp, vp,
                                    nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle rejected the forward inputs")
        return (out, ks, vs) if want_kv else out
