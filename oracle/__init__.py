"""fp64 CPU oracle of CCA prefill (global-aware pooling + fused core/local attention).

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this package; the CUDA library never does, and the two
share no code.  The arithmetic lives in ``cca_oracle.c`` (plain fp64 loops,
OpenMP over rows); this module only widens inputs to fp64 exactly and marshals
numpy arrays through ctypes.

Formulas followed ("Core Context Aware Transformers for Long Context Language
Modeling", Method section of the digest page):
  pooling:  c_i   = softmax(Q_{ig} K'_{I_i}^T / sqrt(d)) X^G_{I_i}
  fusion:   Att_i = softmax(Q_i [K^G_{T_i}; K^L_{U_i}]^T / sqrt(d)) [V^G_{T_i}; V^L_{U_i}]
with the visibility sets read as: core j visible to query i iff
(j+1)*g <= max(0, i-w+1); local window [max(0, i-w+1), i].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cca_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libcca_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle with gcc (-O2 -fopenmp, no -ffast-math)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int64)
    i = ctypes.c_int
    lib.cca_oracle_pool.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, ctypes.c_double]
    lib.cca_oracle_pool.restype = None
    lib.cca_oracle_attn.argtypes = [dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, i, i, ctypes.c_double]
    lib.cca_oracle_attn.restype = None
    lib.cca_oracle_attn_rows.argtypes = [dp, dp, dp, dp, dp, ip, ctypes.c_int64, dp, dp,
                                         i, i, i, i, i, i, i, ctypes.c_double]
    lib.cca_oracle_attn_rows.restype = None
    lib.cca_oracle_pool_mode.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, ctypes.c_double, i]
    lib.cca_oracle_pool_mode.restype = None
    lib.cca_oracle_attn_mode.argtypes = [dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, i, i, ctypes.c_double, i]
    lib.cca_oracle_attn_mode.restype = None
    lib.cca_oracle_attn_rows_mode.argtypes = [dp, dp, dp, dp, dp, ip, ctypes.c_int64, dp, dp,
                                              i, i, i, i, i, i, i, ctypes.c_double, i]
    lib.cca_oracle_attn_rows_mode.restype = None
    lib.cca_oracle_threads.argtypes = []
    lib.cca_oracle_threads.restype = ctypes.c_int
    lib.cca_oracle_set_threads.argtypes = [ctypes.c_int]
    lib.cca_oracle_set_threads.restype = None
    return lib


def widen(x) -> np.ndarray:
    """Exact fp64 copy of a torch tensor (bf16/f16/f32/f64) or numpy array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu")
            if x.dtype != torch.float64:
                x = x.to(torch.float32)  # exact for bf16/f16/f32
            x = x.to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def threads() -> int:
    return load().cca_oracle_threads()


def set_threads(n: int) -> None:
    load().cca_oracle_set_threads(int(n))


def _shapes(Q, K):
    B, Hq, N, d = Q.shape
    Bk, Hkv, Nk, dk = K.shape
    assert (B, N, d) == (Bk, Nk, dk) and Hq % Hkv == 0
    return B, Hq, Hkv, N, d


def pool(Q, K, V, g: int, scale: float | None = None, lib=None, pool_mode: int = 0):
    """Global-aware pooling -> (Kc, Vc), each [B, Hkv, N/g, d] fp64.
    pool_mode 0: softmax weights of the group-last query (the method); 1: mean; 2: max;
    3: each query head's own softmax weights, averaged over the heads sharing the KV head."""
    lib = lib or load()
    Q, K, V = widen(Q), widen(K), widen(V)
    B, Hq, Hkv, N, d = _shapes(Q, K)
    assert N % g == 0
    scale = float(d) ** -0.5 if scale is None else float(scale)
    Kc = np.zeros((B, Hkv, N // g, d))
    Vc = np.zeros((B, Hkv, N // g, d))
    lib.cca_oracle_pool_mode(_ptr(Q), _ptr(K), _ptr(V), _ptr(Kc), _ptr(Vc), B, Hq, Hkv, N, d, g, scale,
                             int(pool_mode))
    return Kc, Vc


def attn(Q, K, V, Kc, Vc, g: int, w: int, scale: float | None = None, lib=None, window_mode: int = 0):
    """Fused core/local attention -> (O [B,Hq,N,d], LSE [B,Hq,N]) in fp64.
    window_mode 1: raw window starts at the group boundary g*(lo(i)//g) (no gap)."""
    lib = lib or load()
    Q, K, V, Kc, Vc = (widen(t) for t in (Q, K, V, Kc, Vc))
    B, Hq, Hkv, N, d = _shapes(Q, K)
    assert Kc.shape == (B, Hkv, N // g, d) and Vc.shape == Kc.shape
    scale = float(d) ** -0.5 if scale is None else float(scale)
    O = np.zeros((B, Hq, N, d))
    LSE = np.zeros((B, Hq, N))
    lib.cca_oracle_attn_mode(_ptr(Q), _ptr(K), _ptr(V), _ptr(Kc), _ptr(Vc), _ptr(O), _ptr(LSE),
                             B, Hq, Hkv, N, d, g, w, scale, int(window_mode))
    return O, LSE


def attn_rows(Q, K, V, Kc, Vc, g: int, w: int, rows, scale: float | None = None, lib=None,
              window_mode: int = 0):
    """Fused attention for selected (b, h, i) rows -> (O [n, d], LSE [n])."""
    lib = lib or load()
    Q, K, V, Kc, Vc = (widen(t) for t in (Q, K, V, Kc, Vc))
    B, Hq, Hkv, N, d = _shapes(Q, K)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    scale = float(d) ** -0.5 if scale is None else float(scale)
    n = rows.shape[0]
    O = np.zeros((n, d))
    LSE = np.zeros((n,))
    lib.cca_oracle_attn_rows_mode(_ptr(Q), _ptr(K), _ptr(V), _ptr(Kc), _ptr(Vc),
                                  rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n,
                                  _ptr(O), _ptr(LSE), B, Hq, Hkv, N, d, g, w, scale, int(window_mode))
    return O, LSE


def prefill(Q, K, V, g: int, w: int, scale: float | None = None, lib=None, pool_mode: int = 0,
            window_mode: int = 0):
    """End-to-end: pooling in fp64 (core tokens are not rounded), then attention."""
    Kc, Vc = pool(Q, K, V, g, scale, lib=lib, pool_mode=pool_mode)
    O, LSE = attn(Q, K, V, Kc, Vc, g, w, scale, lib=lib, window_mode=window_mode)
    return O, LSE, Kc, Vc
