"""Thin Python binding of libcca.so (include/cca.h), argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
allocates outputs with torch (device memory is plumbing), checks that tensors
match the C ABI's layout, and forwards raw device pointers.  There is no
fallback: if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

CCA_OK = 0
CCA_ERR_INVALID_ARG = -1
CCA_ERR_UNSUPPORTED = -2
CCA_ERR_CUDA = -3
CCA_ERR_TIMEOUT = -4
CCA_ERR_SCRATCH_LIMIT = -5
CCA_BF16 = 0
CCA_F32 = 1

_DTYPE = {torch.bfloat16: CCA_BF16, torch.float32: CCA_F32}


class CcaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


class CcaParams(ctypes.Structure):
    """Mirror of cca_params_t."""
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("N", ctypes.c_int32), ("d", ctypes.c_int32), ("g", ctypes.c_int32),
                ("w", ctypes.c_int32), ("dtype", ctypes.c_int32), ("scale", ctypes.c_float),
                ("dev_status", ctypes.c_void_p), ("window_mode", ctypes.c_int32),
                ("pool_mode", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()

EXPORTED = ["cca_pool", "cca_attn_fwd", "cca_attn_fwd_rows", "cca_decode_fwd", "cca_decode_workspace_size",
            "cca_decode_kernels", "cca_pool_group",
            "cca_decode_fwd_noalloc", "cca_prefill_bwd", "cca_prefill_bwd_workspace_size",
            "cca_prefill_host", "cca_prefill_host_workspace_size",
            "cca_status_string", "cca_abi_version", "cca_test_set_wait_limit_ns", "cca_test_skip_q_load",
            "cca_test_decode_path"]


def library_path() -> str:
    return os.environ.get("CCA_LIBRARY", _build.LIB)


def load_library():
    """Load libcca.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libcca.so not found at {path}: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        vp = ctypes.c_void_p
        pp = ctypes.POINTER(CcaParams)
        lib.cca_pool.argtypes = [vp, vp, vp, vp, vp, pp, vp]
        lib.cca_pool.restype = ctypes.c_int
        lib.cca_attn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, pp, vp]
        lib.cca_attn_fwd.restype = ctypes.c_int
        ci = ctypes.c_int
        lib.cca_attn_fwd_rows.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, pp, vp]
        lib.cca_attn_fwd_rows.restype = ctypes.c_int
        lib.cca_decode_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, pp, vp, ctypes.c_uint64, vp]
        lib.cca_decode_fwd.restype = ctypes.c_int
        lib.cca_decode_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, pp, vp]
        lib.cca_decode_fwd_noalloc.restype = ctypes.c_int
        lib.cca_prefill_bwd.argtypes = [vp] * 11 + [pp, vp, ctypes.c_uint64, vp]
        lib.cca_prefill_bwd.restype = ctypes.c_int
        lib.cca_prefill_bwd_workspace_size.argtypes = [pp]
        lib.cca_prefill_bwd_workspace_size.restype = ctypes.c_uint64
        lib.cca_prefill_host.argtypes = [vp] * 7 + [pp, vp, ctypes.c_uint64, vp]
        lib.cca_prefill_host.restype = ctypes.c_int
        lib.cca_prefill_host_workspace_size.argtypes = [pp]
        lib.cca_prefill_host_workspace_size.restype = ctypes.c_uint64
        lib.cca_decode_kernels.argtypes = [pp, ctypes.c_int]
        lib.cca_decode_kernels.restype = ctypes.c_int
        lib.cca_decode_workspace_size.argtypes = [pp]
        lib.cca_decode_workspace_size.restype = ctypes.c_uint64
        lib.cca_pool_group.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, pp, vp]
        lib.cca_pool_group.restype = ctypes.c_int
        lib.cca_status_string.argtypes = [ctypes.c_int]
        lib.cca_status_string.restype = ctypes.c_char_p
        lib.cca_abi_version.argtypes = []
        lib.cca_abi_version.restype = ctypes.c_int
        lib.cca_test_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        lib.cca_test_set_wait_limit_ns.restype = None
        lib.cca_test_skip_q_load.argtypes = [ctypes.c_int]
        lib.cca_test_skip_q_load.restype = None
        lib.cca_test_decode_path.argtypes = [ctypes.c_int]
        lib.cca_test_decode_path.restype = None
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().cca_status_string(int(status)).decode()


def make_params(B, Hq, Hkv, N, d, g, w, dtype, scale=0.0, dev_status=None, window_mode=0,
                pool_mode=0) -> CcaParams:
    return CcaParams(int(B), int(Hq), int(Hkv), int(N), int(d), int(g), int(w), int(dtype),
                     float(scale), dev_status, int(window_mode), int(pool_mode))


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(t: torch.Tensor, name: str, dtype, shape):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dims(Q, K):
    if Q.dim() != 4 or K.dim() != 4:
        raise ValueError("Q and K must be [B, H, N, d]")
    B, Hq, N, d = Q.shape
    Hkv = K.shape[1]
    return B, Hq, Hkv, N, d


def cca_pool(Q, K, V, g: int, Kc=None, Vc=None, scale: float = 0.0, stream=None, pool_mode: int = 0):
    """Global-aware pooling: returns (Kc, Vc), each [B, Hkv, N/g, d].
    pool_mode 0: softmax weights of the group-last query (GQA: the r heads' logits averaged);
    1: mean; 2: element-wise max; 3: GQA pooling averaged after the softmax (each query head's
    own softmax weights, averaged over the r heads sharing the KV head; r <= 8)."""
    lib = load_library()
    B, Hq, Hkv, N, d = _dims(Q, K)
    if Q.dtype not in _DTYPE:
        raise ValueError(f"unsupported dtype {Q.dtype}")
    _check(Q, "Q", Q.dtype, (B, Hq, N, d))
    _check(K, "K", Q.dtype, (B, Hkv, N, d))
    _check(V, "V", Q.dtype, (B, Hkv, N, d))
    G = N // g if g > 0 else 0
    if Kc is None:
        Kc = torch.empty((B, Hkv, G, d), dtype=Q.dtype, device=Q.device)
    if Vc is None:
        Vc = torch.empty((B, Hkv, G, d), dtype=Q.dtype, device=Q.device)
    _check(Kc, "Kc", Q.dtype, (B, Hkv, G, d))
    _check(Vc, "Vc", Q.dtype, (B, Hkv, G, d))
    prm = make_params(B, Hq, Hkv, N, d, g, 1, _DTYPE[Q.dtype], scale, pool_mode=pool_mode)
    st = lib.cca_pool(Q.data_ptr(), K.data_ptr(), V.data_ptr(), Kc.data_ptr(), Vc.data_ptr(),
                      ctypes.byref(prm), _stream_handle(stream))
    if st != CCA_OK:
        raise CcaError(st, "cca_pool")
    return Kc, Vc


def cca_attn_fwd(Q, K, V, Kc, Vc, g: int, w: int, O=None, LSE=None, scale: float = 0.0,
                 dev_status=None, stream=None, window_mode: int = 0):
    """Fused core/local attention: returns (O [B,Hq,N,d], LSE [B,Hq,N] fp32).
    window_mode 1: the raw window starts at the group boundary g*(lo(i)//g)."""
    lib = load_library()
    B, Hq, Hkv, N, d = _dims(Q, K)
    if Q.dtype not in _DTYPE:
        raise ValueError(f"unsupported dtype {Q.dtype}")
    G = N // g if g > 0 else 0
    _check(Q, "Q", Q.dtype, (B, Hq, N, d))
    _check(K, "K", Q.dtype, (B, Hkv, N, d))
    _check(V, "V", Q.dtype, (B, Hkv, N, d))
    _check(Kc, "Kc", Q.dtype, (B, Hkv, G, d))
    _check(Vc, "Vc", Q.dtype, (B, Hkv, G, d))
    if O is None:
        O = torch.empty_like(Q)
    if LSE is None:
        LSE = torch.empty((B, Hq, N), dtype=torch.float32, device=Q.device)
    _check(O, "O", Q.dtype, (B, Hq, N, d))
    _check(LSE, "LSE", torch.float32, (B, Hq, N))
    status_ptr = None
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, (1,))
        status_ptr = dev_status.data_ptr()
    prm = make_params(B, Hq, Hkv, N, d, g, w, _DTYPE[Q.dtype], scale, status_ptr, window_mode=window_mode)
    st = lib.cca_attn_fwd(Q.data_ptr(), K.data_ptr(), V.data_ptr(), Kc.data_ptr(), Vc.data_ptr(),
                          O.data_ptr(), LSE.data_ptr(), ctypes.byref(prm), _stream_handle(stream))
    if st != CCA_OK:
        raise CcaError(st, "cca_attn_fwd")
    return O, LSE


def cca_attn_fwd_rows(Q, K, V, Kc, Vc, g: int, w: int, N: int, q_off: int, kv_off: int, O=None, LSE=None,
                      scale: float = 0.0, dev_status=None, stream=None, window_mode: int = 0):
    """Fused attention for the query rows [q_off, q_off + n_q) of an N-token sequence.
    Q [B,Hq,n_q,d] holds those rows, K, V [B,Hkv,n_kv,d] the raw tokens from kv_off on,
    Kc, Vc [B,Hkv,N/g,d] the whole sequence's core tokens.  Returns (O [B,Hq,n_q,d],
    LSE [B,Hq,n_q] fp32), equal to rows q_off .. q_off + n_q - 1 of cca_attn_fwd over N."""
    lib = load_library()
    B, Hq, n_q, d = Q.shape
    Hkv, n_kv = K.shape[1], K.shape[2]
    if Q.dtype not in _DTYPE:
        raise ValueError(f"unsupported dtype {Q.dtype}")
    G = N // g if g > 0 else 0
    _check(Q, "Q", Q.dtype, (B, Hq, n_q, d))
    _check(K, "K", Q.dtype, (B, Hkv, n_kv, d))
    _check(V, "V", Q.dtype, (B, Hkv, n_kv, d))
    _check(Kc, "Kc", Q.dtype, (B, Hkv, G, d))
    _check(Vc, "Vc", Q.dtype, (B, Hkv, G, d))
    if O is None:
        O = torch.empty_like(Q)
    if LSE is None:
        LSE = torch.empty((B, Hq, n_q), dtype=torch.float32, device=Q.device)
    _check(O, "O", Q.dtype, (B, Hq, n_q, d))
    _check(LSE, "LSE", torch.float32, (B, Hq, n_q))
    status_ptr = None
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, (1,))
        status_ptr = dev_status.data_ptr()
    prm = make_params(B, Hq, Hkv, N, d, g, w, _DTYPE[Q.dtype], scale, status_ptr, window_mode=window_mode)
    st = lib.cca_attn_fwd_rows(Q.data_ptr(), K.data_ptr(), V.data_ptr(), Kc.data_ptr(), Vc.data_ptr(),
                               O.data_ptr(), LSE.data_ptr(), int(q_off), int(n_q), int(kv_off), int(n_kv),
                               ctypes.byref(prm), _stream_handle(stream))
    if st != CCA_OK:
        raise CcaError(st, "cca_attn_fwd_rows")
    return O, LSE


def cca_prefill(Q, K, V, g: int, w: int, scale: float = 0.0, out=None, stream=None, pool_mode: int = 0,
                window_mode: int = 0):
    """Both steps of CCA prefill: pooling, then fused attention.
    Returns (O, LSE, Kc, Vc).  `out` may hold preallocated (O, LSE, Kc, Vc)."""
    O = LSE = Kc = Vc = None
    if out is not None:
        O, LSE, Kc, Vc = out
    Kc, Vc = cca_pool(Q, K, V, g, Kc, Vc, scale, stream, pool_mode=pool_mode)
    O, LSE = cca_attn_fwd(Q, K, V, Kc, Vc, g, w, O, LSE, scale, None, stream, window_mode=window_mode)
    return O, LSE, Kc, Vc


def causal_attention(Q, K, V, scale: float = 0.0, O=None, LSE=None, stream=None):
    """Full causal softmax attention through the same fused kernel: with g = 1 every
    token is its own core and with w >= N no core is visible, so the visible set of
    query i is exactly tokens [0, i] (the closed form the oracle is pinned to).
    K and V serve as their own core tensors (shape [B, Hkv, N/1, d])."""
    N = Q.shape[2]
    return cca_attn_fwd(Q, K, V, K, V, 1, N, O, LSE, scale, None, stream)


def decode_workspace_size(B, Hq, Hkv, Ncap, d, g, w, dtype) -> int:
    prm = make_params(B, Hq, Hkv, Ncap, d, g, w, _DTYPE[dtype])
    return int(load_library().cca_decode_workspace_size(ctypes.byref(prm)))


def decode_kernels(B, Hq, Hkv, Ncap, d, g, w, dtype, pos: int, window_mode: int = 0) -> int:
    """Kernels one cca_decode_fwd call at `pos` launches on the current device (1 or 2)."""
    prm = make_params(B, Hq, Hkv, Ncap, d, g, w, _DTYPE[dtype], window_mode=window_mode)
    n = int(load_library().cca_decode_kernels(ctypes.byref(prm), int(pos)))
    if n < 0:
        raise CcaError(n, "cca_decode_kernels")
    return n


def cca_decode_fwd(q, K, V, Kc, Vc, pos: int, g: int, w: int, O=None, LSE=None, workspace=None,
                   scale: float = 0.0, stream=None, window_mode: int = 0):
    """One decoding step: row `pos` of the fused attention over the caches.
    q [B, Hq, d]; K, V [B, Hkv, Ncap, d]; Kc, Vc [B, Hkv, Ncap/g, d].
    Returns (O [B, Hq, d], LSE [B, Hq])."""
    lib = load_library()
    if q.dim() != 3 or K.dim() != 4:
        raise ValueError("q must be [B, Hq, d] and K [B, Hkv, Ncap, d]")
    B, Hq, d = q.shape
    Hkv, Ncap = K.shape[1], K.shape[2]
    if q.dtype not in _DTYPE:
        raise ValueError(f"unsupported dtype {q.dtype}")
    G = Ncap // g if g > 0 else 0
    _check(q, "q", q.dtype, (B, Hq, d))
    _check(K, "K", q.dtype, (B, Hkv, Ncap, d))
    _check(V, "V", q.dtype, (B, Hkv, Ncap, d))
    _check(Kc, "Kc", q.dtype, (B, Hkv, G, d))
    _check(Vc, "Vc", q.dtype, (B, Hkv, G, d))
    if O is None:
        O = torch.empty_like(q)
    if LSE is None:
        LSE = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _check(O, "O", q.dtype, (B, Hq, d))
    _check(LSE, "LSE", torch.float32, (B, Hq))
    prm = make_params(B, Hq, Hkv, Ncap, d, g, w, _DTYPE[q.dtype], scale, window_mode=window_mode)
    need = int(lib.cca_decode_workspace_size(ctypes.byref(prm)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must be a CUDA buffer of at least {need} bytes")
    st = lib.cca_decode_fwd(q.data_ptr(), K.data_ptr(), V.data_ptr(), Kc.data_ptr(), Vc.data_ptr(),
                            O.data_ptr(), LSE.data_ptr(), int(pos), ctypes.byref(prm), workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if st != CCA_OK:
        raise CcaError(st, "cca_decode_fwd")
    return O, LSE


def cca_pool_group(q, K, V, Kc, Vc, j: int, g: int, scale: float = 0.0, stream=None, pool_mode: int = 0):
    """Pool the newly completed group j of the caches in place (Kc[:, :, j], Vc[:, :, j]),
    scored by q [B, Hq, d], the query of the group's last token."""
    lib = load_library()
    B, Hq, d = q.shape
    Hkv, Ncap = K.shape[1], K.shape[2]
    G = Ncap // g if g > 0 else 0
    _check(q, "q", q.dtype, (B, Hq, d))
    _check(K, "K", q.dtype, (B, Hkv, Ncap, d))
    _check(V, "V", q.dtype, (B, Hkv, Ncap, d))
    _check(Kc, "Kc", q.dtype, (B, Hkv, G, d))
    _check(Vc, "Vc", q.dtype, (B, Hkv, G, d))
    prm = make_params(B, Hq, Hkv, Ncap, d, g, 1, _DTYPE[q.dtype], scale, pool_mode=pool_mode)
    st = lib.cca_pool_group(q.data_ptr(), K.data_ptr(), V.data_ptr(), Kc.data_ptr(), Vc.data_ptr(), int(j),
                            ctypes.byref(prm), _stream_handle(stream))
    if st != CCA_OK:
        raise CcaError(st, "cca_pool_group")
    return Kc, Vc


def cca_prefill_bwd(Q, K, V, Kc, Vc, O, LSE, dO, g: int, w: int, scale: float = 0.0, pool_mode: int = 0,
                    window_mode: int = 0, dQ=None, dK=None, dV=None, workspace=None, stream=None,
                    dev_status=None):
    """Gradients (dQ, dK, dV), fp32, of sum(dO * O) for CCA prefill (pooling + attention).
    dev_status: optional int32 CUDA tensor of one element that receives CCA_ERR_TIMEOUT
    if a tensor-core kernel gives up waiting."""
    lib = load_library()
    B, Hq, Hkv, N, d = _dims(Q, K)
    G = N // g if g > 0 else 0
    for name, t, shape in (("Q", Q, (B, Hq, N, d)), ("K", K, (B, Hkv, N, d)), ("V", V, (B, Hkv, N, d)),
                           ("Kc", Kc, (B, Hkv, G, d)), ("Vc", Vc, (B, Hkv, G, d)), ("O", O, (B, Hq, N, d)),
                           ("dO", dO, (B, Hq, N, d))):
        _check(t, name, Q.dtype, shape)
    _check(LSE, "LSE", torch.float32, (B, Hq, N))
    dQ = torch.empty((B, Hq, N, d), dtype=torch.float32, device=Q.device) if dQ is None else dQ
    dK = torch.empty((B, Hkv, N, d), dtype=torch.float32, device=Q.device) if dK is None else dK
    dV = torch.empty((B, Hkv, N, d), dtype=torch.float32, device=Q.device) if dV is None else dV
    _check(dQ, "dQ", torch.float32, (B, Hq, N, d))
    _check(dK, "dK", torch.float32, (B, Hkv, N, d))
    _check(dV, "dV", torch.float32, (B, Hkv, N, d))
    status_ptr = None
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, (1,))
        status_ptr = dev_status.data_ptr()
    prm = make_params(B, Hq, Hkv, N, d, g, w, _DTYPE[Q.dtype], scale, status_ptr, window_mode=window_mode,
                      pool_mode=pool_mode)
    need = int(lib.cca_prefill_bwd_workspace_size(ctypes.byref(prm)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=Q.device)
    nbytes = workspace.numel() * workspace.element_size()
    st = lib.cca_prefill_bwd(Q.data_ptr(), K.data_ptr(), V.data_ptr(), Kc.data_ptr(), Vc.data_ptr(), O.data_ptr(),
                             LSE.data_ptr(), dO.data_ptr(), dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(),
                             ctypes.byref(prm), workspace.data_ptr(), nbytes, _stream_handle(stream))
    if st != CCA_OK:
        raise CcaError(st, "cca_prefill_bwd")
    return dQ, dK, dV


def _check_host(t: torch.Tensor, name: str, dtype, shape):
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError(f"{name} must be a CPU tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def prefill_host_workspace_size(B, Hq, Hkv, N, d, g, w, dtype) -> int:
    prm = make_params(B, Hq, Hkv, N, d, g, w, _DTYPE[dtype])
    return int(load_library().cca_prefill_host_workspace_size(ctypes.byref(prm)))


def cca_prefill_host(Q, K, V, g: int, w: int, scale: float = 0.0, out=None, with_lse: bool = True,
                     with_cores: bool = False, workspace=None, device=None, stream=None, pool_mode: int = 0,
                     window_mode: int = 0):
    """The prefill step on HOST tensors (pinned for overlap): the library copies Q, K, V in,
    pools, attends and copies the outputs back, pipelined over slices of KV heads.
    Returns (O, LSE or None, Kc or None, Vc or None) as CPU tensors; `out` may hold them
    preallocated.  The outputs are valid once `stream` has been synchronised."""
    lib = load_library()
    B, Hq, Hkv, N, d = _dims(Q, K)
    if Q.dtype not in _DTYPE:
        raise ValueError(f"unsupported dtype {Q.dtype}")
    G = N // g if g > 0 else 0
    _check_host(Q, "Q", Q.dtype, (B, Hq, N, d))
    _check_host(K, "K", Q.dtype, (B, Hkv, N, d))
    _check_host(V, "V", Q.dtype, (B, Hkv, N, d))
    pin = Q.is_pinned()
    if out is None:
        O = torch.empty((B, Hq, N, d), dtype=Q.dtype, pin_memory=pin)
        LSE = torch.empty((B, Hq, N), dtype=torch.float32, pin_memory=pin) if with_lse else None
        Kc = torch.empty((B, Hkv, G, d), dtype=Q.dtype, pin_memory=pin) if with_cores else None
        Vc = torch.empty((B, Hkv, G, d), dtype=Q.dtype, pin_memory=pin) if with_cores else None
    else:
        O, LSE, Kc, Vc = out
    _check_host(O, "O", Q.dtype, (B, Hq, N, d))
    if LSE is not None:
        _check_host(LSE, "LSE", torch.float32, (B, Hq, N))
    if (Kc is None) != (Vc is None):
        raise ValueError("Kc and Vc must be given together")
    if Kc is not None:
        _check_host(Kc, "Kc", Q.dtype, (B, Hkv, G, d))
        _check_host(Vc, "Vc", Q.dtype, (B, Hkv, G, d))
    prm = make_params(B, Hq, Hkv, N, d, g, w, _DTYPE[Q.dtype], scale, window_mode=window_mode,
                      pool_mode=pool_mode)
    need = int(lib.cca_prefill_host_workspace_size(ctypes.byref(prm)))
    if workspace is None:
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must be a CUDA buffer of at least {need} bytes")
    ptr = (lambda t: None if t is None else t.data_ptr())
    with torch.cuda.device(workspace.device):
        st = lib.cca_prefill_host(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), ptr(LSE), ptr(Kc),
                                  ptr(Vc), ctypes.byref(prm), workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if st != CCA_OK:
        raise CcaError(st, "cca_prefill_host")
    return O, LSE, Kc, Vc


class CcaAttentionFunction(torch.autograd.Function):
    """Autograd wrapper of the prefill step: forward = cca_prefill (pooling + fused
    attention), backward = cca_prefill_bwd.  Both run in the library's kernels; this
    class only saves tensors and casts the fp32 gradients to the inputs' dtype."""

    @staticmethod
    def forward(ctx, Q, K, V, g, w, scale, pool_mode, window_mode):
        Q, K, V = Q.contiguous(), K.contiguous(), V.contiguous()
        O, LSE, Kc, Vc = cca_prefill(Q, K, V, g, w, scale, pool_mode=pool_mode, window_mode=window_mode)
        ctx.save_for_backward(Q, K, V, Kc, Vc, O, LSE)
        ctx.cfg = (g, w, scale, pool_mode, window_mode)
        return O

    @staticmethod
    def backward(ctx, dO):
        Q, K, V, Kc, Vc, O, LSE = ctx.saved_tensors
        g, w, scale, pool_mode, window_mode = ctx.cfg
        dQ, dK, dV = cca_prefill_bwd(Q, K, V, Kc, Vc, O, LSE, dO.contiguous().to(Q.dtype), g, w, scale,
                                     pool_mode=pool_mode, window_mode=window_mode)
        return dQ.to(Q.dtype), dK.to(K.dtype), dV.to(V.dtype), None, None, None, None, None


def cca_attention(Q, K, V, g: int, w: int, scale: float = 0.0, pool_mode: int = 0, window_mode: int = 0):
    """CCA attention output O [B, Hq, N, d] with gradients for Q, K and V (prefill step)."""
    return CcaAttentionFunction.apply(Q, K, V, g, w, scale, pool_mode, window_mode)
