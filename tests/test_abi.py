"""Host-only checks of the C ABI: the library loads, exports every function
include/*.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from sparse_long_context_cca_gb300 import api
from sparse_long_context_cca_gb300 import build as cbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return api.load_library()


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(cca_\w+)\s*\(", src))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"cca_pool", "cca_attn_fwd", "cca_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(api.EXPORTED) == set(names)


def test_abi_version_and_strings(lib):
    assert lib.cca_abi_version() == 3
    for code in (0, -1, -2, -3, -4, 7):
        assert isinstance(api.status_string(code), str) and api.status_string(code)


# Fake, 16-byte aligned pointers: every call below must be rejected on the host
# before any CUDA call, so they are never dereferenced.
P = [0x1000 * (k + 1) for k in range(7)]


def call_pool(lib, **kw):
    base = dict(B=1, Hq=2, Hkv=2, N=256, d=128, g=16, w=32, dtype=api.CCA_BF16)
    base.update(kw)
    prm = api.make_params(**base)
    ptrs = kw.pop("_ptrs", P[:5]) if "_ptrs" in kw else P[:5]
    return lib.cca_pool(*ptrs, ctypes.byref(prm), None)


def call_attn(lib, ptrs=None, **kw):
    base = dict(B=1, Hq=2, Hkv=2, N=256, d=128, g=16, w=32, dtype=api.CCA_BF16)
    base.update(kw)
    prm = api.make_params(**base)
    ptrs = ptrs or P
    return lib.cca_attn_fwd(*ptrs, ctypes.byref(prm), None)


@pytest.mark.parametrize("kw", [dict(N=250), dict(g=0), dict(w=0), dict(B=0), dict(Hq=3, Hkv=2),
                                dict(Hkv=0), dict(N=0), dict(dtype=5), dict(scale=float("nan"))])
def test_attn_rejects_bad_shapes(lib, kw):
    assert call_attn(lib, **kw) == api.CCA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(N=250), dict(g=0), dict(Hq=3, Hkv=2), dict(dtype=9)])
def test_pool_rejects_bad_shapes(lib, kw):
    assert call_pool(lib, **kw) == api.CCA_ERR_INVALID_ARG


def test_rejects_null_and_misaligned(lib):
    for k in range(7):
        bad = list(P)
        bad[k] = 0
        assert call_attn(lib, ptrs=bad) == api.CCA_ERR_INVALID_ARG
        bad[k] = P[k] + 8
        assert call_attn(lib, ptrs=bad) == api.CCA_ERR_INVALID_ARG
    prm = api.make_params(1, 2, 2, 256, 128, 16, 32, api.CCA_BF16)
    assert lib.cca_pool(P[0], 0, P[2], P[3], P[4], ctypes.byref(prm), None) == api.CCA_ERR_INVALID_ARG
    assert lib.cca_pool(P[0], P[1] + 4, P[2], P[3], P[4], ctypes.byref(prm), None) == api.CCA_ERR_INVALID_ARG
    assert lib.cca_attn_fwd(*P, None, None) == api.CCA_ERR_INVALID_ARG


def test_unsupported_head_dims(lib):
    assert call_attn(lib, d=96) == api.CCA_ERR_UNSUPPORTED
    assert call_attn(lib, d=64, dtype=api.CCA_BF16) == api.CCA_ERR_UNSUPPORTED
    assert call_pool(lib, d=256) == api.CCA_ERR_UNSUPPORTED


def test_python_binding_requires_cuda_tensors(lib):
    import torch
    x = torch.zeros(1, 2, 16, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        api.cca_pool(x, x, x, 4)


def test_decode_rejects_bad_arguments(lib):
    prm = api.make_params(1, 4, 4, 1024, 128, 16, 256, api.CCA_BF16)
    need = lib.cca_decode_workspace_size(ctypes.byref(prm))
    assert need > 0
    args = P[:7]
    assert lib.cca_decode_fwd(*args, -1, ctypes.byref(prm), P[0], need, None) == api.CCA_ERR_INVALID_ARG
    assert lib.cca_decode_fwd(*args, 1024, ctypes.byref(prm), P[0], need, None) == api.CCA_ERR_INVALID_ARG
    assert lib.cca_decode_fwd(*args, 5, ctypes.byref(prm), P[0], need - 16, None) == api.CCA_ERR_INVALID_ARG
    assert lib.cca_decode_fwd(*args, 5, ctypes.byref(prm), 0, need, None) == api.CCA_ERR_INVALID_ARG
    prm3 = api.make_params(1, 6, 2, 1024, 128, 16, 256, api.CCA_BF16)   # 3 query heads per KV head
    assert lib.cca_decode_fwd(*args, 5, ctypes.byref(prm3), P[0], 1 << 30, None) == api.CCA_ERR_UNSUPPORTED
    bad = api.make_params(1, 4, 4, 1000, 128, 16, 256, api.CCA_BF16)    # N % g != 0
    assert lib.cca_decode_workspace_size(ctypes.byref(bad)) == 0


def test_pool_group_rejects_bad_group(lib):
    prm = api.make_params(1, 4, 4, 1024, 128, 16, 1, api.CCA_BF16)
    assert lib.cca_pool_group(*P[:5], -1, ctypes.byref(prm), None) == api.CCA_ERR_INVALID_ARG
    assert lib.cca_pool_group(*P[:5], 64, ctypes.byref(prm), None) == api.CCA_ERR_INVALID_ARG


def test_rejects_unknown_modes(lib):
    for kw in (dict(window_mode=2), dict(window_mode=-1), dict(pool_mode=4), dict(pool_mode=-1)):
        prm = api.make_params(1, 2, 2, 256, 128, 16, 32, api.CCA_BF16, **kw)
        assert lib.cca_attn_fwd(*P, ctypes.byref(prm), None) == api.CCA_ERR_INVALID_ARG
        assert lib.cca_pool(*P[:5], ctypes.byref(prm), None) == api.CCA_ERR_INVALID_ARG


def test_post_softmax_gqa_pooling_head_limit(lib):
    # pool_mode 3 keeps one running softmax state per query head of a KV head: at most 8
    prm = api.make_params(1, 16, 1, 256, 128, 16, 32, api.CCA_BF16, pool_mode=3)
    assert lib.cca_pool(*P[:5], ctypes.byref(prm), None) == api.CCA_ERR_UNSUPPORTED
    assert lib.cca_pool_group(*P[:5], 0, ctypes.byref(prm), None) == api.CCA_ERR_UNSUPPORTED


def test_backward_rejects_bad_arguments(lib):
    prm = api.make_params(1, 2, 2, 256, 128, 16, 32, api.CCA_BF16)
    need = lib.cca_prefill_bwd_workspace_size(ctypes.byref(prm))
    assert need > 0
    ptrs = [0x1000 * (k + 1) for k in range(11)]
    assert lib.cca_prefill_bwd(*ptrs, ctypes.byref(prm), 0xC000, need - 16, None) == api.CCA_ERR_INVALID_ARG
    bad = list(ptrs)
    bad[8] = 0
    assert lib.cca_prefill_bwd(*bad, ctypes.byref(prm), 0xC000, need, None) == api.CCA_ERR_INVALID_ARG
    prm_bad = api.make_params(1, 2, 2, 250, 128, 16, 32, api.CCA_BF16)
    assert lib.cca_prefill_bwd_workspace_size(ctypes.byref(prm_bad)) == 0


def test_prefill_host_rejects_bad_arguments(lib):
    prm = api.make_params(2, 4, 2, 256, 128, 16, 32, api.CCA_BF16)
    need = lib.cca_prefill_host_workspace_size(ctypes.byref(prm))
    ptrs = [0x1000 * (k + 1) for k in range(7)]
    ws = 0x10000
    # 4 (batch, KV head) pairs -> slices of one pair, three slice buffers of
    # Q, O (2 query heads each), K, V, LSE, Kc, Vc, each rounded up to 256 bytes
    up = lambda x: (x + 255) // 256 * 256
    q, kv, c, lse = 2 * 256 * 128 * 2, 256 * 128 * 2, 16 * 128 * 2, 2 * 256 * 4
    assert need == 3 * (2 * up(q) + 2 * up(kv) + up(lse) + 2 * up(c))
    assert lib.cca_prefill_host(*ptrs, ctypes.byref(prm), ws, need - 1, None) == api.CCA_ERR_INVALID_ARG
    for k in (0, 1, 2, 3):
        bad = list(ptrs)
        bad[k] = None
        assert lib.cca_prefill_host(*bad, ctypes.byref(prm), ws, need, None) == api.CCA_ERR_INVALID_ARG
    only_kc = list(ptrs)
    only_kc[6] = None
    assert lib.cca_prefill_host(*only_kc, ctypes.byref(prm), ws, need, None) == api.CCA_ERR_INVALID_ARG
    assert lib.cca_prefill_host(*ptrs, ctypes.byref(prm), None, need, None) == api.CCA_ERR_INVALID_ARG
    assert lib.cca_prefill_host(*ptrs, ctypes.byref(prm), ws + 8, need, None) == api.CCA_ERR_INVALID_ARG
    prm64 = api.make_params(2, 4, 2, 256, 64, 16, 32, api.CCA_BF16)
    need64 = lib.cca_prefill_host_workspace_size(ctypes.byref(prm64))
    assert lib.cca_prefill_host(*ptrs, ctypes.byref(prm64), ws, need64, None) == api.CCA_ERR_UNSUPPORTED
    bad_shape = api.make_params(2, 4, 2, 250, 128, 16, 32, api.CCA_BF16)
    assert lib.cca_prefill_host_workspace_size(ctypes.byref(bad_shape)) == 0
    # a large problem is cut into about eight slices and keeps three buffers
    big = api.make_params(1, 32, 32, 32768, 128, 16, 1024, api.CCA_BF16)
    per_pair = 2 * 32768 * 128 * 2 * 2 + 32768 * 4 + 2 * 2048 * 128 * 2
    assert lib.cca_prefill_host_workspace_size(ctypes.byref(big)) == 3 * 4 * per_pair


def test_prefill_host_binding_requires_cpu_tensors(lib):
    import torch
    Q = torch.zeros(1, 2, 32, 128, dtype=torch.bfloat16, device="meta")
    with pytest.raises(ValueError):
        api.cca_prefill_host(Q, Q, Q, 16, 8)


def call_rows(lib, q_off, n_q, kv_off, n_kv, **kw):
    base = dict(B=1, Hq=2, Hkv=2, N=1024, d=128, g=16, w=100, dtype=api.CCA_BF16)
    base.update(kw)
    prm = api.make_params(**base)
    return lib.cca_attn_fwd_rows(*P, q_off, n_q, kv_off, n_kv, ctypes.byref(prm), None)


@pytest.mark.parametrize("args", [
    (0, 0, 0, 10),          # no rows
    (-1, 10, 0, 10),        # negative offset
    (1000, 25, 901, 124),   # rows past N
    (500, 10, 402, 108),    # K/V start after row 500's window start (401)
    (500, 10, 401, 100),    # K/V end before the last row
    (500, 10, 401, 700),    # K/V past N
    (500, 10, -1, 600),     # negative K/V offset
])
def test_rows_rejects_bad_ranges(lib, args):
    assert call_rows(lib, *args) == api.CCA_ERR_INVALID_ARG


def test_rows_window_mode_moves_the_first_raw_token(lib):
    # with window_mode 1, row 500's window starts at the group boundary 400, so K/V from 401
    # leave a token out: rejected (with window_mode 0 the same range would be valid)
    assert call_rows(lib, 500, 10, 401, 109, window_mode=1) == api.CCA_ERR_INVALID_ARG


def test_decode_kernels_rejects_bad_arguments(lib):
    prm = api.make_params(1, 2, 2, 256, 128, 16, 32, api.CCA_BF16)
    assert lib.cca_decode_kernels(ctypes.byref(prm), 256) == api.CCA_ERR_INVALID_ARG
    assert lib.cca_decode_kernels(ctypes.byref(prm), -1) == api.CCA_ERR_INVALID_ARG
    bad = api.make_params(1, 2, 2, 250, 128, 16, 32, api.CCA_BF16)
    assert lib.cca_decode_kernels(ctypes.byref(bad), 5) == api.CCA_ERR_INVALID_ARG


def test_plain_c_caller(lib, tmp_path):
    """The boundary is a C ABI: a C program built against include/cca.h and linked with
    libcca.so makes host-only calls (version, strings, sizes, rejected arguments)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "c_abi_host_only"
    libdir = os.path.dirname(api.library_path())
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c_abi_host_only.c"), "-L", libdir, "-lcca",
                        "-Wl,-rpath," + libdir, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout
