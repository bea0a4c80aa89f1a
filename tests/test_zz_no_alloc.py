"""The decode entry point that allocates nothing (cca_decode_fwd_noalloc).

It serves callers that cannot obtain device memory for this library, e.g. a
plug-in whose host framework owns every allocation, or a decode loop with a
fixed memory budget.  It must give the same results as cca_decode_fwd with a
caller workspace; its scratch is one fixed array shared by all calls, so two
calls in a row must not see each other's leftovers.  This file runs last so
that a failure here leaves every other test already run.
"""
import ctypes

import pytest
import torch

import oracle
from parity import check_out
from sparse_long_context_cca_gb300 import api
from sparse_long_context_cca_gb300.inputs import make_qkv
from sparse_long_context_cca_gb300.workloads import Workload

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, K, V, Kc, Vc, pos, g, w):
    B, Hq, d = q.shape
    Hkv, Ncap = K.shape[1], K.shape[2]
    dtype = api.CCA_BF16 if q.dtype == torch.bfloat16 else api.CCA_F32
    prm = api.make_params(B, Hq, Hkv, Ncap, d, g, w, dtype)
    O = torch.empty_like(q)
    LSE = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    st = lib.cca_decode_fwd_noalloc(q.data_ptr(), K.data_ptr(), V.data_ptr(), Kc.data_ptr(), Vc.data_ptr(),
                                    O.data_ptr(), LSE.data_ptr(), int(pos), ctypes.byref(prm),
                                    torch.cuda.current_stream().cuda_stream)
    assert st == api.CCA_OK, api.status_string(st)
    return O, LSE


CASES = [
    (Workload("noalloc bf16 B2 Hq8 Hkv2 N4096 g16 w512", 2, 8, 2, 4096, 128, 16, 512, "bf16", 21, 0.01), (4095, 1300)),
    (Workload("noalloc f32 B1 Hq4 Hkv4 N1024 g8 w200", 1, 4, 4, 1024, 64, 8, 200, "f32", 22, 0.02), (1023, 50)),
]


def test_noalloc_decode_matches_workspace_entry_point():
    """Both entry points launch the same kernels with the same split count, so their
    results must agree bit for bit; the first case is also checked against the oracle."""
    lib = api.load_library()
    # Two calls in a row per case, and the cases back to back, all through the same scratch.
    for n, (wl, positions) in enumerate(CASES):
        Q, K, V = make_qkv(wl, "cuda")
        Kc, Vc = api.cca_pool(Q, K, V, wl.g)
        for pos in positions:
            q = Q[:, :, pos].contiguous()
            O_ref, L_ref = api.cca_decode_fwd(q, K, V, Kc, Vc, pos, wl.g, wl.w)
            O, L = _noalloc(lib, q, K, V, Kc, Vc, pos, wl.g, wl.w)
            torch.cuda.synchronize()
            assert torch.equal(O, O_ref) and torch.equal(L, L_ref), f"{wl.name} pos {pos}"
            if n == 0:
                rows = [(b, h, pos) for b in range(wl.B) for h in range(wl.Hq)]
                Oe, Le = oracle.attn_rows(Q, K, V, Kc, Vc, wl.g, wl.w, rows)
                check_out(O.reshape(-1, wl.d), L.reshape(-1), Oe, Le, q.dtype, f"{wl.name} pos {pos} vs oracle")


def test_noalloc_decode_at_the_scratch_limit():
    """B * Hq = 126 query rows at d = 128 with 64 splits per row fill the 4 MiB array up
    to its last partial (126 * 64 * 130 * 4 bytes); two calls in a row must match the
    workspace entry point bit for bit."""
    lib = api.load_library()
    wl = Workload("noalloc bf16 B1 Hq126 Hkv63 N16384 g16 w16384", 1, 126, 63, 16384, 128, 16, 16384, "bf16", 23,
                  0.01)
    prm = api.make_params(wl.B, wl.Hq, wl.Hkv, wl.N, wl.d, wl.g, wl.w, api.CCA_BF16)
    need = lib.cca_decode_workspace_size(ctypes.byref(prm))
    assert need == 126 * 64 * 130 * 4 and need <= (4 << 20) < need + 64 * 130 * 4
    Q, K, V = make_qkv(wl, "cuda")
    Kc, Vc = api.cca_pool(Q, K, V, wl.g)
    for pos in (wl.N - 1, wl.N - 2):  # 16384 and 16383 visible keys: 64 splits of at least 256
        q = Q[:, :, pos].contiguous()
        O_ref, L_ref = api.cca_decode_fwd(q, K, V, Kc, Vc, pos, wl.g, wl.w)
        O, L = _noalloc(lib, q, K, V, Kc, Vc, pos, wl.g, wl.w)
        torch.cuda.synchronize()
        assert torch.equal(O, O_ref) and torch.equal(L, L_ref), f"pos {pos}"
    del Q, K, V, Kc, Vc
    torch.cuda.empty_cache()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = api.load_library()
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    p = t.data_ptr()
    # 64 x 64 query heads need 64*64*64*130*4 bytes of partials, far above the fixed 4 MiB
    prm = api.make_params(64, 64, 64, 1024, 128, 16, 256, api.CCA_BF16)
    assert lib.cca_decode_workspace_size(ctypes.byref(prm)) > (4 << 20)
    st = lib.cca_decode_fwd_noalloc(p, p, p, p, p, p, p, 5, ctypes.byref(prm), None)
    assert st == api.CCA_ERR_SCRATCH_LIMIT
    assert "scratch" in api.status_string(st)
    # one query row past the limit at d = 128 (127 rows), and at d = 64 (249 rows)
    for B, Hq, d in ((1, 127, 128), (1, 249, 64)):
        prm = api.make_params(B, Hq, Hq, 1024, d, 16, 256, api.CCA_BF16)
        assert lib.cca_decode_fwd_noalloc(p, p, p, p, p, p, p, 5, ctypes.byref(prm), None) == api.CCA_ERR_SCRATCH_LIMIT
    for B, Hq, d in ((1, 126, 128), (2, 124, 64)):  # the largest shapes that fit are accepted
        prm = api.make_params(B, Hq, Hq, 1024, d, 16, 256, api.CCA_BF16)
        assert lib.cca_decode_workspace_size(ctypes.byref(prm)) <= (4 << 20)
