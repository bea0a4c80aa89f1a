"""Seeded random shapes through the CUDA path against the fp64 oracle: batch,
head counts and GQA ratio, ragged N (any multiple of g), group sizes from 1 to
64, windows from 1 token to beyond N, both window modes and all pooling modes,
bf16 (d = 128) and fp32 (d = 64, 128).  Every case runs the prefill (pooling +
attention); every third case also runs the backward and a decode step."""
import numpy as np
import pytest
import torch

import oracle
from oracle.backward import prefill_grads
from parity import check_cores, check_out
from sparse_long_context_cca_gb300 import api
from sparse_long_context_cca_gb300.inputs import make_qkv
from sparse_long_context_cca_gb300.workloads import Workload

pytestmark = pytest.mark.gpu


def random_cases(n=24, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for k in range(n):
        dtype = "bf16" if k % 3 else "f32"
        d = 128 if dtype == "bf16" else int(rng.choice([64, 128]))
        B = int(rng.integers(1, 3))
        Hkv = int(rng.choice([1, 2, 3]))
        r = int(rng.choice([1, 2, 4]))
        g = int(rng.choice([1, 2, 3, 5, 8, 16, 24, 64]))
        G = int(rng.integers(1, max(2, 700 // g)))
        N = g * G
        w = int(rng.choice([1, 2, int(rng.integers(1, N + 1)), N, N + 50, 1024]))
        pool_mode = int(rng.choice([0, 0, 1, 2]))
        window_mode = int(rng.integers(0, 2))
        wl = Workload(f"rand{k} B{B} Hq{Hkv * r} Hkv{Hkv} N{N} d{d} g{g} w{w} {dtype} p{pool_mode} m{window_mode}",
                      B, Hkv * r, Hkv, N, d, g, w, dtype, 100 + k, 0.02)
        cases.append((wl, pool_mode, window_mode))
    return cases


CASES = random_cases()


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_random_shape(case):
    w, pool_mode, window_mode = case
    idx = CASES.index(case)
    Q, K, V = make_qkv(w, "cuda")
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w, pool_mode=pool_mode, window_mode=window_mode)
    torch.cuda.synchronize()
    Oref, Lref, Kref, Vref = oracle.prefill(Q, K, V, w.g, w.w, pool_mode=pool_mode, window_mode=window_mode)
    check_cores(Kc, Vc, Kref, Vref, Q.dtype, w.name)
    # attention alone on the GPU's own core tokens (separates pooling from attention error)
    Oa, La = oracle.attn(Q, K, V, Kc, Vc, w.g, w.w, window_mode=window_mode)
    check_out(O, LSE, Oa, La, Q.dtype, w.name + " (attention)")
    check_out(O, LSE, Oref, Lref, Q.dtype, w.name + " (end to end)")
    if idx % 3 != 1:
        return
    # backward
    gen = torch.Generator(device="cuda").manual_seed(w.seed + 7)
    dO = torch.randn(Q.shape, generator=gen, device="cuda").to(Q.dtype)
    dQ, dK, dV = api.cca_prefill_bwd(Q, K, V, Kc, Vc, O, LSE, dO, w.g, w.w, pool_mode=pool_mode,
                                     window_mode=window_mode)
    torch.cuda.synchronize()
    rQ, rK, rV = prefill_grads(Q, K, V, dO, w.g, w.w, pool_mode=pool_mode, window_mode=window_mode)
    for name, got, ref in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV)):
        err = np.abs(got.double().cpu().numpy() - ref)
        scale = np.abs(ref).max()
        if Q.dtype == torch.float32:
            assert err.max() <= 1e-4 * scale + 1e-6, (w.name, name, err.max(), scale)
        else:
            assert err.max() <= 2e-2 * scale, (w.name, name, err.max(), scale)
            assert err.mean() <= 2e-3 * scale, (w.name, name, err.mean(), scale)
    # decode step at the last position (window mode 0 only: the decode call takes the mode too)
    pos = w.N - 1
    q = Q[:, :, pos].contiguous()
    Od, Ld = api.cca_decode_fwd(q, K, V, Kc, Vc, pos, w.g, w.w, window_mode=window_mode)
    torch.cuda.synchronize()
    rows = [(b, h, pos) for b in range(w.B) for h in range(w.Hq)]
    Or, Lr = oracle.attn_rows(Q, K, V, Kc, Vc, w.g, w.w, rows, window_mode=window_mode)
    check_out(Od.reshape(-1, w.d), Ld.reshape(-1), Or, Lr, Q.dtype, w.name + " (decode)")
