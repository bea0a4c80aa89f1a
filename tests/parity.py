"""Comparison helpers shared by the GPU parity tests (tolerances stated here).

bf16 runs: max|dO| <= 2e-2 * max|O_ref| and mean|dO| <= 2e-3 (output), LSE
within 5e-3 absolute; core tokens within one bf16 ulp (2^-7 relative) plus
1e-3 * max|Kc|.  fp32 runs: max|dO| <= 1e-4, LSE within 1e-5, core tokens
within 1e-5.  References are the fp64 CPU oracle on the same inputs.
"""
import numpy as np
import torch

import oracle

BF16_O_MAX_REL = 2e-2
BF16_O_MEAN = 2e-3
BF16_LSE = 5e-3
F32_O = 1e-4
F32_LSE = 1e-5


def to64(t):
    return oracle.widen(t)


def check_out(O, LSE, Oref, Lref, dtype, what=""):
    o = to64(O)
    lse = to64(LSE)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what + ": non-finite output"
    err = np.abs(o - Oref)
    lerr = np.abs(lse - Lref)
    if dtype == torch.float32:
        assert err.max() <= F32_O, f"{what}: max|dO|={err.max():.3g}"
        assert lerr.max() <= F32_LSE, f"{what}: max|dLSE|={lerr.max():.3g}"
    else:
        assert err.max() <= BF16_O_MAX_REL * np.abs(Oref).max(), f"{what}: max|dO|={err.max():.3g}"
        assert err.mean() <= BF16_O_MEAN, f"{what}: mean|dO|={err.mean():.3g}"
        assert lerr.max() <= BF16_LSE, f"{what}: max|dLSE|={lerr.max():.3g}"
    return float(err.max()), float(err.mean()), float(lerr.max())


def check_cores(Kc, Vc, Kref, Vref, dtype, what=""):
    for name, got, ref in (("Kc", Kc, Kref), ("Vc", Vc, Vref)):
        g = to64(got)
        err = np.abs(g - ref)
        if dtype == torch.float32:
            assert err.max() <= 1e-5, f"{what}: {name} max err {err.max():.3g}"
        else:
            tol = 2.0 ** -7 * np.abs(ref) + 1e-3 * np.abs(ref).max()
            bad = err > tol
            assert not bad.any(), f"{what}: {name} {bad.sum()} elements off, max err {err.max():.3g}"
