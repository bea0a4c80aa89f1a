"""The autograd wrapper (forward = cca_prefill, backward = cca_prefill_bwd) gives the
fp64 oracle's gradients of a scalar loss, through torch.autograd."""
import numpy as np
import pytest
import torch

from oracle.backward import prefill_grads
from sparse_long_context_cca_gb300 import api
from sparse_long_context_cca_gb300.inputs import make_qkv
from sparse_long_context_cca_gb300.workloads import Workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,d,pool_mode,window_mode", [("bf16", 128, 0, 0), ("f32", 64, 1, 1), ("bf16", 128, 2, 0)])
def test_autograd_matches_oracle(dtype, d, pool_mode, window_mode):
    w = Workload(f"autograd {dtype}", 1, 4, 2, 384, d, 16, 100, dtype, 77, 0.01)
    Q, K, V = (t.requires_grad_(True) for t in make_qkv(w, "cuda"))
    gen = torch.Generator(device="cuda").manual_seed(3)
    dO = torch.randn(Q.shape, generator=gen, device="cuda").to(Q.dtype)
    O = api.cca_attention(Q, K, V, w.g, w.w, pool_mode=pool_mode, window_mode=window_mode)
    (O.float() * dO.float()).sum().backward()
    torch.cuda.synchronize()
    rQ, rK, rV = prefill_grads(Q.detach(), K.detach(), V.detach(), dO, w.g, w.w, pool_mode=pool_mode,
                               window_mode=window_mode)
    for name, got, ref in (("dQ", Q.grad, rQ), ("dK", K.grad, rK), ("dV", V.grad, rV)):
        assert got.dtype == Q.dtype
        err = np.abs(got.double().cpu().numpy() - ref)
        scale = np.abs(ref).max()
        if dtype == "f32":
            assert err.max() <= 1e-4 * scale + 1e-6, (name, err.max())
        else:
            # the gradient is also rounded to bf16 on the way out: one more 2^-8 relative
            assert err.max() <= 2e-2 * scale, (name, err.max())
            assert err.mean() <= 3e-3 * scale, (name, err.mean())
