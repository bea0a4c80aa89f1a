"""Groups of 256 to 1024 tokens against the fp64 oracle.

With the raw window aligned to group boundaries (window_mode 1), the second
128-row half of an attention work item can start its band several 128-key tiles
after its last core tile, and a whole band can sit inside one group.  These
cases take the attention kernel's path that holds back such a tile's score MMA
until the K/V ring can take its copies; every case also runs the backward and a
decode step."""
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


def wl(B, Hq, Hkv, N, d, g, w, dtype="bf16", seed=41):
    return Workload(f"large-group B{B} Hq{Hq} Hkv{Hkv} N{N} d{d} g{g} w{w} {dtype}", B, Hq, Hkv, N, d, g, w,
                    dtype, seed, 0.01)


CASES = [
    (wl(1, 2, 2, 2048, 128, 256, 4), 1), (wl(1, 2, 2, 2048, 128, 256, 300), 1),
    (wl(1, 2, 1, 3072, 128, 512, 4), 1), (wl(1, 2, 2, 3072, 128, 512, 700), 1),
    (wl(1, 2, 2, 4096, 128, 1024, 100), 1), (wl(1, 2, 2, 3072, 128, 512, 4), 0),
    (wl(1, 2, 2, 2304, 128, 384, 1), 1), (wl(1, 2, 2, 2048, 64, 512, 4, "f32"), 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name} m{c[1]}")
def test_large_group(case):
    w, window_mode = case
    Q, K, V = make_qkv(w, "cuda")
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w, window_mode=window_mode)
    torch.cuda.synchronize()
    Oref, Lref, Kref, Vref = oracle.prefill(Q, K, V, w.g, w.w, window_mode=window_mode)
    check_cores(Kc, Vc, Kref, Vref, Q.dtype, w.name)
    Oa, La = oracle.attn(Q, K, V, Kc, Vc, w.g, w.w, window_mode=window_mode)
    check_out(O, LSE, Oa, La, Q.dtype, w.name + " (attention)")
    check_out(O, LSE, Oref, Lref, Q.dtype, w.name + " (end to end)")

    gen = torch.Generator(device="cuda").manual_seed(w.seed + 7)
    dO = torch.randn(Q.shape, generator=gen, device="cuda").to(Q.dtype)
    dQ, dK, dV = api.cca_prefill_bwd(Q, K, V, Kc, Vc, O, LSE, dO, w.g, w.w, window_mode=window_mode)
    torch.cuda.synchronize()
    rQ, rK, rV = prefill_grads(Q, K, V, dO, w.g, w.w, window_mode=window_mode)
    for name, got, ref in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV)):
        err = np.abs(got.double().cpu().numpy() - ref)
        scale = np.abs(ref).max()
        if Q.dtype == torch.float32:
            assert err.max() <= 1e-4 * scale + 1e-6, (w.name, name, err.max(), scale)
        else:
            assert err.max() <= 2e-2 * scale, (w.name, name, err.max(), scale)
            assert err.mean() <= 2e-3 * scale, (w.name, name, err.mean(), scale)

    for pos in (w.N - 1, w.N - w.g - 1):
        q = Q[:, :, pos].contiguous()
        Od, Ld = api.cca_decode_fwd(q, K, V, Kc, Vc, pos, w.g, w.w, window_mode=window_mode)
        torch.cuda.synchronize()
        rows = [(b, h, pos) for b in range(w.B) for h in range(w.Hq)]
        Or, Lr = oracle.attn_rows(Q, K, V, Kc, Vc, w.g, w.w, rows, window_mode=window_mode)
        check_out(Od.reshape(-1, w.d), Ld.reshape(-1), Or, Lr, Q.dtype, f"{w.name} (decode at {pos})")
