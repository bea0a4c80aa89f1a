"""Backward pass on the GPU against the fp64 backward oracle (autograd of the
dense forward, itself pinned by finite differences)."""
import numpy as np
import pytest
import torch

import oracle
from oracle.backward import prefill_grads
from sparse_long_context_cca_gb300 import api
from sparse_long_context_cca_gb300.inputs import make_qkv
from sparse_long_context_cca_gb300.workloads import Workload

pytestmark = pytest.mark.gpu


def wl(B, Hq, Hkv, N, d, g, w, dtype="bf16", seed=31):
    return Workload(f"bwd B{B} Hq{Hq} Hkv{Hkv} N{N} d{d} g{g} w{w} {dtype}", B, Hq, Hkv, N, d, g, w, dtype, seed, 0.01)


CASES = [
    (wl(1, 2, 2, 256, 64, 16, 32, "f32"), 0, 0), (wl(1, 4, 2, 384, 128, 8, 50, "f32"), 0, 1),
    (wl(1, 2, 2, 256, 64, 4, 20, "f32"), 1, 0), (wl(1, 2, 1, 320, 64, 5, 40, "f32"), 2, 0),
    (wl(1, 4, 4, 512, 128, 16, 64), 0, 0), (wl(2, 4, 2, 512, 128, 16, 100), 0, 1),
    (wl(1, 2, 2, 256, 128, 1, 40), 0, 0),
    # several core tiles (G = 260), ragged last tile, GQA r = 4
    (wl(1, 4, 1, 1040, 128, 4, 70), 0, 0),
    # window of one token, mean pooling, group-aligned window
    (wl(1, 2, 2, 640, 128, 8, 1), 1, 1),
    # max pooling, window wider than a tile
    (wl(1, 2, 2, 384, 128, 16, 300), 2, 0),
    # window covers the whole sequence: no core is ever visible
    (wl(1, 2, 2, 256, 128, 16, 512), 0, 0),
    # the pooling backward folded into the raw-token rows: groups that straddle
    # 128-key tiles, groups longer than a tile, ragged N with GQA
    (wl(1, 2, 2, 768, 128, 24, 100), 0, 0),
    (wl(1, 4, 2, 768, 128, 192, 200), 0, 0),
    (wl(1, 2, 1, 1000, 128, 40, 150), 1, 1),
    (wl(1, 8, 2, 520, 128, 8, 60), 0, 1),
]


@pytest.mark.parametrize("w,pool_mode,window_mode", CASES, ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_backward_parity(w, pool_mode, window_mode):
    Q, K, V = make_qkv(w, "cuda")
    gen = torch.Generator(device="cuda").manual_seed(w.seed + 100)
    dO = torch.randn(Q.shape, generator=gen, device="cuda").to(Q.dtype)
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w, pool_mode=pool_mode, window_mode=window_mode)
    dQ, dK, dV = api.cca_prefill_bwd(Q, K, V, Kc, Vc, O, LSE, dO, w.g, w.w, pool_mode=pool_mode,
                                     window_mode=window_mode)
    torch.cuda.synchronize()
    rQ, rK, rV = prefill_grads(Q, K, V, dO, w.g, w.w, pool_mode=pool_mode, window_mode=window_mode)
    for name, got, ref in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV)):
        g = got.double().cpu().numpy()
        assert np.isfinite(g).all(), name
        err = np.abs(g - ref)
        scale = np.abs(ref).max()
        if Q.dtype == torch.float32:
            assert err.max() <= 1e-4 * scale + 1e-6, (name, err.max(), scale)
        else:
            assert err.max() <= 2e-2 * scale, (name, err.max(), scale)
            assert err.mean() <= 2e-3 * scale, (name, err.mean(), scale)


@pytest.mark.parametrize("w,pool_mode", [(wl(1, 2, 1, 8448, 128, 16, 256, seed=41), 0),
                                         (wl(1, 1, 1, 8448, 128, 24, 300, seed=42), 1)],
                         ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_backward_core_tiles_over_several_query_chunks(w, pool_mode):
    """The tensor-core backward splits each core tile's query range into chunks of 64 query
    tiles and adds the chunks' dKc/dVc shares together; at N = 8448 (66 query tiles) the
    first core tiles are seen from both chunks, the last core tile is ragged, and r = 2 in
    the first case."""
    Q, K, V = make_qkv(w, "cuda")
    gen = torch.Generator(device="cuda").manual_seed(w.seed + 100)
    dO = torch.randn(Q.shape, generator=gen, device="cuda").to(Q.dtype)
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w, pool_mode=pool_mode)
    dQ, dK, dV = api.cca_prefill_bwd(Q, K, V, Kc, Vc, O, LSE, dO, w.g, w.w, pool_mode=pool_mode)
    torch.cuda.synchronize()
    rQ, rK, rV = prefill_grads(Q, K, V, dO, w.g, w.w, pool_mode=pool_mode)
    for name, got, ref in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV)):
        g = got.double().cpu().numpy()
        assert np.isfinite(g).all(), name
        err = np.abs(g - ref)
        scale = np.abs(ref).max()
        assert err.max() <= 2e-2 * scale, (name, err.max(), scale)
        assert err.mean() <= 2e-3 * scale, (name, err.mean(), scale)
