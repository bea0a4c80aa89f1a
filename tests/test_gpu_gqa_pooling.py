"""The alternative grouped-query pooling (pool_mode 3: each query head's own softmax
weights over the group, averaged over the r heads sharing the KV head) through the
CUDA path against the fp64 oracle: the prefill (pooling + attention), the decode
step's group pooling, the backward, and the GQA 64K workload at full size.

Groups that fit one pooling chunk take the kernel's one-pass path (g <= 16 at
d = 128 bf16, g <= 32 at d = 64 bf16, g <= 8 at d = 128 f32, g <= 16 at d = 64
f32); longer groups take the two-pass path (K statistics first, then the
weighted sums)."""
import numpy as np
import pytest
import torch

import oracle
from oracle.backward import prefill_grads
from parity import BF16_LSE, BF16_O_MAX_REL, BF16_O_MEAN, check_cores, check_out
from sparse_long_context_cca_gb300 import api
from sparse_long_context_cca_gb300.inputs import make_qkv
from sparse_long_context_cca_gb300.workloads import GQA_64K, Workload

pytestmark = pytest.mark.gpu


def wl(B, Hq, Hkv, N, d, g, w, dtype="bf16", seed=61):
    return Workload(f"gqa-post B{B} Hq{Hq} Hkv{Hkv} N{N} d{d} g{g} w{w} {dtype}", B, Hq, Hkv, N, d, g, w, dtype,
                    seed, 0.02)


PREFILL_CASES = [
    (wl(1, 8, 2, 1024, 128, 16, 200), 0),       # r = 4, one chunk per group
    (wl(2, 8, 1, 768, 128, 8, 100), 1),         # r = 8, small groups, aligned window
    (wl(1, 4, 2, 1536, 128, 64, 300), 0),       # r = 2, four chunks per group: two passes
    (wl(1, 8, 2, 960, 128, 24, 128), 0),        # ragged last chunk (24 = 16 + 8)
    (wl(1, 2, 2, 512, 128, 16, 64), 0),         # r = 1: equals the method's pooling
    (wl(1, 4, 1, 640, 128, 1, 50), 0),          # one-token groups
    (wl(1, 4, 2, 1000, 128, 40, 333), 1),       # ragged N, two passes, aligned window
    (wl(1, 4, 2, 512, 64, 16, 70, "f32"), 0),   # f32, d = 64: one chunk
    (wl(1, 8, 2, 576, 128, 24, 90, "f32"), 0),  # f32, d = 128: three chunks, two passes
]


@pytest.mark.parametrize("w,window_mode", PREFILL_CASES, ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_prefill_parity(w, window_mode):
    Q, K, V = make_qkv(w, "cuda")
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w, pool_mode=3, window_mode=window_mode)
    torch.cuda.synchronize()
    Or, Lr, Kr, Vr = oracle.prefill(Q, K, V, w.g, w.w, pool_mode=3, window_mode=window_mode)
    check_cores(Kc, Vc, Kr, Vr, Q.dtype, f"{w.name} cores")
    check_out(O, LSE, Or, Lr, Q.dtype, f"{w.name} output")
    if w.Hq > w.Hkv and w.g > 1:
        # the mode is really different from the logit-mean pooling on these inputs
        K0, _ = oracle.pool(Q, K, V, w.g, pool_mode=0)
        assert np.abs(K0 - Kr).max() > 1e-3


def test_pooling_repeats_bitwise():
    w = wl(1, 8, 2, 2064, 128, 48, 200)
    Q, K, V = make_qkv(w, "cuda")
    a = api.cca_pool(Q, K, V, w.g, pool_mode=3)
    b = api.cca_pool(Q, K, V, w.g, pool_mode=3)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("w", [wl(1, 8, 2, 512, 128, 16, 64), wl(1, 4, 1, 384, 128, 48, 64),
                               wl(2, 4, 2, 256, 64, 16, 32, "f32")], ids=lambda x: x.name)
def test_pool_group(w):
    """The decode step's group pooling in the same mode: pooling every group one at a
    time gives the oracle's core tokens."""
    Q, K, V = make_qkv(w, "cuda")
    Kg = torch.zeros((w.B, w.Hkv, w.N // w.g, w.d), dtype=Q.dtype, device="cuda")
    Vg = torch.zeros_like(Kg)
    for j in range(w.N // w.g):
        api.cca_pool_group(Q[:, :, (j + 1) * w.g - 1].contiguous(), K, V, Kg, Vg, j, w.g, pool_mode=3)
    torch.cuda.synchronize()
    Kr, Vr = oracle.pool(Q, K, V, w.g, pool_mode=3)
    check_cores(Kg, Vg, Kr, Vr, Q.dtype, f"{w.name} pool_group")


BWD_CASES = [wl(1, 8, 2, 512, 128, 16, 64), wl(1, 4, 2, 640, 128, 40, 100), wl(1, 4, 2, 256, 64, 8, 40, "f32")]


@pytest.mark.parametrize("w", BWD_CASES, ids=lambda x: x.name)
def test_backward_parity(w):
    Q, K, V = make_qkv(w, "cuda")
    gen = torch.Generator(device="cuda").manual_seed(w.seed + 100)
    dO = torch.randn(Q.shape, generator=gen, device="cuda").to(Q.dtype)
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w, pool_mode=3)
    dQ, dK, dV = api.cca_prefill_bwd(Q, K, V, Kc, Vc, O, LSE, dO, w.g, w.w, pool_mode=3)
    torch.cuda.synchronize()
    rQ, rK, rV = prefill_grads(Q, K, V, dO, w.g, w.w, pool_mode=3)
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


def test_gqa_64k_full_size():
    """GQA 64K (32 query heads over 8 KV heads) in this mode at full size, in the
    benchmark's launch configuration: sampled groups of three KV heads and sampled rows
    of one query head of each against the oracle."""
    w = GQA_64K
    torch.cuda.empty_cache()
    Q, K, V = make_qkv(w, "cuda")
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w, pool_mode=3)
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    r = w.Hq // w.Hkv
    for kv in (0, 3, 7):
        hs = slice(kv * r, (kv + 1) * r)
        q, k, v = Q[:, hs], K[:, kv:kv + 1], V[:, kv:kv + 1]
        Kr, Vr = oracle.pool(q, k, v, w.g, pool_mode=3)
        groups = np.unique(np.concatenate([[0, w.n_groups - 1], rng.integers(0, w.n_groups, 64)]))
        gi = torch.as_tensor(groups, device=Kc.device)
        check_cores(Kc[0, kv, gi], Vc[0, kv, gi], Kr[0, 0, groups], Vr[0, 0, groups], Q.dtype, f"kv{kv}")
        rows = sorted({0, w.w - 1, w.w, w.w + w.g - 1, w.N // 2, w.N - 1} | set(rng.integers(0, w.N, 40).tolist()))
        hh = int(rng.integers(0, r))
        Or, Lr = oracle.attn_rows(q, k, v, Kr, Vr, w.g, w.w, [(0, hh, i) for i in rows])
        o = oracle.widen(O[0, kv * r + hh, rows])
        err = np.abs(o - Or)
        assert err.max() <= BF16_O_MAX_REL * np.abs(Or).max(), (kv, err.max())
        assert err.mean() <= BF16_O_MEAN, (kv, err.mean())
        assert np.abs(oracle.widen(LSE[0, kv * r + hh, rows]) - Lr).max() <= BF16_LSE
