"""Parity at the full workload sizes, in the launch configuration the benchmark
times: the whole prefill runs on the GPU; the fp64 oracle recomputes sampled
rows (boundary rows of the window/core edges and tiles plus random rows) of a
few heads, and the sampled groups' core tokens."""
import numpy as np
import pytest
import torch

import oracle
from parity import BF16_LSE, BF16_O_MAX_REL, BF16_O_MEAN, check_cores
from sparse_long_context_cca_gb300 import api
from sparse_long_context_cca_gb300.inputs import make_qkv
from sparse_long_context_cca_gb300.workloads import GQA_64K, MHA_32K, MHA_128K, sweep

pytestmark = pytest.mark.gpu


def sample_rows(N, g, w, rng, n_random):
    edges = [0, 1, w - 2, w - 1, w, w + g - 2, w + g - 1, w + g, 127, 128, 129, N // 2, N - 129, N - 128,
             N - 2, N - 1]
    rows = {i for i in edges if 0 <= i < N}
    rows |= set(rng.integers(0, N, size=n_random).tolist())
    return sorted(rows)


def check_workload(wl, heads, n_random=48):
    torch.cuda.empty_cache()
    Q, K, V = make_qkv(wl, "cuda")
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, wl.g, wl.w)
    torch.cuda.synchronize()
    assert torch.isfinite(LSE).all()
    rng = np.random.default_rng(wl.seed)
    r = wl.Hq // wl.Hkv
    for (b, h) in heads:
        kv = h // r
        hs = slice(kv * r, (kv + 1) * r)
        q = Q[b:b + 1, hs]
        k = K[b:b + 1, kv:kv + 1]
        v = V[b:b + 1, kv:kv + 1]
        Kr, Vr = oracle.pool(q, k, v, wl.g)
        groups = np.unique(np.concatenate([[0, wl.n_groups - 1], rng.integers(0, wl.n_groups, 64)]))
        gi = torch.as_tensor(groups, device=Kc.device)
        check_cores(Kc[b, kv, gi], Vc[b, kv, gi], Kr[0, 0, groups], Vr[0, 0, groups], Q.dtype,
                    f"{wl.name} b{b} kv{kv}")
        rows = sample_rows(wl.N, wl.g, wl.w, rng, n_random)
        sel = [(0, h - kv * r, i) for i in rows]
        Or, Lr = oracle.attn_rows(q, k, v, Kr, Vr, wl.g, wl.w, sel)
        o = oracle.widen(O[b, h, rows])
        err = np.abs(o - Or)
        assert err.max() <= BF16_O_MAX_REL * np.abs(Or).max(), (wl.name, h, err.max())
        assert err.mean() <= BF16_O_MEAN, (wl.name, h, err.mean())
        lerr = np.abs(oracle.widen(LSE[b, h, rows]) - Lr)
        assert lerr.max() <= BF16_LSE, (wl.name, h, lerr.max())
    del Q, K, V, O, LSE, Kc, Vc


def test_mha_32k():
    check_workload(MHA_32K, [(0, 0), (0, 17), (0, 31)])


def test_mha_128k():
    check_workload(MHA_128K, [(0, 0), (0, 31)], n_random=32)


def test_gqa_64k():
    check_workload(GQA_64K, [(0, 0), (0, 5), (0, 31)])


@pytest.mark.parametrize("wl", sweep(), ids=lambda w: w.name)
def test_sweep(wl):
    check_workload(wl, [(1, 7)], n_random=24)


def test_mha_1m_tokens():
    """The largest context exercised: one million tokens (B1, 2 heads), where the last row
    sees 65,472 cores plus its 1024-token window; sampled rows and groups of both heads."""
    from sparse_long_context_cca_gb300.workloads import Workload
    wl = Workload("mha B1 H2 d128 N1048576 g16 w1024", 1, 2, 2, 1 << 20, 128, 16, 1024, "bf16", 31, 0.01)
    check_workload(wl, [(0, 0), (0, 1)], n_random=24)


@pytest.mark.parametrize("wl", [MHA_32K, MHA_128K, GQA_64K], ids=lambda w: w.name)
def test_decode_full_size(wl):
    """The decode step at the full workload sizes, in the benchmark's launch configuration
    (at 128K the one-launch cluster merge, at 32K and GQA 64K the split + merge kernels):
    the last position and the middle one, all heads, against the prefill's own rows and,
    for a few heads, against the fp64 oracle over the GPU's core tokens."""
    torch.cuda.empty_cache()
    Q, K, V = make_qkv(wl, "cuda")
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, wl.g, wl.w)
    r = wl.Hq // wl.Hkv
    for pos in (wl.N - 1, wl.N // 2 + 5):
        q = Q[:, :, pos].contiguous()
        Od, Ld = api.cca_decode_fwd(q, K, V, Kc, Vc, pos, wl.g, wl.w)
        torch.cuda.synchronize()
        a, b = Od.float(), O[:, :, pos].float()
        assert (a - b).abs().max().item() <= 2e-2 * b.abs().max().item(), pos
        assert (Ld - LSE[:, :, pos]).abs().max().item() <= 5e-3, pos
        for h in (0, wl.Hq - 1):
            kv = h // r
            Or, Lr = oracle.attn_rows(Q[:, h:h + 1], K[:, kv:kv + 1], V[:, kv:kv + 1], Kc[:, kv:kv + 1],
                                      Vc[:, kv:kv + 1], wl.g, wl.w, [(0, 0, pos)])
            err = np.abs(oracle.widen(Od[0, h]) - Or[0])
            assert err.max() <= BF16_O_MAX_REL * np.abs(Or).max(), (pos, h, err.max())
            assert abs(float(Ld[0, h]) - Lr[0]) <= BF16_LSE, (pos, h)
    del Q, K, V, O, LSE, Kc, Vc
