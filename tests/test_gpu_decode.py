"""Decode step on the GPU: one new token per sequence attends to the visible
core tokens and its window, i.e. row `pos` of the fused attention; groups are
pooled as they complete.  Checked against the fp64 oracle's rows and against
the prefill kernels."""
import numpy as np
import pytest
import torch

import oracle
from parity import check_cores, check_out
from sparse_long_context_cca_gb300 import api
from sparse_long_context_cca_gb300.inputs import make_qkv
from sparse_long_context_cca_gb300.workloads import Workload

pytestmark = pytest.mark.gpu


def wl(B, Hq, Hkv, N, d, g, w, dtype="bf16", seed=11):
    return Workload(f"decode B{B} Hq{Hq} Hkv{Hkv} N{N} d{d} g{g} w{w} {dtype}", B, Hq, Hkv, N, d, g, w, dtype,
                    seed, 0.01)


CASES = [wl(1, 4, 4, 4096, 128, 16, 1024), wl(2, 8, 2, 2048, 128, 16, 256), wl(1, 4, 1, 3000, 128, 8, 500),
         wl(1, 2, 2, 1024, 64, 4, 100), wl(1, 4, 2, 1024, 128, 16, 200, "f32"), wl(1, 2, 2, 512, 64, 32, 64, "f32"),
         # eight query heads per KV head (bf16 d = 128 and d = 64, f32 d = 128)
         wl(1, 8, 1, 2048, 128, 16, 300), wl(2, 16, 2, 1024, 64, 8, 200), wl(1, 8, 1, 768, 128, 16, 100, "f32")]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_decode_rows_match_oracle(w):
    Q, K, V = make_qkv(w, "cuda")
    Kc, Vc = api.cca_pool(Q, K, V, w.g)
    Kr, Vr = oracle.pool(Q, K, V, w.g)
    rng = np.random.default_rng(w.seed)
    positions = sorted({0, 1, w.w - 2, w.w - 1, w.w, w.w + w.g - 1, w.w + w.g, w.N // 2, w.N - 1}
                       | set(rng.integers(0, w.N, 6).tolist()))
    ws = torch.empty(api.decode_workspace_size(w.B, w.Hq, w.Hkv, w.N, w.d, w.g, w.w, Q.dtype),
                     dtype=torch.uint8, device="cuda")
    for pos in positions:
        if not 0 <= pos < w.N:
            continue
        q = Q[:, :, pos].contiguous()
        O, LSE = api.cca_decode_fwd(q, K, V, Kc, Vc, pos, w.g, w.w, workspace=ws)
        torch.cuda.synchronize()
        rows = [(b, h, pos) for b in range(w.B) for h in range(w.Hq)]
        Oa, La = oracle.attn_rows(Q, K, V, Kc, Vc, w.g, w.w, rows)   # the GPU's own core tokens
        check_out(O.reshape(-1, w.d), LSE.reshape(-1), Oa, La, Q.dtype, f"{w.name} pos {pos} attention")
        Oe, Le = oracle.attn_rows(Q, K, V, Kr, Vr, w.g, w.w, rows)   # fp64 core tokens
        check_out(O.reshape(-1, w.d), LSE.reshape(-1), Oe, Le, Q.dtype, f"{w.name} pos {pos} end-to-end")


def test_decode_matches_prefill_row():
    w = wl(1, 8, 8, 2048, 128, 16, 512)
    Q, K, V = make_qkv(w, "cuda")
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w)
    for pos in (0, 700, 1500, 2047):
        Od, Ld = api.cca_decode_fwd(Q[:, :, pos].contiguous(), K, V, Kc, Vc, pos, w.g, w.w)
        torch.cuda.synchronize()
        a, b = Od.float(), O[:, :, pos].float()
        assert (a - b).abs().max().item() <= 2e-2 * b.abs().max().item()
        assert (Ld - LSE[:, :, pos]).abs().max().item() <= 5e-3


@pytest.mark.parametrize("w", [wl(2, 8, 2, 1024, 128, 16, 128), wl(1, 2, 2, 640, 64, 5, 50, "f32"),
                               wl(1, 4, 4, 512, 128, 1, 16)], ids=lambda w: w.name)
def test_pool_group_matches_full_pooling(w):
    Q, K, V = make_qkv(w, "cuda")
    Kc, Vc = api.cca_pool(Q, K, V, w.g)
    Kg = torch.zeros_like(Kc)
    Vg = torch.zeros_like(Vc)
    for j in (0, 1, w.N // w.g // 2, w.N // w.g - 1):
        api.cca_pool_group(Q[:, :, (j + 1) * w.g - 1].contiguous(), K, V, Kg, Vg, j, w.g)
    torch.cuda.synchronize()
    Kr, Vr = oracle.pool(Q, K, V, w.g)
    for j in (0, 1, w.N // w.g // 2, w.N // w.g - 1):
        check_cores(Kg[:, :, j], Vg[:, :, j], Kr[:, :, j], Vr[:, :, j], Q.dtype, f"{w.name} group {j}")


def test_incremental_decode_loop():
    """Prefill the first P tokens, then decode one token at a time, pooling each group
    as soon as its last token is decoded; every step equals the oracle's row."""
    w = wl(1, 4, 2, 1536, 128, 16, 256)
    Q, K, V = make_qkv(w, "cuda")
    P = 1000
    G = w.N // w.g
    Kc = torch.zeros((w.B, w.Hkv, G, w.d), dtype=Q.dtype, device="cuda")
    Vc = torch.zeros_like(Kc)
    # cores of the groups complete inside the prefix
    for j in range(P // w.g):
        api.cca_pool_group(Q[:, :, (j + 1) * w.g - 1].contiguous(), K, V, Kc, Vc, j, w.g)
    Kr, Vr = oracle.pool(Q, K, V, w.g)
    ws = torch.empty(api.decode_workspace_size(w.B, w.Hq, w.Hkv, w.N, w.d, w.g, w.w, Q.dtype),
                     dtype=torch.uint8, device="cuda")
    for pos in range(P, P + 70):
        q = Q[:, :, pos].contiguous()
        O, LSE = api.cca_decode_fwd(q, K, V, Kc, Vc, pos, w.g, w.w, workspace=ws)
        if (pos + 1) % w.g == 0:
            api.cca_pool_group(q, K, V, Kc, Vc, (pos + 1) // w.g - 1, w.g)
        torch.cuda.synchronize()
        rows = [(0, h, pos) for h in range(w.Hq)]
        Oe, Le = oracle.attn_rows(Q, K, V, Kr, Vr, w.g, w.w, rows)
        check_out(O.reshape(-1, w.d), LSE.reshape(-1), Oe, Le, Q.dtype, f"step {pos}")


@pytest.mark.parametrize("pool_mode", [1, 2])
def test_pool_group_variants(pool_mode):
    w = wl(1, 4, 2, 512, 128, 16, 64)
    Q, K, V = make_qkv(w, "cuda")
    Kg = torch.zeros((w.B, w.Hkv, w.N // w.g, w.d), dtype=Q.dtype, device="cuda")
    Vg = torch.zeros_like(Kg)
    for j in range(w.N // w.g):
        api.cca_pool_group(Q[:, :, (j + 1) * w.g - 1].contiguous(), K, V, Kg, Vg, j, w.g, pool_mode=pool_mode)
    torch.cuda.synchronize()
    Kr, Vr = oracle.pool(Q, K, V, w.g, pool_mode=pool_mode)
    check_cores(Kg, Vg, Kr, Vr, Q.dtype, f"pool_group mode {pool_mode}")


@pytest.mark.parametrize("path", [0, 2], ids=["auto", "cluster"])
def test_decode_group_aligned_window(path):
    lib = api.load_library()
    lib.cca_test_decode_path(path)
    try:
        _decode_group_aligned_window()
    finally:
        lib.cca_test_decode_path(0)


def _decode_group_aligned_window():
    w = wl(1, 4, 2, 2048, 128, 16, 300)
    Q, K, V = make_qkv(w, "cuda")
    Kc, Vc = api.cca_pool(Q, K, V, w.g)
    for pos in (5, 299, 300, 316, 1000, 2047):
        O, LSE = api.cca_decode_fwd(Q[:, :, pos].contiguous(), K, V, Kc, Vc, pos, w.g, w.w, window_mode=1)
        torch.cuda.synchronize()
        rows = [(0, h, pos) for h in range(w.Hq)]
        Oa, La = oracle.attn_rows(Q, K, V, Kc, Vc, w.g, w.w, rows, window_mode=1)
        check_out(O.reshape(-1, w.d), LSE.reshape(-1), Oa, La, Q.dtype, f"aligned window pos {pos}")


@pytest.mark.parametrize("graphed", [False, True], ids=["eager", "graph"])
def test_chained_steps_wait_for_the_step_before(graphed):
    """Decode steps through several layers where each layer's query is the previous
    layer's output: the split kernel is a programmatic dependent of the merge kernel before
    it, which lets its dependents start as soon as it has waited for its own split kernel,
    before it writes O.  Each step must still read the finished O of the one before, so the
    chain (launched back to back on one stream, eagerly or as one CUDA graph) equals the
    same steps run one at a time with a synchronisation in between."""
    w = wl(1, 8, 2, 2048, 128, 16, 300, seed=31)
    n_layers = 6
    gen = torch.Generator(device="cuda").manual_seed(77)
    layers = []
    for _ in range(n_layers):
        K, V = (torch.randn((w.B, w.Hkv, w.N, w.d), generator=gen, device="cuda").mul_(w.d ** -0.25)
                .to(torch.bfloat16) for _ in range(2))
        Kc, Vc = (torch.randn((w.B, w.Hkv, w.N // w.g, w.d), generator=gen, device="cuda").mul_(w.d ** -0.25)
                  .to(torch.bfloat16) for _ in range(2))
        ws = torch.empty(api.decode_workspace_size(w.B, w.Hq, w.Hkv, w.N, w.d, w.g, w.w, torch.bfloat16),
                         dtype=torch.uint8, device="cuda")
        layers.append((K, V, Kc, Vc, ws))
    pos = w.N - 1
    q0 = torch.randn((w.B, w.Hq, w.d), generator=gen, device="cuda").to(torch.bfloat16)
    outs = [torch.empty_like(q0) for _ in range(n_layers)]
    lses = [torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda") for _ in range(n_layers)]

    def chain():
        q = q0
        for (K, V, Kc, Vc, ws), O, L in zip(layers, outs, lses):
            api.cca_decode_fwd(q, K, V, Kc, Vc, pos, w.g, w.w, O, L, ws)
            q = O

    # one step at a time
    ref = []
    q = q0
    for K, V, Kc, Vc, ws in layers:
        O, L = api.cca_decode_fwd(q, K, V, Kc, Vc, pos, w.g, w.w, workspace=ws)
        torch.cuda.synchronize()
        ref.append((O.clone(), L.clone()))
        q = O
    if graphed:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            chain()
    for _ in range(5):
        # poison what each kernel reads from the one before it: a split kernel reading its
        # query (the previous layer's O) or a merge reading its workspace too early would
        # propagate NaN
        for O in outs:
            O.fill_(float("nan"))
        for *_, ws in layers:
            ws.fill_(0xFF)
        torch.cuda.synchronize()
        if graphed:
            graph.replay()
        else:
            chain()
        torch.cuda.synchronize()
        for (O, L), (rO, rL) in zip(zip(outs, lses), ref):
            assert torch.equal(O, rO) and torch.equal(L, rL)
    # and the chain's first layer against the oracle
    Oa, La = oracle.attn_rows(q0.unsqueeze(2).expand(w.B, w.Hq, w.N, w.d), layers[0][0], layers[0][1],
                              layers[0][2], layers[0][3], w.g, w.w,
                              [(0, h, pos) for h in range(w.Hq)])
    check_out(ref[0][0].reshape(-1, w.d), ref[0][1].reshape(-1), Oa, La, torch.bfloat16, "chained layer 0")


@pytest.fixture
def decode_path():
    lib = api.load_library()
    yield lambda path: lib.cca_test_decode_path(path)
    lib.cca_test_decode_path(0)


@pytest.mark.parametrize("path", [1, 2], ids=["split+merge", "cluster"])
@pytest.mark.parametrize("w", [CASES[0], CASES[1], CASES[3], CASES[4], CASES[5], CASES[6]], ids=lambda w: w.name)
def test_both_decode_paths_match_oracle(w, path, decode_path):
    """The two ways the splits are merged: through the workspace by a second kernel, or
    inside a thread-block cluster by the first CTA (one launch)."""
    decode_path(path)
    Q, K, V = make_qkv(w, "cuda")
    Kc, Vc = api.cca_pool(Q, K, V, w.g)
    for pos in (w.N - 1, w.N // 2, w.w + 3, 5):
        q = Q[:, :, pos].contiguous()
        O, LSE = api.cca_decode_fwd(q, K, V, Kc, Vc, pos, w.g, w.w)
        O2, L2 = api.cca_decode_fwd(q, K, V, Kc, Vc, pos, w.g, w.w)
        torch.cuda.synchronize()
        assert torch.equal(O, O2) and torch.equal(LSE, L2)
        rows = [(b, h, pos) for b in range(w.B) for h in range(w.Hq)]
        Oa, La = oracle.attn_rows(Q, K, V, Kc, Vc, w.g, w.w, rows)
        check_out(O.reshape(-1, w.d), LSE.reshape(-1), Oa, La, Q.dtype, f"{w.name} pos {pos} path {path}")


def test_decode_kernel_count(decode_path):
    """The call says how many kernels it launches: one where the splits merge inside their
    cluster (the 128K caches of 32 heads), two where a merge kernel follows (the 32K ones,
    and grouped-query heads with few (b, kv) pairs)."""
    bf = torch.bfloat16
    assert api.decode_kernels(1, 32, 32, 131072, 128, 16, 1024, bf, 131071) == 1
    assert api.decode_kernels(1, 32, 32, 32768, 128, 16, 1024, bf, 32767) == 2
    assert api.decode_kernels(1, 32, 8, 65536, 128, 16, 1024, bf, 65535) == 2
    decode_path(1)
    assert api.decode_kernels(1, 32, 32, 131072, 128, 16, 1024, bf, 131071) == 2
    decode_path(2)
    assert api.decode_kernels(1, 32, 32, 32768, 128, 16, 1024, bf, 32767) == 1
