"""CUDA graph capture of the library's launches.

The prefill step (pooling + fused attention) and a decode step (split kernel and
its merge, the merge a programmatic dependent launch, then the pooling of the
group the token completes) are captured once with torch.cuda.CUDAGraph and
replayed after new inputs are written into the captured buffers.  A replay must
give the same bits as the same calls made eagerly on those inputs: the launches
take their tensor maps and arguments by value, read nothing from the host while
they run, and allocate nothing."""
import ctypes

import pytest
import torch

from sparse_long_context_cca_gb300 import api
from sparse_long_context_cca_gb300.inputs import make_qkv
from sparse_long_context_cca_gb300.workloads import Workload

pytestmark = pytest.mark.gpu


def wl(seed, dtype="bf16", d=128):
    return Workload(f"graph {dtype} d{d} seed{seed}", 1, 4, 2, 1536, d, 16, 300, dtype, seed, 0.01)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_prefill_step_replays_bitwise(dtype, d):
    g, w = 16, 300
    Q, K, V = make_qkv(wl(11, dtype, d), "cuda")
    Kc, Vc = api.cca_pool(Q, K, V, g)  # eager first: buffers and per-device setup outside capture
    O, LSE = api.cca_attn_fwd(Q, K, V, Kc, Vc, g, w)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        api.cca_pool(Q, K, V, g, Kc, Vc)
        api.cca_attn_fwd(Q, K, V, Kc, Vc, g, w, O, LSE)
    for seed in (12, 13):
        q, k, v = make_qkv(wl(seed, dtype, d), "cuda")
        Q.copy_(q)
        K.copy_(k)
        V.copy_(v)
        graph.replay()
        rKc, rVc = api.cca_pool(q, k, v, g)
        rO, rL = api.cca_attn_fwd(q, k, v, rKc, rVc, g, w)
        torch.cuda.synchronize()
        assert torch.equal(Kc, rKc) and torch.equal(Vc, rVc), seed
        assert torch.equal(O, rO) and torch.equal(LSE, rL), seed


def test_decode_step_replays_bitwise():
    g, w = 16, 300
    Q, K, V = make_qkv(wl(21), "cuda")
    Kc, Vc = api.cca_pool(Q, K, V, g)
    pos = Q.shape[2] - 1  # completes group pos // g
    j = pos // g
    q = Q[:, :, pos].contiguous()
    ws = torch.empty(4 << 20, dtype=torch.uint8, device="cuda")
    O, LSE = api.cca_decode_fwd(q, K, V, Kc, Vc, pos, g, w, workspace=ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        api.cca_decode_fwd(q, K, V, Kc, Vc, pos, g, w, O=O, LSE=LSE, workspace=ws)
        api.cca_pool_group(q, K, V, Kc, Vc, j, g)
    for src in (pos - 5, pos - 700):
        q.copy_(Q[:, :, src])
        graph.replay()
        rKc, rVc = Kc.clone(), Vc.clone()
        torch.cuda.synchronize()
        # eager: the same decode (it does not read group j) and the same pooling
        eKc, eVc = api.cca_pool(Q, K, V, g)
        rO, rL = api.cca_decode_fwd(q, K, V, eKc, eVc, pos, g, w)
        api.cca_pool_group(q, K, V, eKc, eVc, j, g)
        torch.cuda.synchronize()
        assert torch.equal(O, rO) and torch.equal(LSE, rL), src
        assert torch.equal(rKc, eKc) and torch.equal(rVc, eVc), src


def test_noalloc_decode_replays_bitwise():
    lib = api.load_library()
    g, w = 16, 300
    Q, K, V = make_qkv(wl(31), "cuda")
    Kc, Vc = api.cca_pool(Q, K, V, g)
    pos = 1000
    q = Q[:, :, pos].contiguous()
    B, Hq, d = q.shape
    prm = api.make_params(B, Hq, K.shape[1], K.shape[2], d, g, w, api.CCA_BF16)
    O = torch.empty_like(q)
    LSE = torch.empty((B, Hq), dtype=torch.float32, device="cuda")

    def call(stream):
        st = lib.cca_decode_fwd_noalloc(q.data_ptr(), K.data_ptr(), V.data_ptr(), Kc.data_ptr(), Vc.data_ptr(),
                                        O.data_ptr(), LSE.data_ptr(), pos, ctypes.byref(prm), stream)
        assert st == api.CCA_OK, api.status_string(st)

    call(torch.cuda.current_stream().cuda_stream)  # first call on the device: before any capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(torch.cuda.current_stream().cuda_stream)
    q.copy_(Q[:, :, pos - 1])
    graph.replay()
    gO, gL = O.clone(), LSE.clone()
    torch.cuda.synchronize()
    rO, rL = api.cca_decode_fwd(q, K, V, Kc, Vc, pos, g, w)
    torch.cuda.synchronize()
    assert torch.equal(gO, rO) and torch.equal(gL, rL)
