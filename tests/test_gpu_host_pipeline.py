"""cca_prefill_host: the prefill step on host buffers, pipelined over slices of
(batch, KV head) pairs.  Checked against the fp64 oracle, and bit for bit against
the device-buffer path (each slice is the same computation on the same values)."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from parity import check_cores, check_out
from sparse_long_context_cca_gb300 import api
from sparse_long_context_cca_gb300.inputs import make_qkv
from sparse_long_context_cca_gb300.workloads import MHA_32K, Workload

pytestmark = pytest.mark.gpu


def wl(B, Hq, Hkv, N, d, g, w, dtype="bf16", seed=41):
    return Workload(f"host B{B} Hq{Hq} Hkv{Hkv} N{N} d{d} g{g} w{w} {dtype}", B, Hq, Hkv, N, d, g, w, dtype,
                    seed, 0.01)


CASES = [
    # 6 pairs -> 6 slices over 3 buffers (each buffer reused), GQA r = 2, ragged tile
    (wl(2, 6, 3, 400, 128, 16, 100), 0, 0),
    # 16 pairs -> slices of 2, modes on
    (wl(2, 8, 8, 256, 128, 8, 40), 1, 1),
    # one pair: a single slice
    (wl(1, 4, 1, 512, 128, 32, 64), 2, 0),
    # fp32 path
    (wl(1, 4, 4, 256, 64, 16, 32, "f32"), 0, 0),
]


@pytest.mark.parametrize("w,pool_mode,window_mode", CASES, ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_host_pipeline_matches_oracle_and_device_path(w, pool_mode, window_mode):
    Q, K, V = make_qkv(w, "cpu")
    hQ, hK, hV = (t.pin_memory() for t in (Q, K, V))
    O, LSE, Kc, Vc = api.cca_prefill_host(hQ, hK, hV, w.g, w.w, with_cores=True, pool_mode=pool_mode,
                                          window_mode=window_mode)
    torch.cuda.current_stream().synchronize()
    dQ, dK, dV = (t.cuda() for t in (Q, K, V))
    Od, Ld, Kcd, Vcd = api.cca_prefill(dQ, dK, dV, w.g, w.w, pool_mode=pool_mode, window_mode=window_mode)
    torch.cuda.synchronize()
    for name, a, b in (("O", O, Od), ("LSE", LSE, Ld), ("Kc", Kc, Kcd), ("Vc", Vc, Vcd)):
        assert torch.equal(a, b.cpu()), name
    Oref, Lref, Kref, Vref = oracle.prefill(Q, K, V, w.g, w.w, pool_mode=pool_mode, window_mode=window_mode)
    check_out(O, LSE, Oref, Lref, Q.dtype, w.name)
    check_cores(Kc, Vc, Kref, Vref, Q.dtype, w.name)


def test_host_pipeline_pageable_memory_and_reuse():
    """Pageable host buffers work (staged by the driver); a second call with other
    inputs on the same workspace gives that input's result."""
    w = wl(1, 8, 8, 384, 128, 16, 50)
    ws = torch.empty(api.prefill_host_workspace_size(1, 8, 8, 384, 128, 16, 50, torch.bfloat16), dtype=torch.uint8,
                     device="cuda")
    outs = []
    for seed in (3, 4):
        Q, K, V = make_qkv(replace(w, seed=seed), "cpu")
        O, LSE, _, _ = api.cca_prefill_host(Q, K, V, w.g, w.w, workspace=ws)
        torch.cuda.current_stream().synchronize()
        Od, Ld, _, _ = api.cca_prefill(Q.cuda(), K.cuda(), V.cuda(), w.g, w.w)
        torch.cuda.synchronize()
        assert torch.equal(O, Od.cpu()) and torch.equal(LSE, Ld.cpu()), seed
        outs.append(O)
    assert not torch.equal(outs[0], outs[1])


def test_host_pipeline_full_size_32k():
    """The 32K MHA workload through the host entry point equals the device path bit for bit."""
    w = MHA_32K
    Qd, Kd, Vd = make_qkv(w, "cuda")
    hQ, hK, hV = (t.cpu().pin_memory() for t in (Qd, Kd, Vd))
    O, LSE, _, _ = api.cca_prefill_host(hQ, hK, hV, w.g, w.w)
    torch.cuda.current_stream().synchronize()
    Od, Ld, _, _ = api.cca_prefill(Qd, Kd, Vd, w.g, w.w)
    torch.cuda.synchronize()
    assert torch.equal(O, Od.cpu())
    assert torch.equal(LSE, Ld.cpu())
    # sampled rows of two heads against the oracle (MHA: KV head h serves query head h)
    rng = np.random.default_rng(7)
    for h in (0, 29):
        q, k, v = hQ[:, h:h + 1], hK[:, h:h + 1], hV[:, h:h + 1]
        Kr, Vr = oracle.pool(q, k, v, w.g)
        rows = sorted({0, w.w - 1, w.w + w.g - 1, w.N - 1} | set(rng.integers(0, w.N, 28).tolist()))
        Oref, Lref = oracle.attn_rows(q, k, v, Kr, Vr, w.g, w.w, [(0, 0, i) for i in rows])
        check_out(O[0, h, rows], LSE[0, h, rows], Oref, Lref, torch.bfloat16, f"32K head {h}")
