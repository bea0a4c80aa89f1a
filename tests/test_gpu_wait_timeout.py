"""The bf16 attention kernel's bounded waits: when a pipeline wait runs out
(here because a test hook makes the producer skip the query-tile load, a flag
that nothing else sets), every CTA stops, drains what it issued, frees its
tensor memory and writes CCA_ERR_TIMEOUT to the caller's status word; the
context stays usable and the next normal call is correct."""
import pytest
import torch

import oracle
from parity import check_out
from sparse_long_context_cca_gb300 import api
from sparse_long_context_cca_gb300.inputs import make_qkv
from sparse_long_context_cca_gb300.workloads import Workload

pytestmark = pytest.mark.gpu


def test_wait_timeout_reports_status_and_recovers():
    lib = api.load_library()
    w = Workload("timeout B1 H2 d128 N512 g16 w64", 1, 2, 2, 512, 128, 16, 64, "bf16", 3, 0.01)
    Q, K, V = make_qkv(w, "cuda")
    Kc, Vc = api.cca_pool(Q, K, V, w.g)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.cca_test_set_wait_limit_ns(20_000_000)   # 20 ms per wait
    lib.cca_test_skip_q_load(1)
    try:
        api.cca_attn_fwd(Q, K, V, Kc, Vc, w.g, w.w, dev_status=st)
        torch.cuda.synchronize()
    finally:
        lib.cca_test_skip_q_load(0)
        lib.cca_test_set_wait_limit_ns(1_000_000_000)
    assert int(st.item()) == api.CCA_ERR_TIMEOUT
    st.zero_()
    O, LSE = api.cca_attn_fwd(Q, K, V, Kc, Vc, w.g, w.w, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Or, Lr = oracle.attn(Q, K, V, Kc, Vc, w.g, w.w)
    check_out(O, LSE, Or, Lr, Q.dtype, "after time-out")


def test_backward_wait_timeout_reports_status_and_recovers():
    """The tensor-core backward kernels stop the same way: with no copies issued their
    first wait runs out, each CTA frees its tensor memory and reports CCA_ERR_TIMEOUT,
    and the next normal call matches the fp64 backward oracle."""
    import numpy as np
    from oracle.backward import prefill_grads
    lib = api.load_library()
    w = Workload("bwd timeout B1 H2 d128 N384 g16 w64", 1, 2, 2, 384, 128, 16, 64, "bf16", 4, 0.01)
    Q, K, V = make_qkv(w, "cuda")
    gen = torch.Generator(device="cuda").manual_seed(9)
    dO = torch.randn(Q.shape, generator=gen, device="cuda").to(Q.dtype)
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.cca_test_set_wait_limit_ns(20_000_000)
    lib.cca_test_skip_q_load(1)
    try:
        api.cca_prefill_bwd(Q, K, V, Kc, Vc, O, LSE, dO, w.g, w.w, dev_status=st)
        torch.cuda.synchronize()
    finally:
        lib.cca_test_skip_q_load(0)
        lib.cca_test_set_wait_limit_ns(1_000_000_000)
    assert int(st.item()) == api.CCA_ERR_TIMEOUT
    st.zero_()
    dQ, dK, dV = api.cca_prefill_bwd(Q, K, V, Kc, Vc, O, LSE, dO, w.g, w.w, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rQ, rK, rV = prefill_grads(Q, K, V, dO, w.g, w.w)
    for name, got, ref in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV)):
        err = np.abs(got.double().cpu().numpy() - ref)
        assert err.max() <= 2e-2 * np.abs(ref).max(), (name, err.max())
