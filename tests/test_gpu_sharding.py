"""A sequence split across ranks along its length, on the GPU: every shard pools its own
whole groups, the shards' core tokens are put together, and each shard's rows are attended
with cca_attn_fwd_rows from those cores and the raw rows its windows reach back to (its
halo).  The shards run one after another in this process, exchanging by slicing; the
exchange itself (all-gather, point-to-point halo) is tested on CPU ranks.  Checked against
the unsharded prefill and the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from parity import check_out
from sparse_long_context_cca_gb300 import api, sharding
from sparse_long_context_cca_gb300.inputs import make_qkv
from sparse_long_context_cca_gb300.workloads import Workload

pytestmark = pytest.mark.gpu


def wl(B, Hq, Hkv, N, d, g, w, dtype="bf16", seed=83):
    return Workload(f"shard B{B} Hq{Hq} Hkv{Hkv} N{N} d{d} g{g} w{w} {dtype}", B, Hq, Hkv, N, d, g, w, dtype,
                    seed, 0.01)


CASES = [
    (wl(1, 4, 2, 2048, 128, 16, 300), 3, 0),            # GQA; shard edges on groups, not on 256 rows
    (wl(1, 2, 2, 3072, 128, 16, 1024), 3, 0),           # shards of 1024 rows: same items as unsharded
    (wl(2, 2, 2, 1600, 128, 32, 200), 4, 1),            # group-aligned window
    (wl(1, 4, 4, 1000, 128, 8, 100), 5, 0),             # 125 groups over 5 ranks, ragged last item
    (wl(1, 2, 2, 4096, 128, 16, 4096), 2, 0),           # window wider than a shard: halo from rank 0
    (wl(1, 2, 1, 768, 64, 16, 90, "f32"), 3, 0),        # fp32, d = 64
    (wl(1, 2, 2, 640, 128, 16, 64, "f32"), 2, 1),       # fp32, group-aligned window
]


def _slice(t, a, b):
    return t[:, :, a:b].contiguous()


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name} x{c[1]} m{c[2]}")
def test_shards_equal_unsharded(case):
    w, world, window_mode = case
    Q, K, V = make_qkv(w, "cuda")
    shards = [s for s in sharding.plan(w.N, w.g, w.w, world, window_mode) if s.q1 > s.q0]
    # pooling is group-local: each shard pools its own groups
    parts = [api.cca_pool(_slice(Q, s.q0, s.q1), _slice(K, s.q0, s.q1), _slice(V, s.q0, s.q1), w.g)
             for s in shards]
    Kc = torch.cat([p[0] for p in parts], dim=2)
    Vc = torch.cat([p[1] for p in parts], dim=2)
    Ou, Lu, Kcu, Vcu = api.cca_prefill(Q, K, V, w.g, w.w, window_mode=window_mode)
    torch.cuda.synchronize()
    assert torch.equal(Kc, Kcu) and torch.equal(Vc, Vcu)
    rng = np.random.default_rng(w.seed)
    for s in shards:
        O, L = api.cca_attn_fwd_rows(_slice(Q, s.q0, s.q1), _slice(K, s.halo0, s.q1), _slice(V, s.halo0, s.q1),
                                     Kc, Vc, w.g, w.w, w.N, s.q0, s.halo0, window_mode=window_mode)
        torch.cuda.synchronize()
        ref_O, ref_L = Ou[:, :, s.q0:s.q1], Lu[:, :, s.q0:s.q1]
        if s.q0 % 256 == 0:
            # the shard's work items are the unsharded launch's: the same arithmetic
            assert torch.equal(O, ref_O) and torch.equal(L, ref_L), s
        else:
            check_out(O, L, oracle.widen(ref_O), oracle.widen(ref_L), Q.dtype, f"{w.name} shard {s.rank} vs unsharded")
        # sampled rows against the fp64 oracle (the GPU's own cores)
        rows = sorted({s.q0, s.q1 - 1, min(s.q0 + w.w, s.q1 - 1)} | set(rng.integers(s.q0, s.q1, 12).tolist()))
        sel = [(b, h, i) for b in range(w.B) for h in range(w.Hq) for i in rows]
        Oa, La = oracle.attn_rows(Q, K, V, Kc, Vc, w.g, w.w, sel, window_mode=window_mode)
        got_O = torch.stack([O[b, h, i - s.q0] for b, h, i in sel])
        got_L = torch.stack([L[b, h, i - s.q0] for b, h, i in sel])
        check_out(got_O, got_L, Oa, La, Q.dtype, f"{w.name} shard {s.rank} vs oracle")


def test_rows_of_a_window_inside_one_tile():
    """A single row, and rows whose halo starts inside their first key tile; K/V holding
    exactly the rows' windows, or the whole sequence."""
    w = wl(1, 2, 2, 1024, 128, 16, 200)
    Q, K, V = make_qkv(w, "cuda")
    Ou, Lu, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w)
    for q0, n in ((517, 1), (300, 77), (1023, 1)):
        # the exact halo, and K/V from the sequence start through its end (more than needed)
        for kv0, kv1 in ((max(0, q0 - w.w + 1), q0 + n), (0, w.N)):
            O, L = api.cca_attn_fwd_rows(_slice(Q, q0, q0 + n), _slice(K, kv0, kv1), _slice(V, kv0, kv1),
                                         Kc, Vc, w.g, w.w, w.N, q0, kv0)
            torch.cuda.synchronize()
            check_out(O, L, oracle.widen(Ou[:, :, q0:q0 + n]), oracle.widen(Lu[:, :, q0:q0 + n]), Q.dtype,
                      f"rows {q0}+{n}, K/V [{kv0}, {kv1})")
