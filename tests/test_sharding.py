"""Sequence sharding of CCA prefill on CPU ranks (gloo): each rank pools its own groups,
the ranks all-gather the core tokens and send each other the window halos, each rank
attends its own rows, and the result equals the unsharded oracle bit for bit.  The
oracle computes every per-rank step; the module under test only plans and moves rows."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from sparse_long_context_cca_gb300 import sharding
from sparse_long_context_cca_gb300.workloads import Workload


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


CASES = [  # (B, Hq, Hkv, N, d, g, w, window_mode, world)
    (1, 2, 2, 96, 8, 4, 9, 0, 2),
    (1, 4, 2, 120, 8, 3, 50, 0, 3),     # halo wider than a shard: rows from two earlier ranks
    (2, 2, 1, 64, 8, 8, 20, 1, 2),      # group-aligned window
    (1, 2, 2, 80, 8, 16, 200, 0, 3),    # window wider than N: every row is pure causal attention
    (1, 2, 2, 48, 8, 4, 5, 0, 5),       # 12 groups over 5 ranks: uneven shards
]


def _worker(rank, world, port, case, halo_bug, q):
    import oracle
    from sparse_long_context_cca_gb300.inputs import make_qkv
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, Hq, Hkv, N, d, g, w, wm, _ = case
        wl = Workload("shard", B, Hq, Hkv, N, d, g, w, "f32", 77, 0.05)
        Qf, Kf, Vf = (t.double() for t in make_qkv(wl, "cpu"))   # each rank keeps only its shard
        shards = sharding.plan(N, g, w, world, wm)
        if halo_bug:
            # a planted mistake: one window row short for every rank that needs a halo
            shards = [sharding.Shard(s.rank, s.q0, s.q1, min(s.halo0 + 1, s.q0), s.n_cores) for s in shards]
        me = shards[rank]
        Q, K, V = (t[:, :, me.q0:me.q1].contiguous() for t in (Qf, Kf, Vf))
        # 1. pool this rank's own groups (group-local)
        if me.q1 > me.q0:
            kc, vc = (torch.from_numpy(x) for x in oracle.pool(Q, K, V, g, pool_mode=0))
        else:
            kc = vc = torch.zeros((B, Hkv, 0, d), dtype=torch.float64)
        # 2. the exchange: all-gather the core tokens, window halos point to point
        Kc, Vc = sharding.gather_cores(kc, vc, shards, g)
        kw, vw = sharding.exchange_halo(K, V, shards)
        # 3. attend this rank's rows: the raw rows it holds sit at their global positions
        #    (rows outside [halo0, q1) stay zero, so a halo that is too short shows)
        Kg = torch.zeros((B, Hkv, N, d), dtype=torch.float64)
        Vg = torch.zeros_like(Kg)
        Kg[:, :, me.halo0:me.q1] = kw
        Vg[:, :, me.halo0:me.q1] = vw
        Qg = torch.zeros((B, Hq, N, d), dtype=torch.float64)
        Qg[:, :, me.q0:me.q1] = Q
        rows = [(b, h, i) for b in range(B) for h in range(Hq) for i in range(me.q0, me.q1)]
        if rows:
            O, L = oracle.attn_rows(Qg, Kg, Vg, Kc, Vc, g, w, rows, window_mode=wm)
        else:
            O, L = np.zeros((0, d)), np.zeros((0,))
        q.put((rank, rows, O, L, Kc.numpy()))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def _run(case, halo_bug=False):
    world = case[-1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, case, halo_bug, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return out


def _reference(case):
    import oracle
    from sparse_long_context_cca_gb300.inputs import make_qkv
    B, Hq, Hkv, N, d, g, w, wm, _ = case
    wl = Workload("shard", B, Hq, Hkv, N, d, g, w, "f32", 77, 0.05)
    Q, K, V = make_qkv(wl, "cpu")
    return oracle.prefill(Q, K, V, g, w, window_mode=wm)


def test_plan_covers_the_sequence_and_the_windows():
    for N, g, w, wm, world in [(96, 4, 9, 0, 2), (120, 3, 50, 0, 3), (64, 8, 20, 1, 2), (48, 4, 5, 0, 5),
                               (4096, 16, 1024, 0, 8), (4096, 512, 4, 1, 3), (32, 16, 8, 0, 4)]:
        shards = sharding.plan(N, g, w, world, wm)
        assert [s.rank for s in shards] == list(range(world))
        assert shards[0].q0 == 0 and shards[-1].q1 == N
        for a, b in zip(shards, shards[1:]):
            assert a.q1 == b.q0
        for s in shards:
            assert s.q0 % g == 0 and s.q1 % g == 0
            for i in range(s.q0, s.q1):
                assert sharding.window_start(i, w, g, wm) >= s.halo0       # every window row is at hand
                assert sharding.window_lo(i, w) // g <= s.n_cores          # every visible core is gathered
        # the halo transfers cover exactly [halo0, q0) of every rank, once
        sends = sharding.halo_sends(shards)
        for s in shards:
            got = sorted((a, b) for src, dst, a, b in sends if dst == s.rank)
            covered = [x for a, b in got for x in range(a, b)]
            assert covered == list(range(s.halo0, s.q0))


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}Hq{}Hkv{}N{}d{}g{}w{}m{}x{}".format(*c))
def test_sharded_prefill_equals_the_unsharded_oracle(case):
    out = _run(case)
    O_ref, L_ref, Kc_ref, _ = _reference(case)
    for rank, rows, O, L, Kc in out:
        np.testing.assert_array_equal(Kc, Kc_ref)
        for n, (b, h, i) in enumerate(rows):
            np.testing.assert_array_equal(O[n], O_ref[b, h, i])
            assert L[n] == L_ref[b, h, i]


def test_a_short_halo_is_caught():
    case = (1, 2, 2, 96, 8, 4, 9, 0, 2)
    out = _run(case, halo_bug=True)
    O_ref, _, _, _ = _reference(case)
    diffs = [np.abs(O[n] - O_ref[b, h, i]).max() for _, rows, O, _, _ in out for n, (b, h, i) in enumerate(rows)]
    assert max(diffs) > 1e-6


def _oracle_kernels(api):
    """CPU stand-ins for the two library calls shard_prefill makes, written from their ABI
    definitions with the oracle (test infrastructure: the GPU test runs the real kernels)."""
    import oracle

    def cca_pool(Q, K, V, g, scale=0.0, pool_mode=0, **_):
        kc, vc = oracle.pool(Q, K, V, g, pool_mode=pool_mode)
        return torch.from_numpy(kc), torch.from_numpy(vc)

    def cca_attn_fwd_rows(Q, K, V, Kc, Vc, g, w, N, q_off, kv_off, scale=0.0, window_mode=0, **_):
        B, Hq, n_q, d = Q.shape
        Hkv, n_kv = K.shape[1], K.shape[2]
        # rows and raw tokens at their sequence positions; the rest stays zero, so a call that
        # reached outside what it was given would show
        Qg = torch.zeros((B, Hq, N, d), dtype=torch.float64)
        Kg = torch.zeros((B, Hkv, N, d), dtype=torch.float64)
        Vg = torch.zeros_like(Kg)
        Qg[:, :, q_off:q_off + n_q] = Q
        Kg[:, :, kv_off:kv_off + n_kv] = K
        Vg[:, :, kv_off:kv_off + n_kv] = V
        rows = [(b, h, i) for b in range(B) for h in range(Hq) for i in range(q_off, q_off + n_q)]
        O, L = oracle.attn_rows(Qg, Kg, Vg, Kc, Vc, g, w, rows, window_mode=window_mode)
        return (torch.from_numpy(O).reshape(B, Hq, n_q, d), torch.from_numpy(L).reshape(B, Hq, n_q))

    api.cca_pool = cca_pool
    api.cca_attn_fwd_rows = cca_attn_fwd_rows


def _shard_prefill_worker(rank, world, port, case, q):
    from sparse_long_context_cca_gb300 import api
    from sparse_long_context_cca_gb300.inputs import make_qkv
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        _oracle_kernels(api)
        B, Hq, Hkv, N, d, g, w, wm, _ = case
        wl = Workload("shard", B, Hq, Hkv, N, d, g, w, "f32", 77, 0.05)
        Qf, Kf, Vf = (t.double() for t in make_qkv(wl, "cpu"))
        shards = sharding.plan(N, g, w, world, wm)
        me = shards[rank]
        Q, K, V = (t[:, :, me.q0:me.q1].contiguous() for t in (Qf, Kf, Vf))
        O, L, _, _ = sharding.shard_prefill(Q, K, V, shards, g, w, N, window_mode=wm)
        q.put((rank, me.q0, O.numpy(), L.numpy()))
    finally:
        dist.barrier()
        dist.destroy_process_group()


@pytest.mark.parametrize("case", [CASES[1], CASES[2]], ids=lambda c: "B{}Hq{}Hkv{}N{}d{}g{}w{}m{}x{}".format(*c))
def test_shard_prefill_wiring(case):
    """sharding.shard_prefill itself (pool its groups, gather, exchange, attend its rows with
    the right offsets), with the two library calls replaced by their oracle definitions."""
    world = case[-1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_prefill_worker, args=(r, world, port, case, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    O_ref, L_ref, _, _ = _reference(case)
    for rank, q0, O, L in out:
        n = O.shape[2]
        np.testing.assert_array_equal(O, O_ref[:, :, q0:q0 + n])
        np.testing.assert_array_equal(L, L_ref[:, :, q0:q0 + n])
