"""Pins of the CPU oracle to facts fixed outside it.

Each ``pin_*`` function takes an oracle library handle (``oracle.load()`` or a
deliberately broken build of it) and raises AssertionError when the oracle
disagrees with:
  * the hand-worked example in ``golden/worked_example.json``;
  * the hand-derived visible-key counts in ``golden/visibility_counts.json``;
  * closed forms: with g = 1, or with w >= N, CCA is exactly causal softmax
    attention, checked against torch's own scaled_dot_product_attention;
  * special cases of the pooling: equal keys or a zero query give mean
    pooling, a dominant query selects the matching key;
  * invariants: weights sum to one, causality, rows before the first visible
    core are plain sliding-window attention.
None of these re-types the oracle's loops.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _sdpa(Q, K, V, mask=None, causal=False):
    """Reference attention from torch (fp64 CPU), query head h reading KV head h // r."""
    q, k, v = (torch.from_numpy(np.ascontiguousarray(t)) for t in (Q, K, V))
    r = q.shape[1] // k.shape[1]
    k = k.repeat_interleave(r, dim=1)
    v = v.repeat_interleave(r, dim=1)
    if causal:
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
        N = q.shape[2]
        mask = torch.ones(N, N, dtype=torch.bool).tril()
    else:
        mask = torch.from_numpy(mask)
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask)
    logits = (q @ k.transpose(-1, -2)) / math.sqrt(q.shape[-1])
    lse = torch.logsumexp(logits.masked_fill(~mask, float("-inf")), dim=-1)
    return o.numpy(), lse.numpy()


def pin_worked_example(lib):
    ex = _golden("worked_example.json")
    Q = np.array(ex["Q"], dtype=np.float64)[None, None]
    K = np.array(ex["K"], dtype=np.float64)[None, None]
    V = np.array(ex["V"], dtype=np.float64)[None, None]
    g = ex["shape"]["g"]
    Kc, Vc = oracle.pool(Q, K, V, g, lib=lib)
    np.testing.assert_allclose(Kc[0, 0], np.array(ex["pool"]["Kc"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(Vc[0, 0], np.array(ex["pool"]["Vc"]), rtol=0, atol=1e-12)
    for case in ex["attn"]:
        O, LSE = oracle.attn(Q, K, V, Kc, Vc, g, case["w"], lib=lib)
        rows = case.get("rows", list(range(Q.shape[2])))
        np.testing.assert_allclose(O[0, 0, rows], np.array(case["O"]), rtol=0, atol=1e-12)
        np.testing.assert_allclose(LSE[0, 0, rows], np.array(case["LSE"]), rtol=0, atol=1e-12)


def pin_gqa_worked_example(lib):
    ex = _golden("worked_example.json")
    gq = ex["gqa"]
    K = np.array(ex["K"], dtype=np.float64)[None, None]
    V = np.array(ex["V"], dtype=np.float64)[None, None]
    Q = np.zeros((1, 2, 4, 4))
    Q[0, :, 1] = np.array(gq["Q_heads_row1"])
    Kc, Vc = oracle.pool(Q, K, V, 2, lib=lib)
    np.testing.assert_allclose(Kc[0, 0, 0], gq["Kc0"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(Vc[0, 0, 0], gq["Vc0"], rtol=0, atol=1e-12)
    # the alternative GQA pooling: per-head softmax weights averaged after the softmax
    pm = gq["post_softmax_mean"]
    Kc, Vc = oracle.pool(Q, K, V, 2, lib=lib, pool_mode=3)
    for j in (0, 1):
        np.testing.assert_allclose(Kc[0, 0, j], pm["Kc%d" % j], rtol=0, atol=1e-12)
        np.testing.assert_allclose(Vc[0, 0, j], pm["Vc%d" % j], rtol=0, atol=1e-12)


def pin_post_softmax_gqa_pooling(lib):
    """pool_mode 3 against facts outside it: with one query head per KV head it is the
    method's pooling (the worked example's hand values, and pool_mode 0 on random
    inputs); with r heads it is the mean of r single-head poolings, each scored by one
    head's own query (head h of KV head kv is query head kv*r + h)."""
    ex = _golden("worked_example.json")
    Q = np.array(ex["Q"], dtype=np.float64)[None, None]
    K = np.array(ex["K"], dtype=np.float64)[None, None]
    V = np.array(ex["V"], dtype=np.float64)[None, None]
    Kc, Vc = oracle.pool(Q, K, V, ex["shape"]["g"], lib=lib, pool_mode=3)
    np.testing.assert_allclose(Kc[0, 0], np.array(ex["pool"]["Kc"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(Vc[0, 0], np.array(ex["pool"]["Vc"]), rtol=0, atol=1e-12)
    for (B, Hq, Hkv, N, d, g, seed) in [(1, 2, 2, 32, 8, 4, 80), (2, 4, 2, 36, 8, 3, 81),
                                         (1, 8, 2, 40, 16, 5, 82), (1, 4, 1, 24, 8, 1, 83)]:
        Q, K, V = _rand((B, Hq, N, d), seed, 2.0), _rand((B, Hkv, N, d), seed + 1), _rand((B, Hkv, N, d), seed + 2)
        Kc, Vc = oracle.pool(Q, K, V, g, lib=lib, pool_mode=3)
        r = Hq // Hkv
        if r == 1:
            Kc0, Vc0 = oracle.pool(Q, K, V, g, lib=lib, pool_mode=0)
            np.testing.assert_allclose(Kc, Kc0, rtol=0, atol=1e-12)
            np.testing.assert_allclose(Vc, Vc0, rtol=0, atol=1e-12)
            continue
        Km = np.zeros_like(Kc)
        Vm = np.zeros_like(Vc)
        for b in range(B):
            for kv in range(Hkv):
                for hh in range(r):
                    q1 = Q[b:b + 1, kv * r + hh:kv * r + hh + 1]
                    k1, v1 = K[b:b + 1, kv:kv + 1], V[b:b + 1, kv:kv + 1]
                    Kh, Vh = oracle.pool(q1, k1, v1, g, lib=lib, pool_mode=0)
                    Km[b, kv] += Kh[0, 0] / r
                    Vm[b, kv] += Vh[0, 0] / r
        np.testing.assert_allclose(Kc, Km, rtol=0, atol=1e-12)
        np.testing.assert_allclose(Vc, Vm, rtol=0, atol=1e-12)
        Kc0, _ = oracle.pool(Q, K, V, g, lib=lib, pool_mode=0)
        if g == 1:
            # a one-token group pools to its token whatever the weights
            np.testing.assert_array_equal(Kc, K)
            np.testing.assert_array_equal(Kc0, K)
        else:
            # and it is not the logit mean of pool_mode 0 (the heads' queries differ)
            assert np.abs(Kc - Kc0).max() > 1e-3


def pin_visibility_counts(lib):
    data = _golden("visibility_counts.json")
    for case in data["cases"]:
        N, g, w = case["N"], case["g"], case["w"]
        d = 2 if N > 4096 else 8
        Q = np.zeros((1, 1, N, d))
        K = _rand((1, 1, N, d), 1)
        V = _rand((1, 1, N, d), 2)
        Kc, Vc = oracle.pool(Q, K, V, g, lib=lib)
        rows = [(0, 0, i) for i, _, _ in case["rows"]]
        _, LSE = oracle.attn_rows(Q, K, V, Kc, Vc, g, w, rows, lib=lib)
        want = np.array([nc + nl for _, nc, nl in case["rows"]], dtype=np.float64)
        np.testing.assert_allclose(np.exp(LSE), want, rtol=1e-12, atol=0)


def pin_kv_cache_count(lib=None):
    kv = _golden("visibility_counts.json")["kv_cache"]
    per_token = kv["layers"] * 2 * kv["hidden"] * kv["bytes_per_elem"]
    full = kv["N"] * per_token / 2**30
    cca = (kv["N"] // kv["g"] + kv["w"]) * per_token / 2**30
    assert abs(full - kv["full_GiB"]) < 1e-9 and abs(cca - kv["cca_GiB"]) < 1e-9, (full, cca)


def pin_g1_is_causal(lib):
    # g = 1: every token is its own core, so cores [0, lo) + window [lo, i] = all of [0, i].
    for (B, Hq, Hkv, N, d, w, seed) in [(1, 2, 2, 37, 8, 1, 0), (2, 4, 2, 50, 16, 7, 1),
                                         (1, 2, 1, 64, 8, 64, 2)]:
        Q, K, V = _rand((B, Hq, N, d), seed), _rand((B, Hkv, N, d), seed + 10), _rand((B, Hkv, N, d), seed + 20)
        O, LSE, Kc, Vc = oracle.prefill(Q, K, V, 1, w, lib=lib)
        Oref, Lref = _sdpa(Q, K, V, causal=True)
        np.testing.assert_allclose(O, Oref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(LSE, Lref, rtol=0, atol=1e-12)


def pin_wide_window_is_causal(lib):
    # w >= N: lo(i) = 0 for every row, so no core is visible.
    for (N, g, w, seed) in [(48, 4, 48, 3), (48, 8, 100, 4), (60, 2, 61, 5)]:
        Q, K, V = _rand((1, 2, N, 8), seed), _rand((1, 2, N, 8), seed + 1), _rand((1, 2, N, 8), seed + 2)
        O, LSE, _, _ = oracle.prefill(Q, K, V, g, w, lib=lib)
        Oref, Lref = _sdpa(Q, K, V, causal=True)
        np.testing.assert_allclose(O, Oref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(LSE, Lref, rtol=0, atol=1e-12)


def pin_early_rows_are_sliding_window(lib):
    # Rows i < w + g - 1 see no core, only the band [i-w+1, i].
    N, g, w, d = 64, 4, 9, 8
    Q, K, V = _rand((1, 2, N, d), 6), _rand((1, 2, N, d), 7), _rand((1, 2, N, d), 8)
    O, LSE, _, _ = oracle.prefill(Q, K, V, g, w, lib=lib)
    i = np.arange(N)[:, None]
    m = np.arange(N)[None, :]
    band = (m <= i) & (m >= i - w + 1)
    Oref, Lref = _sdpa(Q, K, V, mask=band)
    n = w + g - 1
    np.testing.assert_allclose(O[:, :, :n], Oref[:, :, :n], rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE[:, :, :n], Lref[:, :, :n], rtol=0, atol=1e-12)
    # later rows see cores, so they must differ from the band-only answer
    assert np.abs(O[:, :, n:] - Oref[:, :, n:]).max() > 1e-3


def pin_pool_equal_keys_mean(lib):
    B, H, N, d, g = 1, 2, 32, 8, 4
    Q = _rand((B, H, N, d), 9)
    Kg = _rand((B, H, N // g, 1, d), 10)
    K = np.repeat(Kg, g, axis=3).reshape(B, H, N, d)
    V = _rand((B, H, N, d), 11)
    Kc, Vc = oracle.pool(Q, K, V, g, lib=lib)
    np.testing.assert_allclose(Kc, Kg[:, :, :, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(Vc, V.reshape(B, H, N // g, g, d).mean(axis=3), rtol=0, atol=1e-12)


def pin_pool_zero_query_mean(lib):
    B, H, N, d, g = 1, 2, 40, 8, 5
    Q = _rand((B, H, N, d), 12)
    Q[:, :, g - 1::g] = 0.0      # only the groups' last queries score the group
    K, V = _rand((B, H, N, d), 13), _rand((B, H, N, d), 14)
    Kc, Vc = oracle.pool(Q, K, V, g, lib=lib)
    np.testing.assert_allclose(Kc, K.reshape(B, H, N // g, g, d).mean(axis=3), rtol=0, atol=1e-12)
    np.testing.assert_allclose(Vc, V.reshape(B, H, N // g, g, d).mean(axis=3), rtol=0, atol=1e-12)


def pin_pool_dominant_query_selects(lib):
    B, H, N, d, g = 1, 1, 32, 16, 8
    rng = np.random.default_rng(15)
    K = rng.standard_normal((B, H, N, d))
    K /= np.linalg.norm(K, axis=-1, keepdims=True)   # unit keys: q.k is maximal at the aligned key
    V = rng.standard_normal((B, H, N, d))
    Q = rng.standard_normal((B, H, N, d))
    pick = rng.integers(0, g, size=N // g)
    for j in range(N // g):
        Q[0, 0, (j + 1) * g - 1] = 4000.0 * K[0, 0, j * g + pick[j]]
    Kc, Vc = oracle.pool(Q, K, V, g, lib=lib)
    for j in range(N // g):
        np.testing.assert_allclose(Kc[0, 0, j], K[0, 0, j * g + pick[j]], rtol=0, atol=1e-9)
        np.testing.assert_allclose(Vc[0, 0, j], V[0, 0, j * g + pick[j]], rtol=0, atol=1e-9)


def pin_unit_values(lib):
    # V = 1 everywhere: the pooled values are 1 and every output row is 1.
    B, Hq, Hkv, N, d, g, w = 2, 4, 2, 48, 8, 4, 6
    Q, K = _rand((B, Hq, N, d), 16, 2.0), _rand((B, Hkv, N, d), 17, 2.0)
    V = np.ones((B, Hkv, N, d))
    O, LSE, Kc, Vc = oracle.prefill(Q, K, V, g, w, lib=lib)
    np.testing.assert_allclose(Vc, 1.0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(O, 1.0, rtol=0, atol=1e-13)


def pin_constant_keys_lse(lib):
    # Every key equal to u: all logits of row i equal tau*q_i.u, so
    # LSE_i = tau*q_i.u + ln(count_i) and the output is the plain mean.
    N, g, w, d = 64, 4, 5, 8
    u = _rand((d,), 18)
    Q = _rand((1, 1, N, d), 19)
    K = np.broadcast_to(u, (1, 1, N, d)).copy()
    V = _rand((1, 1, N, d), 20)
    O, LSE, Kc, Vc = oracle.prefill(Q, K, V, g, w, lib=lib)
    counts = _golden("visibility_counts.json")["cases"][1]
    assert (counts["N"], counts["g"], counts["w"]) == (N, g, w)
    for i, nc, nl in counts["rows"]:
        want = Q[0, 0, i] @ u / math.sqrt(d) + math.log(nc + nl)
        assert abs(LSE[0, 0, i] - want) < 1e-12, (i, LSE[0, 0, i], want)


def pin_causality(lib):
    B, Hq, Hkv, N, d, g, w = 1, 2, 1, 64, 8, 4, 7
    Q, K, V = _rand((B, Hq, N, d), 21), _rand((B, Hkv, N, d), 22), _rand((B, Hkv, N, d), 23)
    O, LSE, _, _ = oracle.prefill(Q, K, V, g, w, lib=lib)
    for cut in (5, 20, 41, 63):
        Q2, K2, V2 = Q.copy(), K.copy(), V.copy()
        for t, s in ((Q2, 24), (K2, 25), (V2, 26)):
            t[:, :, cut + 1:] = _rand(t[:, :, cut + 1:].shape, s + cut, 3.0)
        O2, LSE2, _, _ = oracle.prefill(Q2, K2, V2, g, w, lib=lib)
        np.testing.assert_array_equal(O2[:, :, :cut + 1], O[:, :, :cut + 1])
        np.testing.assert_array_equal(LSE2[:, :, :cut + 1], LSE[:, :, :cut + 1])


def pin_dense_mask_formulation(lib):
    """A second formulation: pool with one dense softmax over a [groups, g] matrix,
    then one masked softmax over the concatenation [cores; all tokens]."""
    for (B, Hq, Hkv, N, d, g, w, seed) in [(1, 2, 2, 32, 8, 4, 3, 30), (2, 4, 2, 48, 8, 2, 8, 31),
                                            (1, 4, 1, 64, 16, 8, 20, 32), (1, 2, 2, 24, 8, 1, 1, 33)]:
        Q, K, V = _rand((B, Hq, N, d), seed), _rand((B, Hkv, N, d), seed + 1), _rand((B, Hkv, N, d), seed + 2)
        O, LSE, Kc, Vc = oracle.prefill(Q, K, V, g, w, lib=lib)
        r, G, tau = Hq // Hkv, N // g, 1 / math.sqrt(d)
        qlast = Q[:, :, g - 1::g].reshape(B, Hkv, r, G, d)
        Kg = K.reshape(B, Hkv, G, g, d)
        s = tau * np.einsum("bkrjc,bkjtc->bkjt", qlast, Kg) / r
        a = np.exp(s - s.max(-1, keepdims=True))
        a /= a.sum(-1, keepdims=True)
        Kc2 = np.einsum("bkjt,bkjtc->bkjc", a, Kg)
        Vc2 = np.einsum("bkjt,bkjtc->bkjc", a, V.reshape(B, Hkv, G, g, d))
        np.testing.assert_allclose(Kc, Kc2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(Vc, Vc2, rtol=0, atol=1e-12)
        i = np.arange(N)[:, None]
        lo = np.maximum(0, i - w + 1)
        core_mask = (np.arange(G)[None, :] + 1) * g <= lo
        tok = np.arange(N)[None, :]
        loc_mask = (tok >= lo) & (tok <= i)
        mask = np.concatenate([core_mask, loc_mask], axis=1)
        kv_head = np.arange(Hq) // r
        Kcat = np.concatenate([Kc2, K], axis=2)[:, kv_head]
        Vcat = np.concatenate([Vc2, V], axis=2)[:, kv_head]
        z = tau * np.einsum("bhic,bhmc->bhim", Q, Kcat)
        z = np.where(mask, z, -np.inf)
        zmax = z.max(-1, keepdims=True)
        p = np.exp(z - zmax)
        O2 = np.einsum("bhim,bhmc->bhic", p, Vcat) / p.sum(-1)[..., None]
        LSE2 = zmax[..., 0] + np.log(p.sum(-1))
        np.testing.assert_allclose(O, O2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(LSE, LSE2, rtol=0, atol=1e-12)


def pin_group_aligned_window_counts(lib):
    data = _golden("visibility_counts.json")["group_aligned_window"]
    for case in data["cases"]:
        N, g, w = case["N"], case["g"], case["w"]
        Q = np.zeros((1, 1, N, 8))
        K, V = _rand((1, 1, N, 8), 41), _rand((1, 1, N, 8), 42)
        Kc, Vc = oracle.pool(Q, K, V, g, lib=lib)
        rows = [(0, 0, i) for i, _, _ in case["rows"]]
        _, LSE = oracle.attn_rows(Q, K, V, Kc, Vc, g, w, rows, lib=lib, window_mode=1)
        want = np.array([nc + nl for _, nc, nl in case["rows"]], dtype=np.float64)
        np.testing.assert_allclose(np.exp(LSE), want, rtol=1e-12, atol=0)


def pin_group_aligned_window_no_gap(lib):
    # With g = 1 both windows coincide; with w >= N both are plain causal attention.
    N, d = 40, 8
    Q, K, V = _rand((1, 2, N, d), 43), _rand((1, 2, N, d), 44), _rand((1, 2, N, d), 45)
    for g, w in ((1, 6), (4, 64)):
        O0, L0, _, _ = oracle.prefill(Q, K, V, g, w, lib=lib)
        O1, L1, _, _ = oracle.prefill(Q, K, V, g, w, lib=lib, window_mode=1)
        np.testing.assert_allclose(O1, O0, rtol=0, atol=1e-13)
        np.testing.assert_allclose(L1, L0, rtol=0, atol=1e-13)


def pin_mean_pooling(lib):
    B, H, N, d, g = 1, 2, 40, 8, 5
    Q, K, V = _rand((B, H, N, d), 46, 3.0), _rand((B, H, N, d), 47), _rand((B, H, N, d), 48)
    Kc, Vc = oracle.pool(Q, K, V, g, lib=lib, pool_mode=1)
    np.testing.assert_allclose(Kc, K.reshape(B, H, N // g, g, d).mean(axis=3), rtol=0, atol=1e-12)
    np.testing.assert_allclose(Vc, V.reshape(B, H, N // g, g, d).mean(axis=3), rtol=0, atol=1e-12)


def pin_max_pooling(lib):
    B, H, N, d, g = 1, 2, 40, 8, 5
    Q, K, V = _rand((B, H, N, d), 49), _rand((B, H, N, d), 50), _rand((B, H, N, d), 51)
    Kc, Vc = oracle.pool(Q, K, V, g, lib=lib, pool_mode=2)
    np.testing.assert_array_equal(Kc, K.reshape(B, H, N // g, g, d).max(axis=3))
    np.testing.assert_array_equal(Vc, V.reshape(B, H, N // g, g, d).max(axis=3))


ALL_PINS = [pin_worked_example, pin_gqa_worked_example, pin_visibility_counts, pin_g1_is_causal,
            pin_wide_window_is_causal, pin_early_rows_are_sliding_window, pin_pool_equal_keys_mean,
            pin_pool_zero_query_mean, pin_pool_dominant_query_selects, pin_unit_values,
            pin_constant_keys_lse, pin_causality, pin_dense_mask_formulation,
            pin_group_aligned_window_counts, pin_group_aligned_window_no_gap, pin_mean_pooling, pin_max_pooling,
            pin_post_softmax_gqa_pooling]


def _fd_check(Q, K, V, g, w, pool_mode, window_mode, lib, n_probe=6, seed=0, eps=1e-6):
    """Central finite differences of sum(G * O) through the C oracle's forward, against
    the backward oracle's gradient, at a few random coordinates of Q, K and V."""
    from oracle.backward import prefill_grads
    rng = np.random.default_rng(seed)
    G = rng.standard_normal(Q.shape)
    dQ, dK, dV = prefill_grads(Q, K, V, G, g, w, pool_mode=pool_mode, window_mode=window_mode)
    for X, dX in ((Q, dQ), (K, dK), (V, dV)):
        for _ in range(n_probe):
            idx = tuple(rng.integers(0, s) for s in X.shape)
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            args_p = [Xp if X is T else T for T in (Q, K, V)]
            args_m = [Xm if X is T else T for T in (Q, K, V)]
            Op = oracle.prefill(*args_p, g, w, lib=lib, pool_mode=pool_mode, window_mode=window_mode)[0]
            Om = oracle.prefill(*args_m, g, w, lib=lib, pool_mode=pool_mode, window_mode=window_mode)[0]
            fd = ((Op - Om) * G).sum() / (2 * eps)
            assert abs(fd - dX[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, dX[idx])


def pin_backward_finite_differences(lib):
    B, Hq, Hkv, N, d = 1, 4, 2, 24, 8
    Q, K, V = _rand((B, Hq, N, d), 60), _rand((B, Hkv, N, d), 61), _rand((B, Hkv, N, d), 62)
    for g, w, pm, wm, seed in ((4, 5, 0, 0, 1), (3, 7, 0, 1, 2), (4, 6, 1, 0, 3), (2, 3, 2, 0, 4),
                               (4, 5, 3, 0, 5), (3, 4, 3, 1, 6)):
        _fd_check(Q, K, V, g, w, pm, wm, lib, seed=seed)


def pin_backward_g1_is_causal(lib):
    # g = 1: the forward is causal attention, so are its gradients (torch SDPA autograd).
    from oracle.backward import prefill_grads
    B, H, N, d = 1, 2, 20, 8
    Q, K, V = _rand((B, H, N, d), 63), _rand((B, H, N, d), 64), _rand((B, H, N, d), 65)
    G = _rand((B, H, N, d), 66)
    dQ, dK, dV = prefill_grads(Q, K, V, G, 1, 5)
    q, k, v = (torch.tensor(t, requires_grad=True) for t in (Q, K, V))
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    o.backward(torch.tensor(G))
    for a, b in ((dQ, q.grad), (dK, k.grad), (dV, v.grad)):
        np.testing.assert_allclose(a, b.numpy(), rtol=0, atol=1e-12)


def pin_backward_max_pool_ties(lib):
    # Max pooling at a tie: the whole gradient of a core element goes to the group's first
    # row holding the maximum, none to the later equal rows (the documented subgradient).
    from oracle.backward import pool_dense
    B, H, N, d, g = 1, 1, 8, 4, 4
    k = np.zeros((B, H, N, d))
    k[0, 0, 1] = k[0, 0, 3] = [2.0, 1.0, 5.0, 0.5]  # rows 1 and 3 of group 0 tie at the maximum
    k[0, 0, 4:] = _rand((4, d), 67)
    kt = torch.tensor(k, requires_grad=True)
    vt = torch.tensor(k.copy(), requires_grad=True)
    Kc, Vc = pool_dense(torch.zeros((B, H, N, d), dtype=torch.float64), kt, vt, g, 1.0, pool_mode=2)
    (Kc.sum() + 2.0 * Vc.sum()).backward()
    gk, gv = kt.grad.numpy()[0, 0], vt.grad.numpy()[0, 0]
    np.testing.assert_array_equal(gk[1], np.ones(d))
    np.testing.assert_array_equal(gk[[0, 2, 3]], np.zeros((3, d)))
    np.testing.assert_array_equal(gv[1], 2.0 * np.ones(d))
    np.testing.assert_array_equal(gv[3], np.zeros(d))
    # every element of every group sends its gradient to exactly one row
    np.testing.assert_array_equal(gk.reshape(2, g, d).sum(axis=1), np.ones((2, d)))


BACKWARD_PINS = [pin_backward_finite_differences, pin_backward_g1_is_causal, pin_backward_max_pool_ties]
