"""fp64 gradients of CCA prefill (pooling + fused attention) w.r.t. Q, K and V.

TEST INFRASTRUCTURE, like the rest of ``oracle/``.  The forward is written out
densely in plain PyTorch CPU fp64 ops (one softmax over a [groups, g] matrix for
the pooling, then one masked softmax over the concatenation [cores; tokens]) and
differentiated with torch.autograd; the gradient of a plain definition is the
plain definition of the backward pass.  Pinned in the tests against central
finite differences of the C oracle's forward and, for g = 1, against the
gradients of torch's own causal scaled_dot_product_attention.

Formulas ("Core Context Aware Transformers for Long Context Language
Modeling", Method section, pooling and fusion equations), readings as in the C
oracle: core j visible to query i iff (j+1)*g <= max(0, i-w+1); raw window
[lo(i), i] (window_mode 1: [g*(lo(i)//g), i]); pool_mode 1 mean, 2 element-wise
max, 3 per-query-head softmax weights averaged over the heads sharing a KV head.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import widen


def pool_dense(q, k, v, g: int, tau: float, pool_mode: int = 0):
    """Differentiable pooling -> (Kc, Vc) [B, Hkv, N/g, d].  Max pooling takes, per
    element, the group's first row holding the maximum (a gather at the first argmax),
    so at ties the whole gradient goes to that row: the reading the library documents
    for the subgradient of max."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    r, G = Hq // Hkv, N // g
    Kg = k.reshape(B, Hkv, G, g, d)
    Vg = v.reshape(B, Hkv, G, g, d)
    if pool_mode == 2:
        ik = Kg.argmax(dim=3, keepdim=True)  # first maximal row (torch returns the first)
        iv = Vg.argmax(dim=3, keepdim=True)
        return Kg.gather(3, ik).squeeze(3), Vg.gather(3, iv).squeeze(3)
    if pool_mode == 1:
        a = torch.full((B, Hkv, G, g), 1.0 / g, dtype=q.dtype)
    elif pool_mode == 3:
        # one softmax per query head over its own logits, averaged over the r heads
        qlast = q[:, :, g - 1::g].reshape(B, Hkv, r, G, d)
        s = tau * torch.einsum("bkrjc,bkjtc->bkrjt", qlast, Kg)
        a = torch.softmax(s, dim=-1).mean(dim=2)
    else:
        qlast = q[:, :, g - 1::g].reshape(B, Hkv, r, G, d)
        s = tau * torch.einsum("bkrjc,bkjtc->bkjt", qlast, Kg) / r
        a = torch.softmax(s, dim=-1)
    return torch.einsum("bkjt,bkjtc->bkjc", a, Kg), torch.einsum("bkjt,bkjtc->bkjc", a, Vg)


def dense_forward(q, k, v, g: int, w: int, scale: float | None = None, pool_mode: int = 0,
                  window_mode: int = 0):
    """Differentiable fp64 forward: returns (O [B,Hq,N,d], LSE [B,Hq,N])."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    r, G = Hq // Hkv, N // g
    tau = 1.0 / math.sqrt(d) if scale is None else float(scale)
    Kc, Vc = pool_dense(q, k, v, g, tau, pool_mode)
    i = torch.arange(N)[:, None]
    lo = torch.clamp(i - w + 1, min=0)
    n_core = lo // g
    win = n_core * g if window_mode else lo
    core_mask = torch.arange(G)[None, :] < n_core
    tok = torch.arange(N)[None, :]
    loc_mask = (tok >= win) & (tok <= i)
    mask = torch.cat([core_mask, loc_mask], dim=1)
    kv_head = torch.arange(Hq) // r
    Kcat = torch.cat([Kc, k], dim=2)[:, kv_head]
    Vcat = torch.cat([Vc, v], dim=2)[:, kv_head]
    z = tau * torch.einsum("bhic,bhmc->bhim", q, Kcat)
    z = z.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(z, dim=-1)
    p = torch.exp(z - lse[..., None])
    O = torch.einsum("bhim,bhmc->bhic", p, Vcat)
    return O, lse


def prefill_grads(Q, K, V, dO, g: int, w: int, scale: float | None = None, pool_mode: int = 0,
                  window_mode: int = 0):
    """(dQ, dK, dV) in fp64 for the loss sum(dO * O), from exact fp64 copies of the inputs."""
    q = torch.tensor(widen(Q), requires_grad=True)
    k = torch.tensor(widen(K), requires_grad=True)
    v = torch.tensor(widen(V), requires_grad=True)
    O, _ = dense_forward(q, k, v, g, w, scale, pool_mode, window_mode)
    O.backward(torch.tensor(widen(dO)))
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()
