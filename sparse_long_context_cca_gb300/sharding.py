"""Sequence sharding of CCA prefill across ranks: the index maths and the one exchange step.

A sequence of N tokens is cut into `world` contiguous shards of whole groups, so that
global-aware pooling (each group scored by its own last query, "Core Context Aware
Transformers for Long Context Language Modeling", Method section, pooling equation)
stays inside a shard.  The fused attention of a row (fusion equation) then needs
  - the core tokens of every group wholly before its window: cores come from all
    earlier shards, so the ranks all-gather their pooled core tokens (1/g of K/V);
  - the raw tokens of its window, which for the first rows of a shard reach back into
    earlier shards: a halo of at most w - 1 rows (more with the group-aligned window),
    sent point to point by the ranks that hold them.
This module holds no arithmetic of the method; it plans who needs which rows and moves
them with torch.distributed (any backend with all_gather and send/recv), and `shard_prefill`
runs one rank's part with the library's kernels (pooling of its own groups, then
cca_attn_fwd_rows over its rows).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.distributed as dist


def window_lo(i: int, w: int) -> int:
    return max(0, i - w + 1)


def window_start(i: int, w: int, g: int, window_mode: int = 0) -> int:
    lo = window_lo(i, w)
    return (lo // g) * g if window_mode else lo


@dataclass(frozen=True)
class Shard:
    rank: int
    q0: int           # first query row (and first raw K/V row) this rank holds
    q1: int           # one past its last row; q0 and q1 are multiples of g
    halo0: int        # first raw K/V row its rows' windows reach back to (<= q0)
    n_cores: int      # core tokens visible to its last row: groups [0, n_cores)


def plan(N: int, g: int, w: int, world: int, window_mode: int = 0) -> list[Shard]:
    """Cuts the N / g groups into `world` contiguous runs, as even as possible (the first
    N/g mod world ranks take one group more); a rank with no group gets an empty shard."""
    if N % g:
        raise ValueError("N must be a multiple of g")
    G = N // g
    shards = []
    start = 0
    for r in range(world):
        n = G // world + (1 if r < G % world else 0)
        q0, q1 = start * g, (start + n) * g
        if q1 > q0:
            halo0 = window_start(q0, w, g, window_mode)
            n_cores = window_lo(q1 - 1, w) // g
        else:
            halo0, n_cores = q0, 0
        shards.append(Shard(r, q0, q1, halo0, n_cores))
        start += n
    return shards


def halo_sends(shards: list[Shard]) -> list[tuple[int, int, int, int]]:
    """The point-to-point transfers of the exchange: (src rank, dst rank, row0, row1) for
    every rank whose window rows [halo0, q0) lie in an earlier rank's shard."""
    out = []
    for dst in shards:
        for src in shards:
            if src.rank == dst.rank:
                continue
            a, b = max(dst.halo0, src.q0), min(dst.q0, src.q1)
            if a < b:
                out.append((src.rank, dst.rank, a, b))
    return out


def gather_cores(local_kc: torch.Tensor, local_vc: torch.Tensor, shards: list[Shard], g: int):
    """All-gathers every rank's pooled core tokens [B, Hkv, groups_r, d] into the full
    [B, Hkv, N/g, d] core tensors (group order = rank order).  Shards may differ in size,
    so each contribution is padded to the largest before the collective."""
    rank = dist.get_rank()
    sizes = [(s.q1 - s.q0) // g for s in shards]
    assert local_kc.shape[2] == sizes[rank]
    gmax = max(sizes)
    B, H, _, d = local_kc.shape
    out = []
    for t in (local_kc, local_vc):
        pad = torch.zeros((B, H, gmax, d), dtype=t.dtype, device=t.device)
        pad[:, :, :t.shape[2]] = t
        parts = [torch.empty_like(pad) for _ in shards]
        dist.all_gather(parts, pad.contiguous())
        out.append(torch.cat([p[:, :, :n] for p, n in zip(parts, sizes)], dim=2))
    return out[0], out[1]


def exchange_halo(local_k: torch.Tensor, local_v: torch.Tensor, shards: list[Shard]):
    """Returns this rank's raw K/V rows [halo0, q1) ([B, Hkv, q1 - halo0, d]): its own rows
    [q0, q1) plus the window rows received from the earlier ranks that hold them."""
    rank = dist.get_rank()
    me = shards[rank]
    B, H, _, d = local_k.shape
    k = torch.zeros((B, H, me.q1 - me.halo0, d), dtype=local_k.dtype, device=local_k.device)
    v = torch.zeros_like(k)
    k[:, :, me.q0 - me.halo0:] = local_k
    v[:, :, me.q0 - me.halo0:] = local_v
    reqs = []
    recvs = []
    for src, dst, a, b in halo_sends(shards):
        if src == rank:
            src_sh = shards[src]
            for t in (local_k, local_v):
                reqs.append(dist.isend(t[:, :, a - src_sh.q0:b - src_sh.q0].contiguous(), dst))
        elif dst == rank:
            for buf in (k, v):
                piece = torch.empty((B, H, b - a, d), dtype=local_k.dtype, device=local_k.device)
                reqs.append(dist.irecv(piece, src))
                recvs.append((buf, a, b, piece))
    for r in reqs:
        r.wait()
    for buf, a, b, piece in recvs:
        buf[:, :, a - me.halo0:b - me.halo0] = piece
    return k, v


def shard_prefill(Q, K, V, shards: list[Shard], g: int, w: int, N: int, pool_mode: int = 0,
                  window_mode: int = 0, scale: float = 0.0):
    """This rank's CCA prefill: Q, K, V [B, H, q1 - q0, d] hold its rows [q0, q1) of the
    N-token sequence (CUDA tensors).  Pools its own groups, all-gathers every rank's core
    tokens, receives its window halo, and attends its rows.  Returns (O, LSE) for its rows
    and its own core tokens; equal to rows [q0, q1) of the unsharded prefill."""
    from . import api
    me = shards[dist.get_rank()]
    if me.q1 == me.q0:
        raise ValueError("this rank holds no group")
    kc, vc = api.cca_pool(Q, K, V, g, scale=scale, pool_mode=pool_mode)
    Kc, Vc = gather_cores(kc, vc, shards, g)
    Kh, Vh = exchange_halo(K, V, shards)
    O, LSE = api.cca_attn_fwd_rows(Q, Kh, Vh, Kc, Vc, g, w, N, me.q0, me.halo0, scale=scale,
                                   window_mode=window_mode)
    return O, LSE, kc, vc
