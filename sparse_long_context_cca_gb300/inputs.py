"""Seeded synthetic inputs for CCA prefill.

This module only draws random numbers: it holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.
Recipe: Q, K, V i.i.d. N(0, 1), scaled by d**-0.25 for bf16 workloads (1 for
fp32); round(heavy_frac * N) distinct key positions, drawn by a seeded
permutation, have K scaled by heavy_mult for every batch and KV head; then the
tensors are cast to the workload dtype.  Generation order is Q, K, V, then the
permutation, all from one torch.Generator seeded with the workload seed on the
target device.
"""
from __future__ import annotations

import torch

from .workloads import Workload

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def make_qkv(wl: Workload, device="cpu"):
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed)
    scale = 1.0 if wl.dtype == "f32" else wl.d ** -0.25
    dt = TORCH_DTYPE[wl.dtype]
    out = []
    for H in (wl.Hq, wl.Hkv, wl.Hkv):
        t = torch.randn((wl.B, H, wl.N, wl.d), generator=gen, device=device, dtype=torch.float32)
        if scale != 1.0:
            t.mul_(scale)
        out.append(t)
    Q, K, V = out
    n_heavy = int(round(wl.heavy_frac * wl.N))
    if n_heavy > 0:
        pos = torch.randperm(wl.N, generator=gen, device=device)[:n_heavy]
        K[:, :, pos, :] *= wl.heavy_mult
    return Q.to(dt), K.to(dt), V.to(dt)
