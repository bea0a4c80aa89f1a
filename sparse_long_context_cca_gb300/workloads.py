"""Synthetic CCA prefill workloads, named by what they are.

Shapes follow the models the paper evaluates ("Core Context Aware Transformers
for Long Context Language Modeling": LLaMA2-7B with 32 heads of d=128 at
32K-128K context, LLaMA3.1-8B with 32 query heads over 8 KV heads) with the
method's default group size g=16 and window w=1024.  Values are i.i.d. normal
with a few "heavy hitter" key positions scaled up, standing in for the
attention concentration the paper observes (most weight on a few tokens).
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    g: int
    w: int
    dtype: str          # "f32" or "bf16"
    seed: int
    heavy_frac: float   # fraction of key positions scaled by heavy_mult
    heavy_mult: float = 4.0

    @property
    def n_groups(self) -> int:
        return self.N // self.g

    def small(self, **kw) -> "Workload":
        return replace(self, **kw)


TINY_F32 = Workload("tiny-f32 B1 H2 d64 N256 g16 w32", 1, 2, 2, 256, 64, 16, 32, "f32", 0, 0.02)
MHA_32K = Workload("llama2-7b-mha B1 H32 d128 N32768 g16 w1024", 1, 32, 32, 32768, 128, 16, 1024,
                   "bf16", 1, 0.01)
MHA_128K = Workload("llama2-7b-mha B1 H32 d128 N131072 g16 w1024", 1, 32, 32, 131072, 128, 16, 1024,
                    "bf16", 2, 0.01)
GQA_64K = Workload("llama3.1-8b-gqa B1 Hq32 Hkv8 d128 N65536 g16 w1024", 1, 32, 8, 65536, 128, 16,
                   1024, "bf16", 3, 0.01)


def sweep() -> list[Workload]:
    """B=2, H=32, d=128, N=65536 over g in {8,16,32,64} x w in {256,1024,4096}; seeds 10..21."""
    out = []
    seed = 10
    for g in (8, 16, 32, 64):
        for w in (256, 1024, 4096):
            out.append(Workload(f"mha-sweep B2 H32 d128 N65536 g{g} w{w}", 2, 32, 32, 65536, 128, g,
                                w, "bf16", seed, 0.01))
            seed += 1
    return out


ALL = [TINY_F32, MHA_32K, MHA_128K, GQA_64K] + sweep()


def visible_keys_per_head(N: int, g: int, w: int) -> tuple[int, int]:
    """(core keys, local keys) summed over all queries of one head: exact sums of
    n_core(i) = max(0, i-w+1)//g and n_loc(i) = min(w, i+1)."""
    core = 0
    loc = 0
    for i in range(N):
        lo = i - w + 1 if i - w + 1 > 0 else 0
        core += lo // g
        loc += i - lo + 1
    return core, loc


def attn_flops(wl: Workload) -> float:
    """Algorithmic attention FLOPs: 4*d per (query, visible key, query head)."""
    core, loc = _visible_cached(wl.N, wl.g, wl.w)
    return 4.0 * wl.d * (core + loc) * wl.B * wl.Hq


def pool_bytes(wl: Workload) -> float:
    """Algorithmic pooling bytes: read K, V and the group-last queries; write Kc, Vc."""
    e = 2 if wl.dtype == "bf16" else 4
    ng = wl.N // wl.g
    return float(wl.B * wl.Hkv * (2 * wl.N * wl.d + 2 * ng * wl.d) * e + wl.B * wl.Hq * ng * wl.d * e)


def attn_min_bytes(wl: Workload) -> float:
    """Compulsory attention bytes: Q, K, V, Kc, Vc read once; O and LSE written once."""
    e = 2 if wl.dtype == "bf16" else 4
    ng = wl.N // wl.g
    return float(e * wl.d * (2 * wl.B * wl.Hq * wl.N + 2 * wl.B * wl.Hkv * (wl.N + ng))
                 + 4 * wl.B * wl.Hq * wl.N)


_vis_cache: dict = {}


def _visible_cached(N, g, w):
    key = (N, g, w)
    if key not in _vis_cache:
        _vis_cache[key] = _visible_closed_form(N, g, w)
    return _vis_cache[key]


def _visible_closed_form(N: int, g: int, w: int) -> tuple[int, int]:
    # local: sum_{i<N} min(w, i+1)
    if N <= w:
        loc = N * (N + 1) // 2
    else:
        loc = w * (w + 1) // 2 + (N - w) * w
    # core: sum over lo = 1..N-w of lo // g (lo(i) = i-w+1 for i >= w)
    M = N - w
    if M <= 0:
        core = 0
    else:
        q, rem = divmod(M + 1, g)   # values lo = 0..M ; sum_{x=0}^{M} x//g
        core = g * (q * (q - 1) // 2) + q * rem
    return core, loc
