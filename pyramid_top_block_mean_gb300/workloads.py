"""Seeded synthetic inputs for the selector (shared by the GPU path's tests,
the benchmark and the CPU oracle's tests).

This module only draws random numbers and plants patterns into them; it holds
none of the selector's arithmetic.  Shapes follow the workloads of the pages
about "Block Sparse Attention with Log-Linear Complexity" (agihunt.info
summary, model paragraph: C = 64, K = 8 in pretraining at 4K tokens, K = 32 in
continued pretraining at 16K; rcap.io post, latency bullet: 64K-256K tokens).
No dataset is used: every tensor is drawn from a seeded torch.Generator.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass
class Shape:
    """Problem shape.  Layouts: q [B, Hq, N, d], k [B, Hkv, N, d]."""
    B: int
    N: int
    Hq: int
    Hkv: int
    d: int
    C: int = 64
    K: int = 8
    g: int = 2
    qtile: int = 4
    dtype: str = "bf16"  # "bf16" or "fp32"

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


# The five workload families (sizes as the pages' experiments use them).
TINY = Shape(B=1, N=1024, Hq=1, Hkv=1, d=64, K=4, dtype="fp32")
PRETRAIN = Shape(B=2, N=4096, Hq=16, Hkv=4, d=128, K=8)
CPT = Shape(B=1, N=16384, Hq=16, Hkv=4, d=128, K=32)
SWEEP_NS = (4096, 16384, 65536, 131072, 262144)


def sweep(N: int) -> Shape:
    return Shape(B=1, N=N, Hq=16, Hkv=4, d=128, K=8)


DECODE = Shape(B=64, N=131072 + 16, Hq=32, Hkv=8, d=128, K=32)
DECODE_CACHED = 131072  # keys already in the cache before the first step
DECODE_STEPS = 16


def _gen(seed: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def iid(shape: Shape, seed: int, device: str = "cpu"):
    """q, k iid N(0, 1), drawn in fp32 then cast once to the shape's dtype."""
    g = _gen(seed, device)
    q = torch.randn(shape.B, shape.Hq, shape.N, shape.d, generator=g,
                    device=device, dtype=torch.float32)
    k = torch.randn(shape.B, shape.Hkv, shape.N, shape.d, generator=g,
                    device=device, dtype=torch.float32)
    return q.to(shape.torch_dtype), k.to(shape.torch_dtype)


def values(shape: Shape, seed: int, device: str = "cpu"):
    """v [B, Hkv, N, d] iid N(0, 1) (the values read by attention over the
    selected blocks), from a generator of its own: seed + 7919."""
    g = _gen(seed + 7919, device)
    v = torch.randn(shape.B, shape.Hkv, shape.N, shape.d, generator=g,
                    device=device, dtype=torch.float32)
    return v.to(shape.torch_dtype)


def planted(shape: Shape, seed: int, frac: float = 0.01, amp: float = 3.0,
            noise: float = 0.5, device: str = "cpu"):
    """iid N(0,1) keys, with a fraction `frac` of key positions j (uniform,
    per batch and key head) replaced by amp * q[t, h'] + noise * N(0, I) for
    a later query position t uniform in (j, N) and a query head h' uniform
    in the key head's GQA group."""
    g = _gen(seed, device)
    q = torch.randn(shape.B, shape.Hq, shape.N, shape.d, generator=g,
                    device=device, dtype=torch.float32)
    k = torch.randn(shape.B, shape.Hkv, shape.N, shape.d, generator=g,
                    device=device, dtype=torch.float32)
    n_plant = int(round(frac * shape.N))
    G = shape.G
    for b in range(shape.B):
        for h in range(shape.Hkv):
            if n_plant == 0 or shape.N < 2:
                continue
            j = torch.randperm(shape.N - 1, generator=g, device=device)[:n_plant]
            u = torch.rand(n_plant, generator=g, device=device)
            t = j + 1 + (u * (shape.N - 1 - j).to(torch.float32)).long()
            t = torch.minimum(t, torch.full_like(t, shape.N - 1))
            hh = torch.randint(0, G, (n_plant,), generator=g, device=device)
            eps = torch.randn(n_plant, shape.d, generator=g, device=device)
            k[b, h, j] = amp * q[b, h * G + hh, t] + noise * eps
    return q.to(shape.torch_dtype), k.to(shape.torch_dtype)


def needles(shape: Shape, seed: int, n_needles: int = 8, noise: float = 0.1,
            device: str = "cpu"):
    """iid N(0,1) q and k; per (batch, key head), n_needles distinct leaf
    blocks (uniform in [1, nb-3], i.e. eligible for the last query) get keys
    2*sqrt(d)*u + noise*N(0, I), u the unit vector of the last query's first
    head in the group (a fixed query direction)."""
    g = _gen(seed, device)
    q = torch.randn(shape.B, shape.Hq, shape.N, shape.d, generator=g,
                    device=device, dtype=torch.float32)
    k = torch.randn(shape.B, shape.Hkv, shape.N, shape.d, generator=g,
                    device=device, dtype=torch.float32)
    nb = (shape.N + shape.C - 1) // shape.C
    hi = nb - 3
    blocks = []
    for b in range(shape.B):
        for h in range(shape.Hkv):
            if hi < 1:
                blocks.append([])
                continue
            m = min(n_needles, hi)
            sel = (1 + torch.randperm(hi, generator=g, device=device)[:m]).tolist()
            u = q[b, h * shape.G, shape.N - 1]
            u = u / u.norm()
            for blk in sel:
                lo = blk * shape.C
                eps = torch.randn(shape.C, shape.d, generator=g, device=device)
                k[b, h, lo:lo + shape.C] = 2.0 * math.sqrt(shape.d) * u + noise * eps
            blocks.append(sorted(sel))
    return q.to(shape.torch_dtype), k.to(shape.torch_dtype), blocks


def decode_inputs(shape: Shape, seed: int, device: str = "cpu",
                  steps: int = DECODE_STEPS):
    """K cache [B, Hkv, N_max, d] iid N(0,1) (positions beyond the cached
    length hold the keys the decode steps append), and per-step queries
    q [steps, B, Hq, d] iid N(0,1)."""
    g = _gen(seed, device)
    kc = torch.empty(shape.B, shape.Hkv, shape.N, shape.d,
                     dtype=shape.torch_dtype, device=device)
    # drawn one (batch, head) slab at a time to bound fp32 scratch
    for b in range(shape.B):
        for h in range(shape.Hkv):
            kc[b, h] = torch.randn(shape.N, shape.d, generator=g, device=device,
                                   dtype=torch.float32).to(shape.torch_dtype)
    q = torch.randn(steps, shape.B, shape.Hq, shape.d, generator=g,
                    device=device, dtype=torch.float32).to(shape.torch_dtype)
    return q, kc


def random_shape(gen: torch.Generator, max_blocks: int = 40,
                 C_choices=(2, 4, 8), d_choices=(2, 4, 8),
                 G_choices=(1, 2, 4), K_choices=(1, 2, 3, 4)) -> Shape:
    """A random tiny shape (for brute-force checks of the oracle)."""
    def pick(xs):
        return xs[int(torch.randint(0, len(xs), (1,), generator=gen))]
    C = pick(C_choices)
    nb = int(torch.randint(1, max_blocks + 1, (1,), generator=gen))
    N = max(1, nb * C - int(torch.randint(0, C, (1,), generator=gen)))
    G = pick(G_choices)
    Hkv = int(torch.randint(1, 3, (1,), generator=gen))
    return Shape(B=1 + int(torch.randint(0, 2, (1,), generator=gen)), N=N,
                 Hq=Hkv * G, Hkv=Hkv, d=pick(d_choices), C=C, K=pick(K_choices),
                 dtype="fp32")
