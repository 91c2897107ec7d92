"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic.  Recipe (every workload):

* one CPU ``torch.Generator`` seeded with ``seed``;
* draw ``q`` [B,S,H,D], then ``k`` [B,S,Hkv,D], as ``randn`` fp32 times
  ``sigma_qk``; for the outlier-key workload, on the same generator and right
  after the ``k`` draw, for each (b, kv-head) in order take
  ``randperm(S)[:ceil(frac*S)]`` and multiply those key rows by
  ``outlier_scale`` (a power of two, so exact in bf16);
* draw ``v`` [B,S,Hkv,D] as ``randn`` fp32 times ``sigma_v``;
* round each to bf16 (round-to-nearest-even) once; both sides read those bits.

The workloads are the shapes of long-context attention the method targets:
a tiny non-causal case, a short causal case, a GQA causal case, a long-context
case with a peaked softmax (q, k with standard deviation 3) and a small-head
many-chunk GQA case with 1 % outlier keys.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    S: int
    D: int
    P: int
    causal: bool
    sigma_qk: float = 1.0
    sigma_v: float = 1.0
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def chunk(self) -> int:
        return self.S // self.P

    @property
    def n_pairs_per_head(self) -> int:
        """(query, key) pairs the definition weighs: S^2, or S(S+1)/2 causal."""
        return self.S * (self.S + 1) // 2 if self.causal else self.S * self.S

    @property
    def flops(self) -> int:
        """Exact FLOPs of the two contractions (2 per multiply-add, QK^T and PV)."""
        return 4 * self.B * self.H * self.D * self.n_pairs_per_head

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", B=1, H=2, Hkv=2, S=256, D=64, P=2, causal=False),
    "causal_s4096": Workload("causal_s4096", B=1, H=8, Hkv=8, S=4096, D=128, P=4, causal=True),
    "gqa_s16384": Workload("gqa_s16384", B=2, H=32, Hkv=8, S=16384, D=128, P=8, causal=True),
    "long_s65536": Workload("long_s65536", B=1, H=16, Hkv=16, S=65536, D=128, P=16,
                            causal=True, sigma_qk=3.0),
    "d64_s32768": Workload("d64_s32768", B=4, H=32, Hkv=4, S=32768, D=64, P=32, causal=True,
                           outlier_frac=0.01, outlier_scale=8.0),
}

# the workload the benchmark's headline number is quoted on
HEADLINE = "gqa_s16384"


def make_inputs(w: Workload, seed: int | None = None):
    """Return bf16 CPU tensors (q, k, v) for workload ``w`` (see module doc)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    q = torch.randn((w.B, w.S, w.H, w.D), generator=g, dtype=torch.float32)
    if w.sigma_qk != 1.0:
        q.mul_(w.sigma_qk)
    k = torch.randn((w.B, w.S, w.Hkv, w.D), generator=g, dtype=torch.float32)
    if w.sigma_qk != 1.0:
        k.mul_(w.sigma_qk)
    if w.outlier_frac > 0.0:
        n_out = math.ceil(w.outlier_frac * w.S)
        for b in range(w.B):
            for hk in range(w.Hkv):
                idx = torch.randperm(w.S, generator=g)[:n_out]
                k[b, idx, hk, :] *= w.outlier_scale
    v = torch.randn((w.B, w.S, w.Hkv, w.D), generator=g, dtype=torch.float32)
    if w.sigma_v != 1.0:
        v.mul_(w.sigma_v)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def sample_rows(w: Workload, n_random: int = 256, seed: int = 1, every: int = 128,
                heads=None):
    """Deterministic row sample per (b, h): the first and last row of every
    chunk, every ``every``-th row and ``n_random`` seeded random rows.  Returns
    sorted unique flat ids ``(b*H + h)*S + s`` as an int64 tensor."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    C = w.chunk
    base = set(range(0, w.S, every))
    for c in range(w.P):
        base.add(c * C)
        base.add(c * C + C - 1)
    base.add(w.S - 1)
    base = torch.tensor(sorted(base), dtype=torch.int64)
    ids = []
    hs = range(w.H) if heads is None else heads
    for b in range(w.B):
        for h in hs:
            extra = torch.randint(0, w.S, (n_random,), generator=g, dtype=torch.int64)
            s = torch.unique(torch.cat([base, extra]))
            ids.append((b * w.H + h) * w.S + s)
    return torch.unique(torch.cat(ids))
