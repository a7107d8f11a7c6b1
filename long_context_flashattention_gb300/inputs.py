"""Seeded synthetic inputs shared by the oracle checks, the tests and the bench.

This module holds no attention arithmetic: it only draws numbers.  Both the
CUDA path and the fp64 oracle consume exactly the tensors it returns.

Recipe (the pages fix none of it; see the design notes): a CPU
``torch.Generator`` seeded with the workload's seed draws Q, K, V and dO, in
that order, as fp32 N(0, 1) tensors of shape [B, H, N, d]; each is rounded to
bf16 (round to nearest even).  For the stress variant, ``N // 100`` query
positions drawn by ``torch.randperm(N)`` from the same generator (after the
four tensors) are multiplied by 8 in every head (exact in bf16).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    seed: int
    P: int
    partitions: tuple
    stress_rows: bool = False

    @property
    def causal_pairs(self) -> int:
        return self.B * self.Hq * self.N * (self.N + 1) // 2

    @property
    def flops_fwd(self) -> int:
        return 4 * self.d * self.causal_pairs

    @property
    def flops_bwd(self) -> int:
        return 10 * self.d * self.causal_pairs


WORKLOADS = {
    "tiny": Workload("tiny causal B1 H1 N256 d64", 1, 1, 1, 256, 64, 0, 4,
                     ("contiguous", "balanced", "striped")),
    "llama7b_32k": Workload("llama-7b attention B1 H32 N32768 d128", 1, 32, 32, 32768, 128,
                            1, 8, ("balanced",)),
    "llama7b_128k": Workload("llama-7b attention B1 H32 N131072 d128", 1, 32, 32, 131072,
                             128, 2, 8, ("striped", "contiguous"), stress_rows=True),
    "llama7b_512k": Workload("llama-7b attention B1 H32 N524288 d128", 1, 32, 32, 524288,
                             128, 3, 16, ("balanced",)),
    "gqa_64k": Workload("grouped-query attention B2 Hq32 Hkv8 N65536 d128", 2, 32, 8, 65536,
                        128, 4, 16, ("striped",)),
}


def make_qkvdo(B: int, Hq: int, Hkv: int, N: int, d: int, seed: int,
               stress_rows: bool = False):
    """Return bf16 CPU tensors (q, k, v, dout) per the recipe above."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, N, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    do = torch.randn(B, Hq, N, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    if stress_rows:
        idx = torch.randperm(N, generator=g)[: N // 100]
        q[:, :, idx, :] = q[:, :, idx, :] * 8
    return q, k, v, do


def make_workload(w: Workload):
    return make_qkvdo(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed, w.stress_rows)


def sample_rows(B: int, H: int, N: int, count: int, seed: int, chunk: int | None = None):
    """Seeded flat row indices (b*H + h)*N + i for sampled checks.

    Always includes i = 0 and i = N - 1 (and, when ``chunk`` is given, the
    first and last row of every chunk) for head (0, 0) and the last head; the
    rest are uniform over all rows."""
    g = torch.Generator().manual_seed(seed)
    fixed = []
    for bh in (0, B * H - 1):
        fixed += [bh * N + 0, bh * N + N - 1]
        if chunk:
            for c in range(0, N, chunk):
                fixed += [bh * N + c, bh * N + min(N, c + chunk) - 1]
    fixed = sorted(set(fixed))
    rest = max(0, count - len(fixed))
    rnd = torch.randint(0, B * H * N, (rest,), generator=g).tolist()
    return sorted(set(fixed + rnd))[:max(count, len(fixed))]


def sample_key_rows(N: int, P: int, count: int, seed: int):
    """Seeded key positions (natural order) for element-by-element dK/dV checks.

    Always includes the first keys (seen by every query), the last keys (seen
    by few), both sides of every chunk boundary of the contiguous (N/P) and
    folded (N/(2P)) partitions and of every 32768-row block, and the rest
    uniform over [0, N) without repeats."""
    fixed = {0, 1, 2, 127, 128, N - 129, N - 128, N - 2, N - 1}
    for step in (N // P, N // (2 * P), 32768):
        if step > 0:
            for c in range(step, N, step):
                fixed |= {c - 1, c}
    fixed = {x for x in fixed if 0 <= x < N}
    g = torch.Generator().manual_seed(seed)
    rest = [x for x in torch.randperm(N, generator=g).tolist() if x not in fixed]
    return sorted(fixed | set(rest[:max(0, count - len(fixed))]))


def random_partials(k: int, rows: int, d: int, seed: int, neg_inf_frac: float = 0.0):
    """fp32 partial (O, LSE) pairs for merge tests: O ~ N(0,1), LSE ~ 4 N(0,1);
    a fraction of (partial, row) entries is set to (0, -inf) (a chunk pair in
    which the row sees no key)."""
    g = torch.Generator().manual_seed(seed)
    o = torch.randn(k, rows, d, generator=g, dtype=torch.float32)
    lse = 4.0 * torch.randn(k, rows, generator=g, dtype=torch.float32)
    if neg_inf_frac > 0:
        m = torch.rand(k, rows, generator=g) < neg_inf_frac
        lse[m] = float("-inf")
        o[m] = 0.0
    return o, lse
