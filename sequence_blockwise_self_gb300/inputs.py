"""Seeded synthetic inputs and row samplers.

Shared by the tests, the benchmark and the smoke check, and by both sides of
every parity comparison (the CUDA library and the fp64 oracle).  This module
holds no attention arithmetic: it only draws numbers and picks row indices.

Recipe: q, k, v and dO are drawn as float32 N(0, 1) from a CPU
``torch.Generator`` seeded with ``seed``, in the order q, k, v, dO, and then
rounded to bfloat16 (round to nearest even).  Layout is [B, H, L, d].
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    L: int
    d: int
    n_chunks: int
    causal: bool

    def fwd_flops(self) -> float:
        """4 B Hq L^2 d, halved when causal (the benchmark's FLOP count)."""
        f = 4.0 * self.B * self.Hq * self.L * self.L * self.d
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops()


# The five synthetic workloads: shapes of a BERT-large encoder, a causal MHA
# decoder and the Qwen2-7B attention (28 query heads, 4 kv heads, d = 128).
WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 2, 256, 64, 4, False),
    "encoder": Workload("encoder", 8, 16, 16, 4096, 64, 8, False),
    "decoder_mha": Workload("decoder_mha", 4, 32, 32, 8192, 128, 8, True),
    "gqa_32k": Workload("gqa_32k", 1, 28, 4, 32768, 128, 16, True),
    "gqa_128k": Workload("gqa_128k", 1, 28, 4, 131072, 128, 32, True),
}
WORKLOAD_SEEDS = {"tiny": 0, "encoder": 1, "decoder_mha": 2, "gqa_32k": 3, "gqa_128k": 4}


def make_inputs(B, Hq, Hkv, L, d, seed, with_grad=True):
    """Return bf16 CPU tensors (q, k, v, dO); dO is None if with_grad is False."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, Hq, L, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((B, Hkv, L, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((B, Hkv, L, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    dO = None
    if with_grad:
        dO = torch.randn((B, Hq, L, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return q, k, v, dO


def head_seed(seed: int, tensor: int, b: int, h: int) -> int:
    """Seed of one (tensor, batch, head) slice for head_rows: tensor 0..3 =
    q, k, v, dO."""
    return int(seed) * 1_000_003 + tensor * 100_003 + b * 1_009 + h


def head_rows(L: int, d: int, seed: int):
    """One head's [L, d] bf16 rows ~ N(0,1) (drawn in fp32, rounded)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn((L, d), generator=g, dtype=torch.float32).to(torch.bfloat16)


def make_inputs_by_head(B, Hq, Hkv, L, d, seed, device):
    """q, k, v, dO built one head at a time on the CPU (head_rows, seeds from
    head_seed) straight into tensors on `device`: for problems too large to
    draw whole in host memory; any head can be drawn again alone."""
    out = []
    for t, H in enumerate((Hq, Hkv, Hkv, Hq)):
        x = torch.empty((B, H, L, d), dtype=torch.bfloat16, device=device)
        for b in range(B):
            for h in range(H):
                x[b, h].copy_(head_rows(L, d, head_seed(seed, t, b, h)))
        out.append(x)
    return tuple(out)


def workload_inputs(w: Workload, seed=None, with_grad=True):
    s = WORKLOAD_SEEDS.get(w.name, 0) if seed is None else seed
    return make_inputs(w.B, w.Hq, w.Hkv, w.L, w.d, s, with_grad)


def boundary_rows(L: int, n_chunks: int, causal: bool, lo: int = 0):
    """First and last row of every chunk (encoder) or sub-chunk (causal, 2N
    sub-chunks of length L/(2N)), plus rows lo and L-1; only rows >= lo."""
    parts = 2 * n_chunks if causal else n_chunks
    c = L // parts
    rows = {lo, L - 1}
    for i in range(parts):
        rows.add(i * c)
        rows.add(min(L - 1, (i + 1) * c - 1))
    return {r for r in rows if r >= lo}


def sample_rows(L: int, n_chunks: int, causal: bool, n: int, seed: int, lo: int = 0):
    """Sorted sample of n distinct rows of [lo, L): all chunk boundary rows
    in that range, then uniform draws without replacement from numpy's
    default_rng(seed + 1000)."""
    rows = boundary_rows(L, n_chunks, causal, lo)
    span = L - lo
    if len(rows) >= n or n >= span:
        base = sorted(rows) if n < span else list(range(lo, L))
        return np.array(base[:max(n, len(rows))] if n < span else base, dtype=np.int32)
    rng = np.random.default_rng(seed + 1000)
    rest = np.setdiff1d(np.arange(lo, L), np.array(sorted(rows)))
    extra = rng.choice(rest, size=n - len(rows), replace=False)
    return np.array(sorted(rows | set(int(x) for x in extra)), dtype=np.int32)


# ---------------------------------------------------------------- blockwise FFN

@dataclass(frozen=True)
class FfnWorkload:
    """The feed-forward block after attention: M token rows of hidden size D,
    hidden layer F = 4 D, processed block_rows rows at a time."""
    name: str
    M: int
    D: int
    F: int
    block_rows: int

    def flops(self) -> float:
        """Two GEMMs of 2 M D F each (bias, GELU and residual not counted)."""
        return 4.0 * self.M * self.D * self.F


# Hidden size 3584 = 28 heads x 128 (the GQA attention above), F = 4 D; the
# 128k-token sequence in blocks of 8192 rows.
FFN_WORKLOADS = {
    "ffn_small": FfnWorkload("ffn_small", 1000, 512, 2048, 384),
    "ffn_gqa_128k": FfnWorkload("ffn_gqa_128k", 131072, 3584, 14336, 8192),
}
FFN_SEEDS = {"ffn_small": 20, "ffn_gqa_128k": 21}


def make_ffn_inputs(M, D, F, seed):
    """Return CPU tensors (x, w1, b1, w2, b2): x [M, D] ~ N(0, 1), w1 [F, D] ~
    N(0, 1/D), w2 [D, F] ~ N(0, 1/F) (weights output-major, as a linear
    layer stores them), all rounded to bf16; biases b1 [F], b2 [D] ~
    N(0, 0.01) in fp32.  Drawn as float32 from a CPU torch.Generator seeded
    with `seed`, in the order x, w1, b1, w2, b2."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn((M, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    w1 = (torch.randn((F, D), generator=g, dtype=torch.float32) / D ** 0.5).to(torch.bfloat16)
    b1 = torch.randn((F,), generator=g, dtype=torch.float32) * 0.1
    w2 = (torch.randn((D, F), generator=g, dtype=torch.float32) / F ** 0.5).to(torch.bfloat16)
    b2 = torch.randn((D,), generator=g, dtype=torch.float32) * 0.1
    return x, w1, b1, w2, b2


def ffn_sample_rows(M: int, block_rows: int, n: int, seed: int):
    """Sorted sample of distinct rows: the first and last row of every block
    and of every 128-row tile edge next to a block edge, then uniform draws
    from numpy's default_rng(seed + 2000) up to n rows."""
    rows = {0, M - 1}
    for b in range(0, M, block_rows):
        for r in (b, b + 127, b + 128, min(M, b + block_rows) - 1):
            if 0 <= r < M:
                rows.add(r)
    rows = set(sorted(rows)[:n]) if len(rows) > n else rows
    if len(rows) < n:
        rng = np.random.default_rng(seed + 2000)
        rest = np.setdiff1d(np.arange(M), np.array(sorted(rows)))
        rows |= set(int(r) for r in rng.choice(rest, size=min(n - len(rows), rest.size), replace=False))
    return np.array(sorted(rows), dtype=np.int64)
