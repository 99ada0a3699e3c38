"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers on the CPU (torch.Generator) and shapes
them like the workloads of the pages; it holds none of the method's arithmetic
(no quantization, no scaling, no GEMM).  Both the CUDA path and the CPU oracle
receive the exact same bytes.

Recipes (all CPU, deterministic per seed):
  * ``normal_bf16``: N(0, 1) drawn in float32, rounded to bf16.
  * outliers: floor(numel/1024) distinct positions chosen by randperm are
    multiplied by 400 (in float32, before the bf16 rounding).  This is the
    "1 in 1024 elements scaled x400" outlier model; it makes some 1x128 and
    128x128 groups carry a large max |x| next to ordinary values, the situation
    of the DeepGEMM page's per-tensor outlier example.
  * ``uniform_16bit``: uniform[-1, 1] drawn in float32, rounded to fp16/bf16.
  * ``expert_counts``: multinomial(total, uniform over G experts) counts.
  * ``masked_rows``: valid rows per expert uniform in [0, Mmax].
"""
from __future__ import annotations

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed: int, outliers: bool = False) -> torch.Tensor:
    """bf16 CPU tensor, N(0,1); optionally with the 1-in-1024 x400 outliers."""
    g = _gen(seed)
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if outliers:
        n = x.numel()
        k = n // 1024
        if k > 0:
            g2 = _gen(seed + 1_000_003)
            pos = torch.randperm(n, generator=g2)[:k]
            flat = x.view(-1)
            flat[pos] = flat[pos] * 400.0
    return x.to(torch.bfloat16)


def uniform_16bit(shape, seed: int, dtype=torch.float16) -> torch.Tensor:
    """fp16 (or bf16) CPU tensor, uniform in [-1, 1]."""
    g = _gen(seed)
    x = torch.rand(*shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    return x.to(dtype)


def expert_counts(total: int, num_experts: int, seed: int) -> list[int]:
    """Per-expert token counts: multinomial(total, uniform) with the seed."""
    g = _gen(seed)
    probs = torch.ones(num_experts, dtype=torch.float64)
    draws = torch.multinomial(probs, total, replacement=True, generator=g)
    return torch.bincount(draws, minlength=num_experts).tolist()


def masked_rows(num_experts: int, mmax: int, seed: int) -> torch.Tensor:
    """int32 CPU tensor of valid rows per expert, uniform in [0, mmax]."""
    g = _gen(seed)
    return torch.randint(0, mmax + 1, (num_experts,), generator=g, dtype=torch.int64).to(torch.int32)


def contiguous_layout(counts: list[int], align: int):
    """Row-to-expert map of the contiguous grouped layout.

    Each expert's segment is padded up to a multiple of ``align`` rows; padding
    rows carry expert id -1.  Returns (m_indices int32 tensor, total rows).
    """
    ids = []
    for g, c in enumerate(counts):
        padded = (c + align - 1) // align * align
        ids.extend([g] * c)
        ids.extend([-1] * (padded - c))
    return torch.tensor(ids, dtype=torch.int32), len(ids)
