"""Shared helpers for the GPU parity tests (comparison rules and case builders).

Tolerances: quantize outputs (codes and scale words) must be bit-exact.  GEMM
outputs must satisfy max |D - D_ref| <= 1e-2 * max |D_ref| and cosine
similarity >= 0.99999 against the fp64 oracle on the same inputs; the GPU
GEMMs consume the oracle's quantized bytes, so the GEMM comparison does not
depend on the GPU quantizer.
"""
from __future__ import annotations

import numpy as np
import torch

REL_MAX_ERR = 1e-2
MIN_COS = 0.99999
BF16_NAN = 0x7FC0


def gemm_close(got: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values in the output"
    err = float(np.abs(g - r).max()) if g.size else 0.0
    scale = float(np.abs(r).max()) if r.size else 0.0
    denom = float(np.linalg.norm(g) * np.linalg.norm(r))
    cos = float((g * r).sum() / denom) if denom > 0 else 1.0
    assert err <= REL_MAX_ERR * scale + 1e-30, f"{what}: max err {err:.4e} > {REL_MAX_ERR} * {scale:.4e}"
    assert cos >= MIN_COS, f"{what}: cosine {cos:.8f} < {MIN_COS}"
    return {"max_err": err, "max_ref": scale, "cos": cos}


def nan_filled(shape, device, dtype=torch.bfloat16) -> torch.Tensor:
    """Output buffer pre-filled with NaN, to detect writes outside the valid rows."""
    t = torch.empty(shape, dtype=torch.int16, device=device)
    t.fill_(BF16_NAN)
    return t.view(dtype)


def to_dev(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def sample_entries(M: int, N: int, count: int, seed: int):
    """Sampled (row, col) pairs: random ones plus the four corners and the
    first/last row and column of each edge tile."""
    rng = np.random.default_rng(seed)
    r = list(rng.integers(0, M, count))
    c = list(rng.integers(0, N, count))
    for rr in (0, M - 1):
        for cc in (0, N - 1):
            r.append(rr)
            c.append(cc)
    return np.array(r, dtype=np.int64), np.array(c, dtype=np.int64)
