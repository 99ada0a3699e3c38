"""Pins for the oracle's E4M3 codec (CPU only).

The codec is pinned to (a) the facts the DeepGEMM page prints about E4M3
(largest value 448, smallest subnormal 2^-9, products exact in FP32) and
(b) an independent library routine: torch's float8_e4m3fn conversion, which
rounds to nearest-even for in-range values.
"""
import math

import numpy as np
import pytest
import torch

ALL = np.arange(256, dtype=np.uint8)


def test_decode_page_facts(oracle, facts):
    v = oracle.e4m3_decode(ALL)
    finite = v[np.isfinite(v)]
    assert finite.max() == facts["e4m3_max"]["value"]
    assert finite.min() == -facts["e4m3_max"]["value"]
    pos = finite[finite > 0]
    assert pos.min() == 2.0 ** facts["e4m3_min_subnormal_log2"]["value"]
    # exactly one NaN code per sign, no infinities ("fn" variant)
    assert set(np.flatnonzero(np.isnan(v)).tolist()) == {0x7F, 0xFF}
    assert not np.isinf(v).any()
    # 126 distinct positive finite values, symmetric around zero
    assert len(set(pos.tolist())) == 126
    assert np.array_equal(v[:127], -v[128:255])


def test_decode_matches_torch_float8(oracle):
    ref = torch.tensor(ALL).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(ALL)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(np.where(both_nan, 0, ref), np.where(both_nan, 0, got))
    # sign of zero
    assert math.copysign(1.0, got[0x80]) == -1.0


def _torch_encode(values_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(values_f32.astype(np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_encode_matches_torch_random(oracle):
    rng = np.random.default_rng(7)
    # log-uniform magnitudes across the whole E4M3 range, both signs, below the
    # saturation threshold where torch and satfinite agree
    mags = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(463.0), size=200_000))
    vals = (mags * rng.choice([-1.0, 1.0], size=mags.size)).astype(np.float32)
    got = oracle.e4m3_encode(vals.astype(np.float64))
    assert np.array_equal(got, _torch_encode(vals))


def test_encode_midpoints_tie_to_even(oracle):
    """Exact midpoints between adjacent codes must round to the even code."""
    v = oracle.e4m3_decode(ALL[:0x7F])            # 0 .. 448
    mids = ((v[:-1] + v[1:]) / 2.0).astype(np.float32)
    got = oracle.e4m3_encode(mids.astype(np.float64))
    assert np.array_equal(got, _torch_encode(mids))
    assert np.all(got % 2 == 0)                   # even mantissa LSB


def test_encode_roundtrip_all_codes(oracle):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = oracle.e4m3_encode(oracle.e4m3_decode(codes))
    assert np.array_equal(back, codes)


def test_encode_saturates(oracle, facts):
    big = facts["e4m3_max"]["value"]
    cases = [(464.0, 0x7E), (1e6, 0x7E), (float("inf"), 0x7E), (-float("inf"), 0xFE),
             (-1e30, 0xFE), (448.0, 0x7E), (460.0, 0x7E), (-0.0, 0x80), (0.0, 0x00),
             (2.0 ** -10, 0x00), (-(2.0 ** -10), 0x80), (2.0 ** -10 * 1.0001, 0x01)]
    got = oracle.e4m3_encode(np.array([c[0] for c in cases]))
    assert got.tolist() == [c[1] for c in cases]
    assert oracle.e4m3_decode(np.array([0x7E]))[0] == big


def test_products_exact_in_fp32(oracle, facts):
    """DeepGEMM page: an E4M3 x E4M3 product needs <= 8 significant bits and is
    exact in FP32 (24-bit significand)."""
    v = oracle.e4m3_decode(ALL)
    v = v[np.isfinite(v)]
    prod64 = np.outer(v, v)
    prod32 = np.outer(v.astype(np.float32), v.astype(np.float32))
    assert np.array_equal(prod32.astype(np.float64), prod64)
    # significant bits of every nonzero product
    nz = prod64[prod64 != 0]
    m, _ = np.frexp(np.abs(nz))
    bits = np.zeros(nz.shape, dtype=np.int64)
    mm = m.copy()
    for b in range(1, 30):
        frac = mm * 2.0 ** b
        done = (frac == np.floor(frac)) & (bits == 0)
        bits[done] = b
    assert bits.max() <= facts["e4m3_product_max_significant_bits"]["value"]
