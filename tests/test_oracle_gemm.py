"""Pins for the oracle's GEMMs (CPU only).

The block-scaled NT GEMM is pinned to exact closed forms: small-integer
operands (exact in E4M3 and in the sum), identity and selection matrices
(D equals a dequantized, permuted A), scale linearity D(2^k A) = 2^k D, and the
per-K-block structure of the scales.  Non-square shapes make a transposed
operand fail.  The 16-bit GEMM is pinned to numpy's float64 matmul, an
independent library routine.  The grouped variants are pinned to the dense
GEMM on each expert's rows.

Every dense pin runs on both forms of the block-scaled GEMM: the per-K-block
triple loop (gemm_fp8) and dequantize-then-matmul (gemm_fp8_dequant), which the
full-size GPU parity tests use.
"""
import numpy as np
import pytest

from fine_grained_fp8_persistent_gb300 import inputs

F32, UE = 0, 1
ONE = 0x38       # E4M3 code of 1.0
IMPLS = ["gemm_fp8", "gemm_fp8_dequant"]


def _int_codes(oracle, shape, rng, lo=-4, hi=4):
    vals = rng.integers(lo, hi + 1, size=shape)
    return oracle.e4m3_encode(vals.astype(np.float64)), vals


def _sfa_table(oracle, scales, fmt):
    """Write an (M, nkb) array of scales into the activation table layout."""
    M, nkb = scales.shape
    ld = oracle.align4(M)
    if fmt == F32:
        t = np.zeros((nkb, ld), np.float32)
        t[:, :M] = scales.T
        return t
    t = np.zeros(((nkb + 3) // 4, ld, 4), np.uint8)
    e = np.log2(scales).astype(np.int64) + 127
    for kb in range(nkb):
        t[kb // 4, :M, kb % 4] = e[:, kb]
    return t.view(np.int32).reshape((nkb + 3) // 4, ld)


def _sfb_table(oracle, block_scales, N, fmt):
    """block_scales: (ceil(N/128), nkb) -> one expert's weight table."""
    nnb, nkb = block_scales.shape
    if fmt == F32:
        return block_scales.astype(np.float32)[None]
    per_row = np.repeat(block_scales, 128, axis=0)[:N]
    return _sfa_table(oracle, per_row, UE)[None]


def _pow2(rng, shape, lo=-3, hi=3):
    return np.ldexp(1.0, rng.integers(lo, hi + 1, size=shape))


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("fmt", [F32, UE])
def test_small_integer_exact(oracle, fmt, impl):
    rng = np.random.default_rng(1)
    M, N, K = 24, 40, 384
    a, av = _int_codes(oracle, (M, K), rng)
    b, bv = _int_codes(oracle, (N, K), rng)
    sa = np.ones((M, K // 128))
    sb = np.ones(((N + 127) // 128, K // 128))
    D = getattr(oracle, impl)(a, _sfa_table(oracle, sa, fmt), b, _sfb_table(oracle, sb, N, fmt), fmt)
    assert np.array_equal(D, (av @ bv.T).astype(np.float64))


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("fmt", [F32, UE])
def test_identity_gives_dequantized_a(oracle, fmt, impl):
    rng = np.random.default_rng(2)
    M, K = 30, 256
    a = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x11                  # no NaN codes
    sa = _pow2(rng, (M, K // 128))
    b = np.zeros((K, K), np.uint8)
    b[np.arange(K), np.arange(K)] = ONE
    sb = np.ones((K // 128 + (K % 128 > 0), K // 128))
    D = getattr(oracle, impl)(a, _sfa_table(oracle, sa, fmt), b, _sfb_table(oracle, sb, K, fmt), fmt)
    expect = oracle.e4m3_decode(a) * np.repeat(sa, 128, axis=1)
    assert np.array_equal(D, expect)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("fmt", [F32, UE])
def test_selection_matrix_permutes_and_applies_b_scales(oracle, fmt, impl):
    """B (N x K, N < K) selects column perm[n] of A: D[m,n] = A[m,perm[n]] with
    both scales of the K-block holding perm[n] and of the n-block of row n."""
    rng = np.random.default_rng(3)
    M, N, K = 17, 256, 512
    a, av = _int_codes(oracle, (M, K), rng, -8, 8)
    perm = rng.permutation(K)[:N]
    b = np.zeros((N, K), np.uint8)
    b[np.arange(N), perm] = ONE
    sa = _pow2(rng, (M, K // 128))
    sb = _pow2(rng, (N // 128, K // 128))
    D = getattr(oracle, impl)(a, _sfa_table(oracle, sa, fmt), b, _sfb_table(oracle, sb, N, fmt), fmt)
    n = np.arange(N)
    expect = av[:, perm] * sa[:, perm // 128] * sb[n // 128, perm // 128][None, :]
    assert np.array_equal(D, expect.astype(np.float64))


def _quantized_case(oracle, M, N, K, fmt, seed):
    x = inputs.normal_bf16((M, K), seed, outliers=True).float().numpy()
    w = inputs.normal_bf16((N, K), seed + 1, outliers=True).float().numpy()
    aq, sfa = oracle.quantize_1x128(x, fmt)
    bq, sfb = oracle.quantize_128x128(w, fmt)
    return aq, sfa, bq, sfb


@pytest.mark.parametrize("impl", IMPLS)
def test_scale_linearity(oracle, impl):
    M, N, K = 20, 256, 384
    aq, sfa, bq, sfb = _quantized_case(oracle, M, N, K, F32, 10)
    D = getattr(oracle, impl)(aq, sfa, bq, sfb, F32)
    D2 = getattr(oracle, impl)(aq, (sfa * np.float32(2.0 ** -7)).astype(np.float32), bq, sfb, F32)
    assert np.array_equal(D2, D * 2.0 ** -7)
    alpha = np.float32(0.3)
    D3 = getattr(oracle, impl)(aq, (sfa * alpha).astype(np.float32), bq, sfb, F32)
    # general alpha: the table itself was rounded to FP32, so compare with the
    # exactly scaled table's result
    assert np.allclose(D3, D * float(alpha), rtol=2e-7, atol=1e-6 * np.abs(D).max())
    # UE8M0: adding k to every exponent byte multiplies D by 2^k
    aqu, sfau, bqu, sfbu = _quantized_case(oracle, M, N, K, UE, 11)
    Du = getattr(oracle, impl)(aqu, sfau, bqu, sfbu, UE)
    b = sfau.view(np.uint8).copy()
    b[b != 0] += 3
    Du3 = getattr(oracle, impl)(aqu, b.view(np.int32), bqu, sfbu, UE)
    assert np.array_equal(Du3, Du * 8.0)


@pytest.mark.parametrize("impl", IMPLS)
def test_kblock_additivity(oracle, impl):
    """Doubling the A scale of one K-block adds exactly that block's
    contribution once more; the contribution is the GEMM restricted to it."""
    M, N, K = 12, 128, 512
    aq, sfa, bq, sfb = _quantized_case(oracle, M, N, K, F32, 20)
    D = getattr(oracle, impl)(aq, sfa, bq, sfb, F32)
    kb = 2
    sfa2 = sfa.copy()
    sfa2[kb] *= 2
    D2 = getattr(oracle, impl)(aq, sfa2, bq, sfb, F32)
    only = sfa.copy()
    only[np.arange(K // 128) != kb] = 0
    Dkb = getattr(oracle, impl)(aq, only, bq, sfb, F32)
    assert np.allclose(D2 - D, Dkb, rtol=1e-12, atol=1e-9 * np.abs(D).max())


def test_entries_match_full(oracle):
    M, N, K = 33, 256, 256
    for fmt in (F32, UE):
        aq, sfa, bq, sfb = _quantized_case(oracle, M, N, K, fmt, 30)
        D = oracle.gemm_fp8(aq, sfa, bq, sfb, fmt)
        rng = np.random.default_rng(0)
        r = rng.integers(0, M, 200)
        c = rng.integers(0, N, 200)
        assert np.array_equal(oracle.gemm_fp8_entries(aq, sfa, bq, sfb, fmt, r, c), D[r, c])


def test_f16_matches_numpy(oracle):
    import torch
    M, N, K = 50, 70, 300
    A = inputs.uniform_16bit((M, K), 1).float().numpy()
    B = inputs.uniform_16bit((N, K), 2).float().numpy()
    D = oracle.gemm_f16(A, B)
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    assert np.allclose(D, ref, rtol=1e-13, atol=1e-13)
    r = np.array([0, 49, 10])
    c = np.array([69, 0, 33])
    assert np.array_equal(oracle.gemm_f16_entries(A, B, r, c), D[r, c])
    assert np.allclose(oracle.gemm_f16_matmul(A, B), D, rtol=0, atol=1e-13 * np.abs(D).max())
    Ab = inputs.uniform_16bit((M, K), 3, dtype=torch.bfloat16).float().numpy()
    assert np.allclose(oracle.gemm_f16(Ab, B), Ab.astype(np.float64) @ B.astype(np.float64).T,
                       rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("fmt", [F32, UE])
def test_grouped_contiguous_is_dense_per_segment(oracle, fmt):
    G, N, K = 3, 128, 256
    counts = [70, 0, 130]
    m_idx, M = inputs.contiguous_layout(counts, 128)
    m_idx = m_idx.numpy()
    x = inputs.normal_bf16((M, K), 40, outliers=True).float().numpy()
    w = inputs.normal_bf16((G, N, K), 41, outliers=True).float().numpy()
    aq, sfa = oracle.quantize_1x128(x, fmt)
    bq, sfb = oracle.quantize_128x128(w, fmt)
    D, valid = oracle.grouped_contiguous(aq, sfa, bq, sfb, m_idx, fmt)
    assert np.array_equal(valid.any(axis=1), m_idx >= 0)
    Dfull = [oracle.gemm_fp8(aq, sfa, bq[g], sfb[g:g + 1], fmt) for g in range(G)]
    for m in range(M):
        if m_idx[m] >= 0:
            assert np.array_equal(D[m], Dfull[m_idx[m]][m])


@pytest.mark.parametrize("fmt", [F32, UE])
def test_grouped_masked_is_dense_per_expert(oracle, fmt):
    G, Mmax, N, K = 4, 64, 128, 256
    masked = np.array([0, 64, 17, 1], np.int32)
    x = inputs.normal_bf16((G, Mmax, K), 50, outliers=True).float().numpy()
    w = inputs.normal_bf16((G, N, K), 51, outliers=True).float().numpy()
    qs = [oracle.quantize_1x128(x[g], fmt) for g in range(G)]
    aq = np.stack([q[0] for q in qs])
    sfa = np.stack([q[1] for q in qs])
    bq, sfb = oracle.quantize_128x128(w, fmt)
    D, valid = oracle.grouped_masked(aq, sfa, bq, sfb, masked, fmt)
    for g in range(G):
        assert np.array_equal(valid[g].any(axis=1), np.arange(Mmax) < masked[g])
        Dg = oracle.gemm_fp8(aq[g], sfa[g], bq[g], sfb[g:g + 1], fmt)
        assert np.array_equal(D[g, :masked[g]], Dg[:masked[g]])


@pytest.mark.parametrize("fmt", [F32, UE])
def test_dequant_form_equals_triple_loop(oracle, fmt):
    """Both forms on quantized outlier data: equal up to fp64 summation order."""
    M, N, K = 70, 300, 640
    aq, sfa, bq, sfb = _quantized_case(oracle, M, N, K, fmt, 60)
    D = oracle.gemm_fp8(aq, sfa, bq, sfb, fmt)
    assert np.allclose(oracle.gemm_fp8_dequant(aq, sfa, bq, sfb, fmt), D, rtol=0, atol=1e-13 * np.abs(D).max())


@pytest.mark.parametrize("fmt", [F32, UE])
def test_dequantize_round_trip_bound(oracle, fmt):
    """dequant(quant(x)) is within half an E4M3 step of x: 2^-4 relative in the
    normal range (3 mantissa bits), s * 2^-10 among subnormals (step 2^-9 s).
    The quotient x / s is rounded to FP32 before it is encoded, which can move
    it onto a midpoint: a 2^-20 relative slack covers that rounding."""
    M, N, K = 40, 200, 384
    x = inputs.normal_bf16((M, K), 61, outliers=True).float().numpy().astype(np.float64)
    w = inputs.normal_bf16((N, K), 62, outliers=True).float().numpy().astype(np.float64)
    aq, sfa = oracle.quantize_1x128(x, fmt)
    bq, sfb = oracle.quantize_128x128(w, fmt)
    sa = np.repeat(oracle.a_scales(sfa, M, K, fmt), 128, axis=1)
    sb = np.repeat(oracle.b_scales(sfb, 1, N, K, fmt)[0], 128, axis=1)
    for v, vq, s in ((x, oracle.dequantize_a(aq, sfa, fmt), sa), (w, oracle.dequantize_b(bq, sfb, fmt)[0], sb)):
        assert np.all(np.abs(vq - v) <= np.maximum(2.0 ** -4 * np.abs(v), s * 2.0 ** -10) * (1 + 2.0 ** -20))


@pytest.mark.parametrize("fmt", [F32, UE])
def test_grouped_dequant_forms(oracle, fmt):
    G, N, K = 3, 128, 256
    m_idx, M = inputs.contiguous_layout([70, 0, 130], 128)
    m_idx = m_idx.numpy()
    x = inputs.normal_bf16((M, K), 63, outliers=True).float().numpy()
    w = inputs.normal_bf16((G, N, K), 64, outliers=True).float().numpy()
    aq, sfa = oracle.quantize_1x128(x, fmt)
    bq, sfb = oracle.quantize_128x128(w, fmt)
    D, valid = oracle.grouped_contiguous(aq, sfa, bq, sfb, m_idx, fmt)
    D2, valid2 = oracle.grouped_contiguous_dequant(aq, sfa, bq, sfb, m_idx, fmt)
    assert np.array_equal(valid, valid2)
    assert np.allclose(D2, D, rtol=0, atol=1e-13 * np.abs(D).max())
    Mmax = 64
    masked = np.array([0, 64, 17], np.int32)
    xm = inputs.normal_bf16((G, Mmax, K), 65, outliers=True).float().numpy()
    qs = [oracle.quantize_1x128(xm[g], fmt) for g in range(G)]
    aqm, sfam = np.stack([q[0] for q in qs]), np.stack([q[1] for q in qs])
    D, valid = oracle.grouped_masked(aqm, sfam, bq, sfb, masked, fmt)
    D2, valid2 = oracle.grouped_masked_dequant(aqm, sfam, bq, sfb, masked, fmt)
    assert np.array_equal(valid, valid2)
    assert np.allclose(D2, D, rtol=0, atol=1e-13 * np.abs(D).max())
