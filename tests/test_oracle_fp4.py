"""Pins for the oracle's 4-bit block-scaled formats (CPU only): the E2M1 codec,
the MXFP4 (E8M0 scale per 32) and NVFP4 (E4M3 scale per 16) quantizers, and the
4-bit block-scaled GEMM ("GPU GEMM part 4: tcgen05 & Blackwell", sections 6.1,
6.3 and 7.1).

The E2M1 value table is checked against a generic minifloat grid built from
the format's field widths; the same builder, given E4M3's widths, reproduces
torch's float8_e4m3fn table, which pins the builder itself.  The encoder is
checked against brute-force nearest-value search with ties to the even code.
"""
import numpy as np
import pytest
import torch

from fine_grained_fp8_persistent_gb300 import inputs

MX, NV = 0, 1


def minifloat_values(exp_bits, man_bits, bias, fn_nan):
    """Value of every non-negative code of a sign/exponent/mantissa format
    (subnormals at exponent field 0); fn_nan: the all-ones code is NaN."""
    vals = []
    for c in range(1 << (exp_bits + man_bits)):
        e, m = c >> man_bits, c & ((1 << man_bits) - 1)
        if fn_nan and c == (1 << (exp_bits + man_bits)) - 1:
            vals.append(float("nan"))
        elif e == 0:
            vals.append(m / (1 << man_bits) * 2.0 ** (1 - bias))
        else:
            vals.append((1 + m / (1 << man_bits)) * 2.0 ** (e - bias))
    return np.array(vals)


def test_grid_builder_reproduces_torch_e4m3():
    ref = torch.arange(128, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = minifloat_values(4, 3, 7, fn_nan=True)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(ref[~np.isnan(ref)], got[~np.isnan(got)])


def test_e2m1_table(oracle):
    pos = minifloat_values(2, 1, 1, fn_nan=False)
    assert pos.max() == 6.0                                     # largest E2M1 value
    dec = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert np.array_equal(dec[:8], pos)
    assert np.array_equal(dec[8:], -pos)
    assert np.signbit(dec[8]) and not np.signbit(dec[0])         # code 8 is -0


def test_e2m1_values_lie_on_the_e4m3_grid(oracle):
    v = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert np.array_equal(oracle.e4m3_decode(oracle.e4m3_encode(v)), v)


def _brute_force_e2m1(v):
    grid = minifloat_values(2, 1, 1, fn_nan=False)              # codes 0..7
    a = np.minimum(np.abs(v), 6.0)
    d = np.abs(a[:, None] - grid[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # ties: the even code
    code = np.where(cand.sum(axis=1) > 1, np.argmax(cand & (np.arange(8) % 2 == 0), axis=1), np.argmax(cand, axis=1))
    return (code | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def test_e2m1_encode_is_nearest_even(oracle):
    rng = np.random.default_rng(0)
    grid = minifloat_values(2, 1, 1, fn_nan=False)
    mids = (grid[1:] + grid[:-1]) / 2
    v = np.concatenate([rng.uniform(-8, 8, 50000), np.exp(rng.uniform(-8, 3, 50000)) * rng.choice([-1, 1], 50000),
                        mids, -mids, grid, -grid, [7.0, 1e9, -1e9, 0.0, -0.0, 6.0, 5.999999]])
    assert np.array_equal(oracle.e2m1_encode(v), _brute_force_e2m1(v))


def test_e2m1_round_trip(oracle):
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(oracle.e2m1_encode(oracle.e2m1_decode(codes)), codes)


def _groups(oracle, x, fmt):
    q, sf = oracle.quantize_fp4(x, fmt)
    R, K = x.shape
    s = oracle.fp4_scales(sf, R, K, fmt)
    codes = oracle.fp4_unpack(q)
    return q, sf, s, codes


@pytest.mark.parametrize("fmt", [MX, NV])
def test_packing_low_nibble_first(oracle, fmt):
    x = np.zeros((2, 64), np.float32)
    x[0, 1] = 1.0       # odd element -> high nibble of byte 0
    x[1, 4] = -1.0      # even element -> low nibble of byte 2
    q, sf = oracle.quantize_fp4(x, fmt)
    assert q[0, 0] >> 4 != 0 and q[0, 0] & 0xF == 0
    assert q[1, 2] & 0xF != 0 and q[1, 2] >> 4 == 0
    assert np.count_nonzero(q) == 2


def test_mx_scale_rounds_up(oracle):
    """E8M0 exponent ceil(log2(amax/6)): the largest element of a group lands in
    (3, 6] after scaling, so nothing saturates; a floor would leave it in [4, 8)."""
    x = inputs.normal_bf16((64, 512), 3, outliers=True).float().numpy()
    q, sf, s, codes = _groups(oracle, x, MX)
    amax = np.abs(x).reshape(64, -1, 32).max(axis=2)
    r = amax / s
    assert np.all((r > 3) & (r <= 6))
    deq = oracle.dequantize_fp4(q, sf, MX)
    # no saturation: every element within half a step of the grid (0.25 s below 2 s, then s/2, then s)
    err = np.abs(deq - x) / np.repeat(s, 32, axis=1)
    half = np.where(np.abs(x) / np.repeat(s, 32, axis=1) < 2, 0.25, np.where(np.abs(x) / np.repeat(s, 32, axis=1) < 4, 0.5, 1.0))
    assert np.all(err <= half)


def test_mx_power_of_two_rescale_moves_only_the_scale(oracle):
    x = inputs.normal_bf16((8, 256), 4, outliers=True).float().numpy()
    q, sf = oracle.quantize_fp4(x, MX)
    q2, sf2 = oracle.quantize_fp4(x * np.float32(2.0 ** 5), MX)
    assert np.array_equal(q, q2)
    b, b2 = sf.view(np.uint8), sf2.view(np.uint8)
    used = b != 0
    assert np.array_equal(b2[used], b[used] + 5) and np.array_equal(b2[~used], b[~used])


@pytest.mark.parametrize("fmt", [MX, NV])
def test_zero_group_and_table_layout(oracle, fmt):
    """A zero group has scale 1 and zero codes; the scale of group g of row r is
    byte g % 4 of word (g // 4, r); bytes past the last group and rows past R are 0."""
    sv = oracle.fp4_vec(fmt)
    R, K = 5, 3 * 64                       # an odd number of groups for MX (6), 12 for NV
    ng = K // sv
    x = np.zeros((R, K), np.float32)
    for r in range(R):
        for g in range(ng):
            if (r + g) % 3:
                x[r, g * sv] = 2.0 ** ((r + 2 * g) % 7)     # distinct group maxima
    q, sf, s, codes = _groups(oracle, x, fmt)
    b = sf.view(np.uint8).reshape(sf.shape[0], sf.shape[1], 4)
    one = 127 if fmt == MX else int(oracle.e4m3_encode([1.0])[0])
    for r in range(R):
        for g in range(ng):
            byte = b[g // 4, r, g % 4]
            if (r + g) % 3 == 0:
                assert byte == one and not codes[r, g * sv:(g + 1) * sv].any()
            elif fmt == MX:     # power-of-two scale: the group maximum is exact
                assert oracle.e2m1_decode(codes[r, g * sv:g * sv + 1])[0] * s[r, g] == x[r, g * sv]
            else:               # E4M3 scale of amax / 6: distinct maxima pin the byte's place
                t = x[r, g * sv] / 6.0
                assert abs(s[r, g] - t) <= 2.0 ** -4 * t
    assert not b[:, R:, :].any()
    for g in range(ng, 4 * sf.shape[0]):
        assert not b[g // 4, :, g % 4].any()


def test_nv_scale_and_codes(oracle):
    """NVFP4: the scale is amax / 6 rounded to E4M3 (within half an E4M3 step);
    the group's largest element takes the code of 6; every other element lies
    within half an E2M1 step (times the scale) of its value unless it saturates."""
    x = inputs.normal_bf16((64, 512), 5, outliers=True).float().numpy()
    q, sf, s, codes = _groups(oracle, x, NV)
    amax = np.abs(x).reshape(64, -1, 16).max(axis=2).astype(np.float64)
    assert np.all(np.abs(s - amax / 6) <= 2.0 ** -4 * amax / 6 + 2.0 ** -10)
    vals = oracle.e2m1_decode(codes).reshape(64, -1, 16)
    arg = np.abs(x).reshape(64, -1, 16).argmax(axis=2)
    top = np.take_along_axis(np.abs(vals), arg[..., None], axis=2)[..., 0]
    assert np.all(top == 6.0)
    t = np.abs(x) / np.repeat(s, 16, axis=1)
    half = np.where(t < 2, 0.25, np.where(t < 4, 0.5, 1.0)) * (1 + 2.0 ** -20)
    err = np.abs(oracle.e2m1_decode(codes) - x / np.repeat(s, 16, axis=1))
    assert np.all((err <= half) | (t > 6))


def _fp4_ints(oracle, shape, rng):
    grid = minifloat_values(2, 1, 1, fn_nan=False)
    v = rng.choice(grid, size=shape) * rng.choice([-1.0, 1.0], size=shape)
    return v


def _pack(oracle, v, scales, fmt):
    """Quantize values that are exact grid values times given power-of-two group scales."""
    sv = oracle.fp4_vec(fmt)
    x = (v * np.repeat(scales, sv, axis=1)).astype(np.float32)
    return oracle.quantize_fp4(x, fmt)


@pytest.mark.parametrize("fmt", [MX, NV])
@pytest.mark.parametrize("impl", ["gemm_fp4", "gemm_fp4_dequant"])
def test_fp4_gemm_exact_small_values(oracle, fmt, impl):
    """Grid values (multiples of 1/2 up to 6) with power-of-two scales: every
    product and sum is exact in fp64, so D equals the exact product."""
    rng = np.random.default_rng(7)
    M, N, K = 20, 24, 256
    sv = oracle.fp4_vec(fmt)
    a = _fp4_ints(oracle, (M, K), rng)
    b = _fp4_ints(oracle, (N, K), rng)
    a[:, ::sv] = 6.0          # every group reaches 6, so its scale is exactly the given one
    b[:, ::sv] = -6.0
    sa = np.ldexp(1.0, rng.integers(-3, 4, (M, K // sv)))
    sb = np.ldexp(1.0, rng.integers(-3, 4, (N, K // sv)))
    aq, sfa = _pack(oracle, a, sa, fmt)
    bq, sfb = _pack(oracle, b, sb, fmt)
    D = getattr(oracle, impl)(aq, sfa, bq, sfb, fmt)
    expect = (a * np.repeat(sa, sv, axis=1)) @ (b * np.repeat(sb, sv, axis=1)).T
    assert np.array_equal(D, expect)


@pytest.mark.parametrize("fmt", [MX, NV])
def test_fp4_identity_gives_dequantized_a(oracle, fmt):
    M, K = 9, 128
    x = inputs.normal_bf16((M, K), 8, outliers=True).float().numpy()
    aq, sfa = oracle.quantize_fp4(x, fmt)
    # B = I written by hand: code 2 (1.0) on the diagonal, every scale 1
    # (an NVFP4 quantizer would scale 1.0 by e4m3(1/6) and not return exactly 1)
    bq = np.zeros((K, K // 2), np.uint8)
    for n in range(K):
        bq[n, n // 2] = 2 << (4 * (n % 2))
    shape, dt = oracle.fp4_sf_shape(K, K, fmt)
    sfb = np.zeros(shape, dt)
    one = 127 if fmt == MX else int(oracle.e4m3_encode([1.0])[0])
    ng = K // oracle.fp4_vec(fmt)
    sb = sfb.view(np.uint8).reshape(shape[0], shape[1], 4)
    for g in range(ng):
        sb[g // 4, :K, g % 4] = one
    assert np.array_equal(oracle.dequantize_fp4(bq, sfb, fmt), np.eye(K))
    assert np.array_equal(oracle.gemm_fp4(aq, sfa, bq, sfb, fmt), oracle.dequantize_fp4(aq, sfa, fmt))


@pytest.mark.parametrize("fmt", [MX, NV])
def test_fp4_dequant_form_equals_triple_loop(oracle, fmt):
    M, N, K = 33, 48, 320
    x = inputs.normal_bf16((M, K), 9, outliers=True).float().numpy()
    w = inputs.normal_bf16((N, K), 10, outliers=True).float().numpy()
    aq, sfa = oracle.quantize_fp4(x, fmt)
    bq, sfb = oracle.quantize_fp4(w, fmt)
    D = oracle.gemm_fp4(aq, sfa, bq, sfb, fmt)
    assert np.allclose(oracle.gemm_fp4_dequant(aq, sfa, bq, sfb, fmt), D, rtol=0, atol=1e-13 * np.abs(D).max())
    # the non-square shape makes a transposed operand fail; a swapped scale index too
    assert not np.allclose(oracle.gemm_fp4(aq, sfa, bq, sfb, fmt)[:, ::-1], D)


def test_fp4_scale_linearity_mx(oracle):
    """Adding k to every E8M0 byte of A multiplies D by 2^k exactly."""
    M, N, K = 12, 16, 256
    x = inputs.normal_bf16((M, K), 11, outliers=True).float().numpy()
    w = inputs.normal_bf16((N, K), 12, outliers=True).float().numpy()
    aq, sfa = oracle.quantize_fp4(x, MX)
    bq, sfb = oracle.quantize_fp4(w, MX)
    D = oracle.gemm_fp4(aq, sfa, bq, sfb, MX)
    b = sfa.view(np.uint8).copy()
    b[b != 0] += 3
    assert np.array_equal(oracle.gemm_fp4(aq, b.view(np.int32), bq, sfb, MX), D * 8.0)
