"""Pins for the oracle's 1x128 / 128x128 quantizers (CPU only).

Pinned to the DeepGEMM page's worked outlier example, to the format's exact
rounding bound, to invariants of the scale definition (amax maps to the top of
the E4M3 range; power-of-two rescaling only moves the scale), and to a
cross-check between the two quantizers (a 128x128 block scale is the largest
of the 1x128 scales of its rows).
"""
import numpy as np
import pytest

from fine_grained_fp8_persistent_gb300 import inputs

F32, UE = 0, 1


def _bf16_values(shape, seed, outliers=True):
    return inputs.normal_bf16(shape, seed, outliers=outliers).float().numpy()


def _scales_1x128(oracle, sf, fmt, M, K):
    """(M, K/128) array of the scales held in an activation table."""
    nkb = K // 128
    ld = oracle.align4(M)
    if fmt == F32:
        return sf.reshape(nkb, ld)[:, :M].T.astype(np.float64)
    b = sf.view(np.uint8).reshape(-1)
    out = np.empty((M, nkb))
    for kb in range(nkb):
        out[:, kb] = np.ldexp(1.0, b[((kb // 4) * ld + np.arange(M)) * 4 + kb % 4].astype(np.int64) - 127)
    return out


def _spacing(mag):
    """E4M3 grid spacing at magnitude mag (format definition: 3 mantissa bits,
    subnormal spacing 2^-9 below 2^-6)."""
    mag = np.asarray(mag, dtype=np.float64)
    e = np.floor(np.log2(np.maximum(mag, 2.0 ** -6)))
    return np.where(mag < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))


def test_worked_outlier_example(oracle, facts):
    ex = facts["per_tensor_outlier_example"]
    rng = np.random.default_rng(0)
    x = rng.uniform(-ex["small_bound"], ex["small_bound"], size=128).astype(np.float32)
    x[77] = ex["outlier"]
    q, sf = oracle.quantize_1x128(x[None, :], F32)
    s = float(sf.reshape(-1)[0])
    assert abs(s - ex["scale_printed"]) < 0.0005                      # 40/448 ~ 0.089
    assert s == np.float32(ex["outlier"]) / np.float32(448.0)
    dq = oracle.e4m3_decode(q[0])
    assert dq[77] == 448.0
    small = np.abs(np.delete(dq, 77))
    # small values land near 0.1/0.089 ~ 1.1 at most
    assert small.max() <= 1.125 and abs(small.max() - ex["small_quantized_magnitude_printed"]) < 0.05
    # the outlier degrades the small values: their error is larger than when the
    # same 127 values form a group of their own
    small_x = np.delete(x, 77).astype(np.float64)
    err_out = np.abs(np.delete(dq, 77) * s - small_x).mean()
    q2, sf2 = oracle.quantize_1x128(np.delete(np.append(x, np.float32(0.0)), 77)[None, :], F32)
    err_own = np.abs(oracle.e4m3_decode(q2[0])[:127] * float(sf2.reshape(-1)[0]) - small_x).mean()
    assert err_out > err_own


@pytest.mark.parametrize("fmt", [F32, UE])
def test_rounding_bound_and_range(oracle, fmt):
    M, K = 37, 640
    x = _bf16_values((M, K), seed=3)
    q, sf = oracle.quantize_1x128(x, fmt)
    s = np.repeat(_scales_1x128(oracle, sf, fmt, M, K), 128, axis=1)
    dq = oracle.e4m3_decode(q)
    assert np.isfinite(dq).all() and np.abs(dq).max() <= 448.0
    target = x.astype(np.float64) / s
    if fmt == F32:
        # the FP32 quotient is what gets rounded: within one FP32 ulp of the exact one
        assert np.all(np.abs(target - (x / s.astype(np.float32)).astype(np.float64)) <= np.abs(target) * 2.0 ** -23)
        target = (x / s.astype(np.float32)).astype(np.float64)
    err = np.abs(target - dq)
    assert np.all(err <= _spacing(np.abs(dq)) / 2.0 + 1e-300)
    assert np.array_equal(np.signbit(dq[x != 0]), np.signbit(x[x != 0]))


def test_fp32_amax_maps_to_448(oracle):
    M, K = 64, 512
    x = _bf16_values((M, K), seed=5)
    q, sf = oracle.quantize_1x128(x, F32)
    dq = np.abs(oracle.e4m3_decode(q)).reshape(M, K // 128, 128)
    amax_pos = np.abs(x).reshape(M, K // 128, 128).argmax(axis=2)
    top = np.take_along_axis(dq, amax_pos[..., None], axis=2)[..., 0]
    assert np.all(top == 448.0)
    s = _scales_1x128(oracle, sf, F32, M, K)
    amax = np.abs(x).reshape(M, K // 128, 128).max(axis=2)
    # s * 448 reproduces amax to FP32 rounding
    assert np.all(np.abs(s * 448.0 - amax) <= amax * 2.0 ** -22)


def test_ue8m0_exponent_is_minimal(oracle):
    M, K = 50, 1024
    x = _bf16_values((M, K), seed=9)
    q, sf = oracle.quantize_1x128(x, UE)
    s = _scales_1x128(oracle, sf, UE, M, K)
    amax = np.abs(x).reshape(M, K // 128, 128).max(axis=2).astype(np.float64)
    r = amax / s
    # power of two, no saturation, and the next smaller power would saturate
    assert np.all(np.log2(s) == np.round(np.log2(s)))
    assert np.all(r <= 448.0) and np.all(r > 224.0)
    dq = np.abs(oracle.e4m3_decode(q))
    assert dq.max() <= 448.0


def test_ue8m0_unused_bytes_zero(oracle):
    M, K = 8, 128 * 6        # 6 K-blocks -> 2 packed words, last word half used
    x = _bf16_values((M, K), seed=1)
    _, sf = oracle.quantize_1x128(x, UE)
    assert sf.shape == (2, 8) and sf.dtype == np.int32
    b = sf.view(np.uint8).reshape(2, 8, 4)
    assert np.all(b[1, :, 2:] == 0)
    assert np.all(b[:, :, :2] != 0)


@pytest.mark.parametrize("fmt", [F32, UE])
def test_power_of_two_rescale_moves_only_the_scale(oracle, fmt):
    M, K = 20, 384
    x = _bf16_values((M, K), seed=11)
    q0, sf0 = oracle.quantize_1x128(x, fmt)
    q1, sf1 = oracle.quantize_1x128(x * np.float32(2.0 ** 5), fmt)
    assert np.array_equal(q0, q1)
    s0 = _scales_1x128(oracle, sf0, fmt, M, K)
    s1 = _scales_1x128(oracle, sf1, fmt, M, K)
    assert np.array_equal(s1, s0 * 32.0)


def test_outlier_contained_to_its_group(oracle):
    M, K = 4, 512
    x = _bf16_values((M, K), seed=2, outliers=False)
    q0, sf0 = oracle.quantize_1x128(x, F32)
    y = x.copy()
    y[2, 300] = 1000.0                      # K-block 2 of row 2
    q1, sf1 = oracle.quantize_1x128(y, F32)
    s0 = _scales_1x128(oracle, sf0, F32, M, K)
    s1 = _scales_1x128(oracle, sf1, F32, M, K)
    changed = np.argwhere(s0 != s1)
    assert changed.tolist() == [[2, 2]]
    mask = np.ones((M, K), bool)
    mask[2, 256:384] = False
    assert np.array_equal(q0[mask], q1[mask])


def test_zero_group(oracle):
    x = np.zeros((3, 256), np.float32)
    x[1, 200] = -0.0
    x[2, 130] = 1.5
    q, sf = oracle.quantize_1x128(x, F32)
    s = _scales_1x128(oracle, sf, F32, 3, 256)
    assert s[0, 0] == 1.0 and s[0, 1] == 1.0 and s[2, 0] == 1.0
    assert q[1, 200] == 0x80                # sign of zero kept
    assert np.count_nonzero(q[0]) == 0
    qu, sfu = oracle.quantize_1x128(x, UE)
    assert sfu.view(np.uint8).reshape(-1)[0] == 127


@pytest.mark.parametrize("fmt", [F32, UE])
def test_block_scale_is_max_of_row_scales(oracle, fmt):
    """A 128x128 block's scale is the largest 1x128 scale among its rows (both
    follow amax/448, which is monotone in amax), and the codes agree wherever a
    row's own amax equals the block amax."""
    N, K = 300, 512                             # ragged last n-block (44 rows)
    w = _bf16_values((N, K), seed=21)
    qb, sfb = oracle.quantize_128x128(w, fmt)
    _, sfr = oracle.quantize_1x128(w, fmt)
    row_s = _scales_1x128(oracle, sfr, fmt, N, K)
    nkb = K // 128
    if fmt == F32:
        blk = sfb.reshape((N + 127) // 128, nkb).astype(np.float64)
        per_row = np.repeat(blk, 128, axis=0)[:N]
    else:
        per_row = _scales_1x128(oracle, sfb.reshape(-1), UE, N, K)
    for nb in range((N + 127) // 128):
        rows = slice(nb * 128, min(N, nb * 128 + 128))
        assert np.array_equal(per_row[rows].max(axis=0), row_s[rows].max(axis=0))
        assert np.all(per_row[rows] == per_row[rows][0])
    qr, _ = oracle.quantize_1x128(w, fmt)
    same = np.repeat(per_row == row_s, 128, axis=1)
    assert np.array_equal(qb[0][same], qr[same])


def test_weight_groups_independent(oracle):
    G, N, K = 3, 256, 256
    w = _bf16_values((G, N, K), seed=4)
    q, sf = oracle.quantize_128x128(w, F32)
    for g in range(G):
        qg, sfg = oracle.quantize_128x128(w[g], F32)
        assert np.array_equal(qg[0], q[g]) and np.array_equal(sfg[0], sf[g])
