"""GPU parity of the 4-bit block-scaled path (MXFP4 and NVFP4) against the oracle:
quantize_fp4 bit-exact (packed codes and scale words), and the 4-bit GEMM
within the GEMM tolerance on every tile, on ragged shapes and at full size."""
import functools

import numpy as np
import pytest
import torch

from fine_grained_fp8_persistent_gb300 import inputs
from parity import gemm_close, nan_filled, sample_entries, to_dev

pytestmark = pytest.mark.gpu
FMTS = [0, 1]          # MXFP4, NVFP4


@pytest.fixture(scope="module")
def fg():
    from fine_grained_fp8_persistent_gb300 import binding
    return binding


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _special_rows(K):
    """Rows with exact zeros, -0, values that round onto E2M1 midpoints, tiny
    values, and one huge outlier per group."""
    rows = []
    z = torch.zeros(K)
    rows.append(z.clone())                                   # an all-zero row
    r = torch.zeros(K)
    r[::2] = -0.0
    r[1::7] = 0.25
    r[3::11] = -1.75
    rows.append(r)
    rows.append(torch.full((K,), 3.0e-3))                   # tiny groups
    o = torch.randn(K, generator=torch.Generator().manual_seed(3))
    o[::16] = 3.0e4                                          # an outlier in every group
    rows.append(o)
    rows.append(torch.linspace(-6.5, 6.5, K))               # across the whole E2M1 range
    return torch.stack(rows).to(torch.bfloat16)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("R,K", [(128, 256), (37, 448), (300, 7168), (1, 64), (4096, 7168)])
def test_quantize_fp4_bit_exact(fg, dev, oracle, fmt, R, K):
    x = inputs.normal_bf16((R, K), 20 + R + K, outliers=True)
    if R >= 8:
        x[:5] = _special_rows(K)
    xq, sf = fg.quantize_fp4(x.to(dev), fmt)
    oq, osf = oracle.quantize_fp4(x.float().numpy(), fmt)
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), oq), "E2M1 codes differ"
    assert np.array_equal(sf.cpu().numpy(), osf), "scale words differ"


def _every_value_under_every_scale():
    """NVFP4 groups covering every (bf16 value, E4M3 scale) pair a group can hold:
    for each positive finite E4M3 scale s, groups led by amax = 6 s (whose scale
    is exactly s) followed by every bf16 value of magnitude <= amax, both signs
    (zeros, subnormals and values exactly on the E2M1 rounding midpoints
    included).  Rows of 4096 elements, padded with zeros."""
    import oracle
    bits = np.arange(0x8000, dtype=np.uint32)
    pos = (bits << 16).view(np.float32)
    pos = pos[np.isfinite(pos)]
    scales = oracle.e4m3_decode(np.arange(1, 127, dtype=np.uint8))
    groups = []
    for sv in scales:
        amax = np.float32(6.0 * sv)
        assert float(amax) == 6.0 * float(sv)          # exact in bf16 and FP32
        vals = pos[pos <= amax]
        vals = np.concatenate([vals, -vals])
        vals = np.concatenate([vals, np.zeros((-len(vals)) % 15, np.float32)])
        body = vals.reshape(-1, 15)
        groups.append(np.concatenate([np.full((len(body), 1), amax, np.float32), body], axis=1))
    g = np.concatenate(groups).reshape(-1)
    g = np.concatenate([g, np.zeros((-len(g)) % 4096, np.float32)])
    x = torch.from_numpy(g.reshape(-1, 4096)).to(torch.bfloat16)
    assert torch.equal(x.float(), torch.from_numpy(g.reshape(-1, 4096)))   # every value is a bf16 value
    return x


def test_quantize_nvfp4_every_value_and_scale(fg, dev, oracle):
    """NVFP4 codes of every bf16 value under every E4M3 scale, bit-exact against
    the oracle's FP32 division (the kernel decides them without one)."""
    x = _every_value_under_every_scale()
    xq, sf = fg.quantize_fp4(x.to(dev), 1)
    oq, osf = oracle.quantize_fp4(x.float().numpy(), 1)
    torch.cuda.synchronize()
    assert np.array_equal(sf.cpu().numpy(), osf), "scale words differ"
    got = xq.cpu().numpy()
    bad = np.nonzero(got != oq)
    assert bad[0].size == 0, f"{bad[0].size} code bytes differ, first at {bad[0][0]}, {bad[1][0]}"


@functools.lru_cache(maxsize=6)
def _fp4_case(M, N, K, fmt, seed):
    import oracle
    x = inputs.normal_bf16((M, K), seed, outliers=True).float().numpy()
    w = inputs.normal_bf16((N, K), seed + 1, outliers=True).float().numpy()
    aq, sfa = oracle.quantize_fp4(x, fmt)
    bq, sfb = oracle.quantize_fp4(w, fmt)
    return aq, sfa, bq, sfb


def _run(fg, dev, case, fmt, M, N):
    aq, sfa, bq, sfb = case
    out = nan_filled((M, N), dev)
    fg.gemm_fp4_blockscaled(to_dev(aq, dev), to_dev(sfa, dev), to_dev(bq, dev), to_dev(sfb, dev), fmt, out=out)
    rc, bits = fg.check_status()
    assert rc == 0, (rc, hex(bits), fg.last_error())
    return out


FP4_TILES = ["2x256", "2x128", "1x128"]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("tile", FP4_TILES)
@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (200, 288, 768), (1, 32, 256), (384, 512, 1024),
                                   (130, 96, 512)])
def test_fp4_gemm_every_tile(fg, dev, oracle, monkeypatch, fmt, tile, M, N, K):
    """Every forced tile; K = 768 leaves a short last pipeline unit, N = 288 and 96
    ragged last N tiles, M = 1 and 130 ragged M tiles."""
    monkeypatch.setenv("FGF8_FORCE_TILE", tile)
    case = _fp4_case(M, N, K, fmt, 700 + M + N)
    out = _run(fg, dev, case, fmt, M, N)
    assert fg.last_tile() == f"{'mxf4' if fmt == 0 else 'nvf4'} dense {tile}"
    gemm_close(out.float().cpu().numpy(), oracle.gemm_fp4(*case, fmt), f"fp4 fmt{fmt} {tile} {M}x{N}x{K}")


@pytest.mark.parametrize("fmt", FMTS)
def test_fp4_gemm_long_k(fg, dev, oracle, fmt):
    """K = 16384: 64 K blocks of 256 elements, scale groups wrapping the ring many times."""
    M, N, K = 130, 288, 16384
    case = _fp4_case(M, N, K, fmt, 61)
    out = _run(fg, dev, case, fmt, M, N)
    gemm_close(out.float().cpu().numpy(), oracle.gemm_fp4(*case, fmt), f"fp4 long K fmt{fmt}")


@pytest.mark.parametrize("fmt", FMTS)
def test_fp4_gemm_full_size(fg, dev, oracle, fmt):
    """M = 4096, N = K = 7168 in the launch configuration the library picks: every
    element against the oracle's dequantize-then-matmul form, plus sampled
    entries of its term-by-term triple loop."""
    M = 4096
    N = K = 7168
    case = _fp4_case(M, N, K, fmt, 11)
    out = _run(fg, dev, case, fmt, M, N)
    got = out.float().cpu().numpy()
    gemm_close(got, oracle.gemm_fp4_dequant(*case, fmt), f"fp4 full fmt{fmt}")
    r, c = sample_entries(M, N, 64, seed=5)
    aq, sfa, bq, sfb = case
    loop = np.array([oracle.gemm_fp4(aq[rr:rr + 1], _row_sf(oracle, sfa, rr, M, K, fmt),
                                     bq[cc:cc + 1], _row_sf(oracle, sfb, cc, N, K, fmt), fmt)[0, 0]
                     for rr, cc in zip(r, c)])
    gemm_close(got[r, c], loop, f"fp4 full fmt{fmt} (triple loop)")


@pytest.mark.parametrize("fmt", FMTS)
def test_fp4_gemm_full_size_repeated_pair_tiles(fg, dev, oracle, monkeypatch, fmt):
    """The CTA-pair tiles at full size, several launches each, every element
    against the oracle: a late reader of the scale-word ring that sees the slot's
    next group shows up as outlier-sized errors in one lane quarter of a few
    tiles, in some launches only."""
    M = 4096
    N = K = 7168
    case = _fp4_case(M, N, K, fmt, 11)
    ref = oracle.gemm_fp4_dequant(*case, fmt)
    for tile in ("2x256", "2x128"):
        monkeypatch.setenv("FGF8_FORCE_TILE", tile)
        for rep in range(3):
            out = _run(fg, dev, case, fmt, M, N)
            gemm_close(out.float().cpu().numpy(), ref, f"fp4 full fmt{fmt} {tile} launch {rep}")


def _row_sf(oracle, sf, row, R, K, fmt):
    """The scale table of one row, cut out of an R-row table."""
    shape, dt = oracle.fp4_sf_shape(1, K, fmt)
    t = np.zeros(shape, dt)
    t[:, 0] = sf[:, row]
    return t


def test_fp4_gemm_deterministic_and_empty(fg, dev):
    case = _fp4_case(256, 256, 512, 1, 3)
    outs = [_run(fg, dev, case, 1, 256, 256) for _ in range(2)]
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    e = torch.empty((0, 256), dtype=torch.uint8, device=dev)         # M = 0, K = 512
    shape, dt = fg.fp4_sf_shape(0, 512, 1)
    d = fg.gemm_fp4_blockscaled(e, torch.empty(shape, dtype=dt, device=dev), to_dev(case[2], dev),
                                to_dev(case[3], dev), 1)
    assert d.shape == (0, 256)
