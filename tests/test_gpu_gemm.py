"""GPU parity: dense GEMMs (16-bit and FP8 block-scaled) vs the fp64 oracle."""
import functools

import numpy as np
import pytest
import torch

from fine_grained_fp8_persistent_gb300 import inputs
from parity import gemm_close, nan_filled, sample_entries, to_dev

pytestmark = pytest.mark.gpu
FMTS = [0, 1]


@pytest.fixture(scope="module")
def fg():
    from fine_grained_fp8_persistent_gb300 import binding
    return binding


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


@functools.lru_cache(maxsize=8)
def _fp8_case(M, N, K, fmt, seed):
    import oracle
    x = inputs.normal_bf16((M, K), seed, outliers=True).float().numpy()
    w = inputs.normal_bf16((N, K), seed + 1, outliers=True).float().numpy()
    aq, sfa = oracle.quantize_1x128(x, fmt)
    bq, sfb = oracle.quantize_128x128(w, fmt)
    return aq, sfa, bq, sfb


def _run_fp8(fg, dev, case, fmt, M, N):
    aq, sfa, bq, sfb = case
    out = nan_filled((M, N), dev)
    fg.gemm_fp8_blockscaled(to_dev(aq, dev), to_dev(sfa, dev), to_dev(bq, dev), to_dev(sfb, dev),
                            fmt, out=out)
    rc, bits = fg.check_status()
    assert rc == 0, (rc, hex(bits), fg.last_error())
    return out


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (200, 264, 384), (1, 32, 128), (129, 96, 128),
                                   (256, 512, 1024), (300, 1024, 640)])
def test_fp8_dense_small(fg, dev, oracle, fmt, M, N, K):
    case = _fp8_case(M, N, K, fmt, 100 + M + N + K)
    out = _run_fp8(fg, dev, case, fmt, M, N)
    ref = oracle.gemm_fp8(*case, fmt)
    gemm_close(out.float().cpu().numpy(), ref, f"fp8 {M}x{N}x{K} fmt{fmt}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M", [64, 4096])
def test_fp8_dense_full_size(fg, dev, oracle, fmt, M):
    """The 7168 x 7168 weight at M = 64 (decode) and 4096 (prefill), in the
    launch configuration the library picks for it: every output element against
    the oracle's dequantize-then-matmul form, plus sampled entries against its
    per-K-block triple loop."""
    N = K = 7168
    case = _fp8_case(M, N, K, fmt, 7)
    out = _run_fp8(fg, dev, case, fmt, M, N)
    got = out.float().cpu().numpy()
    gemm_close(got, oracle.gemm_fp8_dequant(*case, fmt), f"fp8 full M={M} fmt{fmt}")
    r, c = sample_entries(M, N, 300, seed=M)
    gemm_close(got[r, c], oracle.gemm_fp8_entries(*case, fmt, r, c), f"fp8 full M={M} fmt{fmt} (triple loop)")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N", [(130, 264), (64, 200)])
def test_fp8_long_k(fg, dev, oracle, fmt, M, N):
    """K = 32768: 256 K blocks, 64 scale words per row, hundreds of pipeline
    units and scale groups per tile (every ring wraps many times)."""
    K = 32768
    case = _fp8_case(M, N, K, fmt, 900 + M)
    out = _run_fp8(fg, dev, case, fmt, M, N)
    gemm_close(out.float().cpu().numpy(), oracle.gemm_fp8(*case, fmt), f"long K {M}x{N}x{K} fmt{fmt}")


def test_ue8m0_full_size_repeated_pair_tiles(fg, dev, oracle, monkeypatch):
    """UE8M0 scales at 4096 x 7168 x 7168 on the CTA-pair tiles, several launches
    each, every element against the oracle (the scale words pass through the same
    TMA-filled ring as the 4-bit kernels', whose late readers once saw the slot's
    next group)."""
    M = 4096
    N = K = 7168
    case = _fp8_case(M, N, K, 1, 7)
    ref = oracle.gemm_fp8_dequant(*case, 1)
    for tile in ("2x256", "2x224", "2x128"):
        monkeypatch.setenv("FGF8_FORCE_TILE", tile)
        for rep in range(2):
            out = _run_fp8(fg, dev, case, 1, M, N)
            gemm_close(out.float().cpu().numpy(), ref, f"ue8m0 full {tile} launch {rep}")


@pytest.mark.parametrize("fmt", FMTS)
def test_fp8_deterministic(fg, dev, fmt):
    case = _fp8_case(256, 512, 1024, fmt, 5)
    outs = [_run_fp8(fg, dev, case, fmt, 256, 512) for _ in range(3)]
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[0].view(torch.int16), outs[2].view(torch.int16))


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (200, 264, 136), (1, 8, 8), (300, 512, 1024)])
def test_f16_small(fg, dev, oracle, dt, M, N, K):
    a = inputs.uniform_16bit((M, K), M + K, dtype=dt)
    b = inputs.uniform_16bit((N, K), N + K + 1, dtype=dt)
    out = fg.gemm_f16(a.to(dev), b.to(dev))
    rc, _ = fg.check_status()
    assert rc == 0
    assert out.dtype == dt
    ref = oracle.gemm_f16(a.float().numpy(), b.float().numpy())
    gemm_close(out.float().cpu().numpy(), ref, f"f16 {M}x{N}x{K}")


def test_f16_full_size(fg, dev, oracle):
    """16-bit 4096^3: every output element against the oracle."""
    M = N = K = 4096
    a = inputs.uniform_16bit((M, K), 11)
    b = inputs.uniform_16bit((N, K), 12)
    out = fg.gemm_f16(a.to(dev), b.to(dev))
    rc, _ = fg.check_status()
    assert rc == 0
    got = out.float().cpu().numpy()
    gemm_close(got, oracle.gemm_f16_matmul(a.float().numpy(), b.float().numpy()), "f16 4096^3")
    r, c = sample_entries(M, N, 300, seed=3)
    gemm_close(got[r, c], oracle.gemm_f16_entries(a.float().numpy(), b.float().numpy(), r, c), "f16 (loop)")


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_f16_long_k(fg, dev, oracle, dt):
    """K = 16384 + 8: 257 K blocks of 64 elements, the last one 8 wide."""
    M, N, K = 200, 264, 16392
    a = inputs.uniform_16bit((M, K), 31, dtype=dt)
    b = inputs.uniform_16bit((N, K), 32, dtype=dt)
    out = fg.gemm_f16(a.to(dev), b.to(dev))
    rc, _ = fg.check_status()
    assert rc == 0
    gemm_close(out.float().cpu().numpy(), oracle.gemm_f16(a.float().numpy(), b.float().numpy()), "f16 long K")


def test_f16_mixed_output_dtype(fg, dev, oracle):
    a = inputs.uniform_16bit((256, 256), 1)
    b = inputs.uniform_16bit((256, 256), 2)
    out = fg.gemm_f16(a.to(dev), b.to(dev), out_dtype=torch.bfloat16)
    assert out.dtype == torch.bfloat16
    gemm_close(out.float().cpu().numpy(), oracle.gemm_f16(a.float().numpy(), b.float().numpy()))


def test_host_validation_errors(fg, dev):
    a = torch.zeros((16, 100), dtype=torch.uint8, device=dev)
    no_scales = torch.zeros((0,), dtype=torch.float32, device=dev)   # K = 100 has no full 128-block
    with pytest.raises(fg.FGF8Error) as e:                           # the library rejects K % 128
        fg.gemm_fp8_blockscaled(a, no_scales, a, no_scales, 0)
    assert e.value.code == 2


def test_host_memory_is_rejected(fg, dev):
    """The C ABI checks that every tensor pointer is memory of the current device
    before any tensor map is encoded: host memory (pinned or pageable) is refused
    with FGF8_ERR_INVALID_ARG and nothing is launched."""
    import ctypes
    M, N, K = 128, 128, 256
    case = _fp8_case(M, N, K, 1, 9)
    aq, sfa, bq, sfb = (to_dev(x, dev) for x in case)
    out = torch.zeros((M, N), dtype=torch.bfloat16, device=dev)
    host_pinned = torch.zeros_like(aq, device="cpu").pin_memory()
    host_pageable = torch.zeros_like(aq, device="cpu")
    lib = fg.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for host in (host_pinned, host_pageable):
        rc = lib.gemm_fp8_blockscaled(host.data_ptr(), sfa.data_ptr(), bq.data_ptr(), sfb.data_ptr(),
                                      out.data_ptr(), M, N, K, 1, stream)
        assert rc == 1 and "not device memory" in fg.last_error(), (rc, fg.last_error())
    torch.cuda.synchronize()
    assert int(out.view(torch.int16).abs().sum()) == 0      # nothing was written
    rc, _ = fg.check_status()
    assert rc == 0


# Every tile configuration the launchers can pick, forced through FGF8_FORCE_TILE
# as "<CTAs per cluster>x<BN>": one CTA per tile, or a CTA pair (M = 256, B split
# across the pair).
MXF8_TILES = ["2x256", "2x224", "2x128", "1x224", "1x128", "1x64", "1x48", "1x32"]
F8F32_TILES = ["2x128", "1x256", "1x128", "1x64", "1x128ws"]
F16_TILES = ["2x256", "2x224", "1x128"]


@pytest.mark.parametrize("tile", MXF8_TILES)
@pytest.mark.parametrize("M,N,K", [(384, 448, 640), (130, 96, 512), (300, 672, 512)])
def test_fp8_ue8m0_every_tile(fg, dev, oracle, monkeypatch, tile, M, N, K):
    monkeypatch.setenv("FGF8_FORCE_TILE", tile)
    case = _fp8_case(M, N, K, 1, 300 + M)
    out = _run_fp8(fg, dev, case, 1, M, N)
    assert fg.last_tile() == f"mxf8 dense {tile}"
    gemm_close(out.float().cpu().numpy(), oracle.gemm_fp8(*case, 1), f"ue8m0 {tile} {M}x{N}x{K}")


@pytest.mark.parametrize("tile", F8F32_TILES)
@pytest.mark.parametrize("M,N,K", [(384, 512, 640), (130, 96, 512)])
def test_fp8_f32scale_every_tile(fg, dev, oracle, monkeypatch, tile, M, N, K):
    monkeypatch.setenv("FGF8_FORCE_TILE", tile)
    case = _fp8_case(M, N, K, 0, 400 + M)
    out = _run_fp8(fg, dev, case, 0, M, N)
    assert fg.last_tile() == f"f8f32 dense {tile}"
    gemm_close(out.float().cpu().numpy(), oracle.gemm_fp8(*case, 0), f"f32 {tile} {M}x{N}x{K}")


# At most 64 rows the decode tiles stage 64-row A tiles (more stages in flight),
# loaded by boxes of M rounded up to 8 rows: ragged N, K with an odd number of
# 128-blocks, more K blocks than stages, and boxes of 8, 16, 40 and 64 rows.
THIN_TILES = [(1, "1x64"), (1, "1x48"), (1, "1x32"), (0, "1x64")]


@pytest.mark.parametrize("fmt,tile", THIN_TILES)
@pytest.mark.parametrize("M,N,K", [(64, 448, 1920), (37, 200, 2048), (1, 96, 3968), (9, 136, 1024),
                                   (16, 264, 512)])
def test_fp8_thin_a_tiles(fg, dev, oracle, monkeypatch, fmt, tile, M, N, K):
    monkeypatch.setenv("FGF8_FORCE_TILE", tile)
    case = _fp8_case(M, N, K, fmt, 500 + M + K)
    out = _run_fp8(fg, dev, case, fmt, M, N)
    assert fg.last_tile() == f"{'mxf8' if fmt else 'f8f32'} dense {tile}"
    gemm_close(out.float().cpu().numpy(), oracle.gemm_fp8(*case, fmt), f"thin {tile} fmt{fmt} {M}x{N}x{K}")


@pytest.mark.parametrize("tile", F16_TILES)
# K = 136 and 200 leave a short last K block; 136 also gives an odd count of K blocks
@pytest.mark.parametrize("M,N,K", [(384, 512, 640), (130, 96, 200), (520, 768, 256), (200, 256, 136)])
def test_f16_every_tile(fg, dev, oracle, monkeypatch, tile, M, N, K):
    monkeypatch.setenv("FGF8_FORCE_TILE", tile)
    a = inputs.uniform_16bit((M, K), 500 + M, dtype=torch.bfloat16)
    b = inputs.uniform_16bit((N, K), 501 + N, dtype=torch.bfloat16)
    out = fg.gemm_f16(a.to(dev), b.to(dev))
    rc, _ = fg.check_status()
    assert rc == 0
    assert fg.last_tile() == f"f16 dense {tile}"
    gemm_close(out.float().cpu().numpy(), oracle.gemm_f16(a.float().numpy(), b.float().numpy()),
               f"f16 {tile} {M}x{N}x{K}")
