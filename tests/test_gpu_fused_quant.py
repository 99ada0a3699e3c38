"""GPU parity: the FP8 GEMM (UE8M0 or FP32 input scales) with 1x128 output
quantization fused into its epilogue.  Against the oracle's own chain (fp64 GEMM,
rounded to bf16, quantized 1x128), within the quantization and GEMM error bounds;
and bit for bit against the same library's unfused chain (gemm_fp8_blockscaled,
then quantize_1x128)."""
import functools

import numpy as np
import pytest
import torch

from fine_grained_fp8_persistent_gb300 import inputs
from parity import to_dev

pytestmark = pytest.mark.gpu
UE8M0 = 1


@pytest.fixture(scope="module")
def fg():
    from fine_grained_fp8_persistent_gb300 import binding
    return binding


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


@functools.lru_cache(maxsize=16)
def _case(M, N, K, seed, in_fmt=UE8M0):
    import oracle
    x = inputs.normal_bf16((M, K), seed, outliers=True).float().numpy()
    w = inputs.normal_bf16((N, K), seed + 1, outliers=True).float().numpy()
    aq, sfa = oracle.quantize_1x128(x, in_fmt)
    bq, sfb = oracle.quantize_128x128(w, in_fmt)
    return aq, sfa, bq, sfb


GUARD = 4096   # bytes after each output that must stay untouched


def _fused(fg, dev, case, M, N, out_fmt, in_fmt=UE8M0):
    aq, sfa, bq, sfb = case
    # outputs pre-filled (0x7F is an E4M3 NaN, so an unwritten code shows) and
    # followed by guard regions that no write may reach
    dq_buf = torch.full((M * N + GUARD,), 0x7F, dtype=torch.uint8, device=dev)
    dq = dq_buf[:M * N].view(M, N)
    shape, dt = fg.sfa_shape(M, N, out_fmt)
    count = shape[0] * shape[1]
    sf_buf = torch.full((count + GUARD // 4,), -1, dtype=torch.int32, device=dev)   # all-ones words
    sfd = sf_buf[:count].view(dt).view(shape)
    fg.gemm_fp8_blockscaled_quant(to_dev(aq, dev), to_dev(sfa, dev), to_dev(bq, dev), to_dev(sfb, dev),
                                  in_fmt, out_fmt, dq=dq, sfd=sfd)
    rc, bits = fg.check_status()
    assert rc == 0, (rc, hex(bits), fg.last_error())
    assert bool((dq_buf[M * N:] == 0x7F).all()), "write past the end of Dq"
    assert bool((sf_buf[count:] == -1).all()), "write past the end of the scale table"
    return dq, sfd


def _unfused(fg, dev, case, M, N, out_fmt, in_fmt=UE8M0):
    aq, sfa, bq, sfb = case
    d = fg.gemm_fp8_blockscaled(to_dev(aq, dev), to_dev(sfa, dev), to_dev(bq, dev), to_dev(sfb, dev), in_fmt)
    return fg.quantize_1x128(d, out_fmt)


def _dequant(oracle, q, sf, out_fmt, M, N):
    """Codes and a scale table in the quantize_1x128 layout -> values (M, N)."""
    vals = oracle.e4m3_decode(q).astype(np.float64)
    g = np.arange(N) // 128
    if out_fmt == UE8M0:
        words = sf.view(np.uint32)
        e = ((words[g // 4, :M].T >> (8 * (g % 4))) & 0xFF).astype(np.int64) - 127
        s = np.ldexp(1.0, e)
    else:
        s = sf[g, :M].T.astype(np.float64)
    return vals * s, s


SHAPES = [(200, 384, 512), (64, 512, 256), (1, 128, 128), (300, 1024, 640), (129, 640, 384)]


# (input scale format, tile): block-scaled tiles 256 or 128 wide; the FP32-scale
# path quantizes on its 256-wide tile
TILES = [(UE8M0, "2x256"), (UE8M0, "2x128"), (UE8M0, "1x128"), (0, "1x256")]


@pytest.mark.parametrize("in_fmt,tile", TILES)
@pytest.mark.parametrize("out_fmt", [0, 1])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_fused_equals_unfused_chain(fg, dev, monkeypatch, in_fmt, tile, out_fmt, M, N, K):
    monkeypatch.setenv("FGF8_FORCE_TILE", tile)
    case = _case(M, N, K, 600 + M + N, in_fmt)
    dq, sfd = _fused(fg, dev, case, M, N, out_fmt, in_fmt)
    assert fg.last_tile() == f"{'mxf8' if in_fmt else 'f8f32'} dense {tile}"
    xq, sf = _unfused(fg, dev, case, M, N, out_fmt, in_fmt)
    assert torch.equal(dq, xq), "codes differ from quantize_1x128 of the GEMM output"
    assert torch.equal(sfd.view(torch.int32), sf.view(torch.int32)), "scale tables differ"


@pytest.mark.parametrize("in_fmt", [0, 1])
@pytest.mark.parametrize("out_fmt", [0, 1])
@pytest.mark.parametrize("M,N,K", SHAPES[:4])
def test_fused_vs_oracle_chain(fg, dev, oracle, in_fmt, out_fmt, M, N, K):
    case = _case(M, N, K, 600 + M + N, in_fmt)
    dq, sfd = _fused(fg, dev, case, M, N, out_fmt, in_fmt)
    d_ref = oracle.gemm_fp8(*case, in_fmt)                                  # fp64
    d_bf16 = torch.from_numpy(d_ref).to(torch.bfloat16).float().numpy()
    q_o, sf_o = oracle.quantize_1x128(d_bf16, out_fmt)
    got, s_got = _dequant(oracle, dq.cpu().numpy(), sfd.cpu().numpy(), out_fmt, M, N)
    ref, s_ref = _dequant(oracle, q_o, sf_o, out_fmt, M, N)
    # each side is within half an E4M3 step of its own bf16 D (2^-4 relative, or
    # 2^-10 of the scale below the normal range); the two D differ by the GEMM's
    # own rounding, well inside 1e-2 of max |D|
    bound = 2.0 ** -3 * np.abs(ref) + 2.0 ** -9 * np.maximum(s_got, s_ref) + 1e-2 * np.abs(d_ref).max()
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) - bound))
    if out_fmt == UE8M0:
        assert np.all(np.abs(np.log2(s_got) - np.log2(s_ref)) <= 1)
    else:
        assert np.allclose(s_got, s_ref, rtol=1e-2, atol=0)


def test_fused_full_size_matches_unfused(fg, dev):
    """The bench's M=4096, N=K=7168 shape: fused against unfused, every byte."""
    M = 4096
    N = K = 7168
    torch.manual_seed(0)
    x = inputs.normal_bf16((M, K), 11, outliers=True).to(dev)
    w = inputs.normal_bf16((N, K), 12, outliers=True).to(dev)
    for in_fmt in (UE8M0, 0):
        aq, sfa = fg.quantize_1x128(x, in_fmt)
        bq, sfb = fg.quantize_128x128(w, in_fmt)
        for out_fmt in (0, 1):
            dq, sfd = fg.gemm_fp8_blockscaled_quant(aq, sfa, bq, sfb, in_fmt, out_fmt)
            d = fg.gemm_fp8_blockscaled(aq, sfa, bq, sfb, in_fmt)
            xq, sf = fg.quantize_1x128(d, out_fmt)
            assert torch.equal(dq, xq)
            assert torch.equal(sfd.view(torch.int32), sf.view(torch.int32))


def test_fused_rejects_unsupported(fg, dev):
    case = _case(64, 512, 256, 7)
    aq, sfa, bq, sfb = (to_dev(a, dev) for a in case)
    shape, dt = fg.sfb_shape(1, 200, 256, UE8M0)
    sfb200 = torch.zeros(shape, dtype=dt, device=dev)
    with pytest.raises(fg.FGF8Error) as e:                                 # N not a multiple of 128
        fg.gemm_fp8_blockscaled_quant(aq, sfa, bq.reshape(-1, 256)[:200], sfb200, UE8M0, 0)
    assert e.value.code == 2
