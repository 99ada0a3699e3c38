"""GPU parity: quantize kernels vs the oracle, bit-exact (codes and scale words)."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_persistent_gb300 import inputs

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


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,K", [(1, 128), (37, 640), (128, 256), (130, 1536), (4096, 7168)])
def test_quantize_1x128_bit_exact(fg, dev, oracle, fmt, M, K):
    x = inputs.normal_bf16((M, K), seed=M * 7 + K, outliers=True)
    xq, sfa = fg.quantize_1x128(x.to(dev), fmt)
    oq, osf = oracle.quantize_1x128(x.float().numpy(), fmt)
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), oq)
    assert sfa.dtype == (torch.float32 if fmt == 0 else torch.int32)
    assert np.array_equal(sfa.cpu().numpy().view(np.uint8), osf.view(np.uint8))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("G,N,K", [(1, 128, 256), (1, 300, 512), (3, 128, 640), (1, 7168, 7168)])
def test_quantize_128x128_bit_exact(fg, dev, oracle, fmt, G, N, K):
    w = inputs.normal_bf16((G, N, K), seed=G + N + K, outliers=True)
    wq, sfb = fg.quantize_128x128(w.to(dev), fmt)
    oq, osf = oracle.quantize_128x128(w.float().numpy(), fmt)
    torch.cuda.synchronize()
    assert np.array_equal(wq.cpu().numpy(), oq)
    assert np.array_equal(sfb.cpu().numpy().view(np.uint8), osf.view(np.uint8))


def test_quantize_special_values(fg, dev, oracle):
    """Zero groups, signed zeros, tiny values and exact midpoints."""
    x = torch.zeros((4, 256), dtype=torch.float32)
    x[1, 5] = -0.0
    x[2, :128] = torch.linspace(-1e-30, 1e-30, 128)
    x[3, :128] = 448.0
    x[3, 128:] = torch.tensor([1.0625, -1.1875, 3.0, 2.0 ** -9] * 32)
    x = x.to(torch.bfloat16)
    for fmt in FMTS:
        xq, sfa = fg.quantize_1x128(x.to(dev), fmt)
        oq, osf = oracle.quantize_1x128(x.float().numpy(), fmt)
        torch.cuda.synchronize()
        assert np.array_equal(xq.cpu().numpy(), oq)
        assert np.array_equal(sfa.cpu().numpy().view(np.uint8), osf.view(np.uint8))


def test_quantize_empty_is_noop(fg, dev):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=dev)
    xq, sfa = fg.quantize_1x128(x, 0)
    assert xq.shape == (0, 256)


def _every_value_under_many_scales():
    """1x128 groups led by amax, then every bf16 value of magnitude <= amax (both
    signs), for amax = every bf16 significand at exponents from 2^-100 to 2^100.
    The FP32 scales amax / 448 then run through all significand patterns of the
    scale's top bits, and the codes cover every E4M3 rounding decision each scale
    can see, ties included; 2^-100 and 2^-60 groups sit on either side of the
    scale below which the kernels divide with the IEEE routine."""
    bits = np.arange(0x8000, dtype=np.uint32)
    pos = (bits << 16).view(np.float32)
    pos = pos[np.isfinite(pos)]
    groups = []
    for e in (-100, -60, -20, -8, -1, 0, 1, 3, 7, 15, 40, 100):
        for m in range(128):
            amax = np.float32(np.ldexp(1.0 + m / 128.0, e))
            vals = pos[pos <= amax]
            vals = np.concatenate([vals, -vals])
            vals = np.concatenate([vals, np.zeros((-len(vals)) % 127, np.float32)])
            body = vals.reshape(-1, 127)
            groups.append(np.concatenate([np.full((len(body), 1), amax, np.float32), body], axis=1))
    g = np.concatenate(groups).reshape(-1)
    g = np.concatenate([g, np.zeros((-len(g)) % 4096, np.float32)])
    return torch.from_numpy(g.reshape(-1, 4096)).to(torch.bfloat16)


def test_quantize_1x128_f32_scales_every_value(fg, dev, oracle):
    """FP32 scales: the kernels divide by the scale without the IEEE division
    routine (Markstein's FMA division); every code must still equal the oracle's,
    which divides in IEEE arithmetic.  About 60 M values under 1536 scales."""
    x = _every_value_under_many_scales()
    xq, sfa = fg.quantize_1x128(x.to(dev), 0)
    oq, osf = oracle.quantize_1x128(x.float().numpy(), 0)
    torch.cuda.synchronize()
    assert np.array_equal(sfa.cpu().numpy().view(np.uint8), osf.view(np.uint8)), "scales differ"
    got = xq.cpu().numpy()
    bad = np.nonzero(got != oq)
    assert bad[0].size == 0, f"{bad[0].size} codes differ, first at {bad[0][0]}, {bad[1][0]}"
