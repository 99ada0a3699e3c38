"""GPU tests of the tile schedulers: cluster launch control (one cluster per tile;
running clusters cancel clusters not yet launched and take their tiles) and the
wave-preserving SM cap of the static persistent grid.

Scheduling changes only which CTA computes a tile, never how: every output must be
bit-identical to the static schedule's.  The problems are sized so that there are
more cluster tiles than clusters fit on the GPU, so cancellation really happens;
one case is also compared with the oracle."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_persistent_gb300 import inputs
from parity import gemm_close, nan_filled, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fg():
    from fine_grained_fp8_persistent_gb300 import binding
    return binding


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


@pytest.fixture
def restore(fg):
    prev_s = fg.set_scheduler(fg.SCHED_STATIC)
    prev_c = fg.set_sm_cap(False)
    yield
    fg.set_scheduler(prev_s)
    fg.set_sm_cap(prev_c)


def _under(fg, mode, cap, fn):
    fg.set_scheduler(mode)
    fg.set_sm_cap(cap)
    out = fn()
    rc, bits = fg.check_status()
    assert rc == 0, (rc, hex(bits), fg.last_error())
    torch.cuda.synchronize()
    return out, fg.last_tile()


def _same_bits(a, b, what):
    for x, y in zip(a if isinstance(a, tuple) else (a,), b if isinstance(b, tuple) else (b,)):
        xb = x.contiguous().view(torch.uint8)
        yb = y.contiguous().view(torch.uint8)
        assert torch.equal(xb, yb), f"{what}: outputs differ between schedules"


def _all_schedules(fg, fn, what):
    ref, tile = _under(fg, fg.SCHED_STATIC, False, fn)
    for mode, cap in ((fg.SCHED_CLC, False), (fg.SCHED_STATIC, True)):
        got, t2 = _under(fg, mode, cap, fn)
        assert t2 == tile
        _same_bits(ref, got, f"{what} ({tile}, scheduler {mode}, cap {cap})")
    return ref


def _fp8_operands(fg, dev, M, N, K, fmt, seed):
    x = inputs.normal_bf16((M, K), seed, outliers=True).to(dev)
    w = inputs.normal_bf16((N, K), seed + 1, outliers=True).to(dev)
    xq, sfa = fg.quantize_1x128(x, fmt)
    wq, sfb = fg.quantize_128x128(w, fmt)
    return xq, sfa, wq.reshape(N, K), sfb


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("tile", [None, "1x128", "2x128", "1x128ws"])
def test_dense_fp8_same_bits(fg, dev, restore, monkeypatch, fmt, tile):
    if tile:
        monkeypatch.setenv("FGF8_FORCE_TILE", tile)
    M, N, K = 4096, 7168, 512
    xq, sfa, wq, sfb = _fp8_operands(fg, dev, M, N, K, fmt, 40)

    def run():
        out = nan_filled((M, N), dev)
        fg.gemm_fp8_blockscaled(xq, sfa, wq, sfb, fmt, out=out)
        return out
    _all_schedules(fg, run, f"dense fp8 fmt{fmt}")


def test_decode_thin_tile_same_bits(fg, dev, restore):
    M, N, K = 64, 7168, 1024
    xq, sfa, wq, sfb = _fp8_operands(fg, dev, M, N, K, 1, 41)

    def run():
        out = nan_filled((M, N), dev)
        fg.gemm_fp8_blockscaled(xq, sfa, wq, sfb, 1, out=out)
        return out
    _all_schedules(fg, run, "decode")


def test_f16_same_bits(fg, dev, restore):
    M, N, K = 4096, 4096, 512
    a = inputs.uniform_16bit((M, K), 42).to(dev)
    b = inputs.uniform_16bit((N, K), 43).to(dev)
    _all_schedules(fg, lambda: fg.gemm_f16(a, b), "f16")


@pytest.mark.parametrize("fmt", [0, 1])
def test_contiguous_same_bits(fg, dev, restore, fmt):
    G, N, K = 8, 4096, 512
    counts = inputs.expert_counts(8192, G, 44)
    m_idx, total = inputs.contiguous_layout(counts, fg.mk_alignment_for_contiguous())
    a = inputs.normal_bf16((total, K), 45, outliers=True).to(dev)
    b = inputs.normal_bf16((G, N, K), 46, outliers=True).to(dev)
    aq, sfa = fg.quantize_1x128(a, fmt)
    bq, sfb = fg.quantize_128x128(b, fmt)
    mi = m_idx.to(dev)

    def run():
        out = nan_filled((total, N), dev)
        fg.grouped_fp8_contiguous(aq, sfa, bq, sfb, mi, fmt, out=out)
        return out
    out = _all_schedules(fg, run, f"contiguous fmt{fmt}")
    pad = (m_idx < 0).nonzero().flatten()
    if pad.numel():
        assert torch.isnan(out[pad.to(dev)].float()).all(), "padding rows were written"


@pytest.mark.parametrize("fmt", [0, 1])
def test_masked_same_bits(fg, dev, restore, fmt):
    G, MM, N, K = 32, 256, 7168, 512
    mm = inputs.masked_rows(G, MM, 47)
    mm[3] = 0                                   # an empty expert
    mm[5] = MM                                  # a full one
    am = inputs.normal_bf16((G, MM, K), 48, outliers=True).to(dev)
    bm = inputs.normal_bf16((G, N, K), 49, outliers=True).to(dev)
    sh, dt = fg.sfa_shape(MM, K, fmt)
    aq = torch.empty((G, MM, K), dtype=torch.uint8, device=dev)
    sfa = torch.empty((G, *sh), dtype=dt, device=dev)
    for g in range(G):
        fg.quantize_1x128(am[g], fmt, aq[g], sfa[g])
    bq, sfb = fg.quantize_128x128(bm, fmt)
    mmd = mm.to(dev)

    def run():
        out = nan_filled((G, MM, N), dev)
        fg.grouped_fp8_masked(aq, sfa, bq, sfb, mmd, fmt, out=out)
        return out
    out = _all_schedules(fg, run, f"masked fmt{fmt}")
    for g in range(G):
        assert torch.isnan(out[g, int(mm[g]):].float()).all(), f"expert {g}: rows past masked_m written"


@pytest.mark.parametrize("fmt", [0, 1])
def test_fp4_same_bits(fg, dev, restore, fmt):
    M, N, K = 4096, 7168, 512
    x = inputs.normal_bf16((M, K), 50, outliers=True).to(dev)
    w = inputs.normal_bf16((N, K), 51, outliers=True).to(dev)
    xq, sfa = fg.quantize_fp4(x, fmt)
    wq, sfb = fg.quantize_fp4(w, fmt)

    def run():
        out = nan_filled((M, N), dev)
        fg.gemm_fp4_blockscaled(xq, sfa, wq, sfb, fmt, out=out)
        return out
    _all_schedules(fg, run, f"fp4 fmt{fmt}")


@pytest.mark.parametrize("fmt", [0, 1])
def test_fused_quant_same_bits(fg, dev, restore, fmt):
    M, N, K = 4096, 7168, 512
    xq, sfa, wq, sfb = _fp8_operands(fg, dev, M, N, K, fmt, 52)
    _all_schedules(fg, lambda: fg.gemm_fp8_blockscaled_quant(xq, sfa, wq, sfb, fmt, 1), f"fused fmt{fmt}")


def test_clc_matches_the_oracle(fg, dev, restore, oracle, monkeypatch):
    """256 single-CTA tiles (more than the SMs): under cluster launch control,
    against the oracle's per-K-block triple loop."""
    monkeypatch.setenv("FGF8_FORCE_TILE", "1x128")
    M, N, K = 2048, 2048, 256
    x = inputs.normal_bf16((M, K), 53, outliers=True).float().numpy()
    w = inputs.normal_bf16((N, K), 54, outliers=True).float().numpy()
    aq, sfa = oracle.quantize_1x128(x, 1)
    bq, sfb = oracle.quantize_128x128(w, 1)
    bq = bq.reshape(N, K)
    fg.set_scheduler(fg.SCHED_CLC)
    out = nan_filled((M, N), dev)
    fg.gemm_fp8_blockscaled(to_dev(aq, dev), to_dev(sfa, dev), to_dev(bq, dev), to_dev(sfb, dev), 1, out=out)
    rc, bits = fg.check_status()
    assert rc == 0, (rc, hex(bits))
    assert fg.last_tile() == "mxf8 dense 1x128"
    gemm_close(out.float().cpu().numpy(), oracle.gemm_fp8(aq, sfa, bq, sfb, 1), "clc 2048^2 x 256")


def test_clc_repeated_launches_and_graph(fg, dev, restore):
    """Back-to-back launches and a CUDA graph replay under cluster launch control
    give the same bits as the static schedule."""
    M, N, K = 4096, 7168, 256
    xq, sfa, wq, sfb = _fp8_operands(fg, dev, M, N, K, 1, 55)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    fg.set_scheduler(fg.SCHED_STATIC)
    fg.gemm_fp8_blockscaled(xq, sfa, wq, sfb, 1, out=ref)
    fg.set_scheduler(fg.SCHED_CLC)
    outs = [torch.empty_like(ref) for _ in range(4)]
    for o in outs:
        fg.gemm_fp8_blockscaled(xq, sfa, wq, sfb, 1, out=o)
    rc, _ = fg.check_status()
    assert rc == 0
    for o in outs:
        _same_bits(ref, o, "repeated clc launch")
    g_out = torch.empty_like(ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fg.gemm_fp8_blockscaled(xq, sfa, wq, sfb, 1, out=g_out)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fg.gemm_fp8_blockscaled(xq, sfa, wq, sfb, 1, out=g_out)
    g_out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    rc, _ = fg.check_status()
    assert rc == 0
    _same_bits(ref, g_out, "clc in a CUDA graph")
