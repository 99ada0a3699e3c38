"""GPU parity: grouped MoE GEMMs (contiguous and masked layouts) vs the oracle."""
import functools

import numpy as np
import pytest
import torch

from fine_grained_fp8_persistent_gb300 import inputs
from parity import gemm_close, nan_filled, to_dev

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


@functools.lru_cache(maxsize=4)
def _contig_case(counts, N, K, fmt, seed):
    import oracle
    m_idx, M = inputs.contiguous_layout(list(counts), 128)
    G = len(counts)
    x = inputs.normal_bf16((M, K), seed, outliers=True).float().numpy()
    w = inputs.normal_bf16((G, N, K), seed + 1, outliers=True).float().numpy()
    aq, sfa = oracle.quantize_1x128(x, fmt)
    bq, sfb = oracle.quantize_128x128(w, fmt)
    return m_idx.numpy(), aq, sfa, bq, sfb


def _run_contig(fg, dev, case, fmt):
    m_idx, aq, sfa, bq, sfb = case
    M, N = aq.shape[0], bq.shape[1]
    out = nan_filled((M, N), dev)
    fg.grouped_fp8_contiguous(to_dev(aq, dev), to_dev(sfa, dev), to_dev(bq, dev), to_dev(sfb, dev),
                              to_dev(m_idx, dev), fmt, out=out)
    return out


@pytest.mark.parametrize("fmt", FMTS)
def test_contiguous_small(fg, dev, oracle, fmt):
    case = _contig_case((70, 0, 130, 128), 256, 384, fmt, 1)
    out = _run_contig(fg, dev, case, fmt)
    rc, bits = fg.check_status()
    assert rc == 0, hex(bits)
    m_idx, aq, sfa, bq, sfb = case
    ref, valid = oracle.grouped_contiguous(aq, sfa, bq, sfb, m_idx, fmt)
    o = out.float().cpu().numpy()
    rows = m_idx >= 0
    gemm_close(o[rows], ref[rows], "contiguous small")
    assert np.isnan(o[~rows]).all(), "padding rows were written"


@pytest.mark.parametrize("fmt", FMTS)
def test_contiguous_full_size(fg, dev, oracle, fmt):
    """8 experts sharing N=4096, K=7168; token counts multinomial(8192, uniform):
    every valid output element against the oracle, padding rows untouched."""
    counts = tuple(inputs.expert_counts(8192, 8, seed=0))
    N, K = 4096, 7168
    case = _contig_case(counts, N, K, fmt, 3)
    out = _run_contig(fg, dev, case, fmt)
    rc, _ = fg.check_status()
    assert rc == 0
    m_idx, aq, sfa, bq, sfb = case
    ref, valid = oracle.grouped_contiguous_dequant(aq, sfa, bq, sfb, m_idx, fmt)
    o = out.float().cpu().numpy()
    rows = m_idx >= 0
    assert np.array_equal(valid.any(axis=1), rows)
    gemm_close(o[rows], ref[rows], "contiguous full")
    assert np.isnan(o[~rows]).all(), "padding rows were written"
    rng = np.random.default_rng(1)
    r = rng.choice(np.flatnonzero(rows), 200)
    c = rng.integers(0, N, 200)
    loop = np.array([oracle.gemm_fp8_entries(aq, sfa, bq[g], sfb[g:g + 1], fmt, [rr], [cc])[0]
                     for rr, cc, g in zip(r, c, m_idx[r])])
    gemm_close(o[r, c], loop, "contiguous full (triple loop)")


# Forced tile configurations of the contiguous layout.  CTA pairs are cut per
# expert segment: segments of 3, 1, 0 and 2 blocks of 128 rows leave half pairs
# whose second CTA stores nothing; N = 456 leaves a ragged last N tile and K = 640
# an odd number of K blocks.
CONTIG_TILES = [(1, "2x224"), (1, "2x128"), (1, "1x224"), (1, "1x128"), (0, "2x128"), (0, "1x256"),
                (0, "1x128")]


@pytest.mark.parametrize("fmt,tile", CONTIG_TILES)
def test_contiguous_every_tile(fg, dev, oracle, monkeypatch, fmt, tile):
    monkeypatch.setenv("FGF8_FORCE_TILE", tile)
    case = _contig_case((300, 70, 0, 200), 456, 640, fmt, 21)
    out = _run_contig(fg, dev, case, fmt)
    rc, bits = fg.check_status()
    assert rc == 0, hex(bits)
    assert fg.last_tile() == f"{'mxf8' if fmt else 'f8f32'} contiguous {tile}"
    m_idx, aq, sfa, bq, sfb = case
    ref, _ = oracle.grouped_contiguous(aq, sfa, bq, sfb, m_idx, fmt)
    o = out.float().cpu().numpy()
    rows = m_idx >= 0
    gemm_close(o[rows], ref[rows], f"contiguous {tile} fmt{fmt}")
    assert np.isnan(o[~rows]).all(), "padding rows were written"


def test_contiguous_bad_row_is_reported(fg, dev):
    case = _contig_case((128, 128), 128, 256, 0, 9)
    m_idx, aq, sfa, bq, sfb = case
    bad = m_idx.copy()
    bad[5] = 1                      # a row of expert 0's block names expert 1
    out = nan_filled((aq.shape[0], 128), dev)
    fg.grouped_fp8_contiguous(to_dev(aq, dev), to_dev(sfa, dev), to_dev(bq, dev), to_dev(sfb, dev),
                              to_dev(bad, dev), 0, out=out)
    rc, bits = fg.check_status()
    assert rc == 6 and bits & 2
    assert bool(torch.isnan(out[5].float()).all())


@functools.lru_cache(maxsize=4)
def _masked_case(G, Mmax, N, K, fmt, seed):
    import oracle
    x = inputs.normal_bf16((G, Mmax, K), seed, outliers=True).float().numpy()
    w = inputs.normal_bf16((G, N, K), seed + 1, outliers=True).float().numpy()
    qs = [oracle.quantize_1x128(x[g], fmt) for g in range(G)]
    aq = np.stack([q[0] for q in qs])
    sfa = np.stack([q[1] for q in qs])
    bq, sfb = oracle.quantize_128x128(w, fmt)
    return aq, sfa, bq, sfb


def _run_masked(fg, dev, case, masked, fmt):
    aq, sfa, bq, sfb = case
    G, Mmax, _ = aq.shape
    N = bq.shape[1]
    out = nan_filled((G, Mmax, N), dev)
    fg.grouped_fp8_masked(to_dev(aq, dev), to_dev(sfa, dev), to_dev(bq, dev), to_dev(sfb, dev),
                          to_dev(np.asarray(masked, np.int32), dev), fmt, out=out)
    return out


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("counts", [(300,), (128,), (1,)])
def test_contiguous_single_expert(fg, dev, oracle, fmt, counts):
    """One expert (G = 1): a single segment, whole, exactly one 128-row block, or
    one row followed by 127 padding rows."""
    case = _contig_case(counts, 264, 640, fmt, 3)
    out = _run_contig(fg, dev, case, fmt)
    rc, bits = fg.check_status()
    assert rc == 0, hex(bits)
    m_idx, aq, sfa, bq, sfb = case
    ref, valid = oracle.grouped_contiguous(aq, sfa, bq, sfb, m_idx, fmt)
    o = out.float().cpu().numpy()
    rows = m_idx >= 0
    gemm_close(o[rows], ref[rows], f"contiguous single expert {counts}")
    assert np.isnan(o[~rows]).all(), "padding rows were written"


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("masked", [(200,), (0,), (1,)])
def test_masked_single_expert(fg, dev, oracle, fmt, masked):
    """One expert (G = 1) with 200, 0 and 1 valid rows of 256."""
    case = _masked_case(1, 256, 264, 640, fmt, 4)
    out = _run_masked(fg, dev, case, masked, fmt)
    rc, bits = fg.check_status()
    assert rc == 0, hex(bits)
    ref, valid = oracle.grouped_masked(*case, np.asarray(masked, np.int32), fmt)
    o = out.float().cpu().numpy()
    v = valid.astype(bool)
    if v.any():
        gemm_close(o[v], ref[v], f"masked single expert {masked}")
    assert np.isnan(o[~v]).all(), "rows beyond masked_m were written"


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("masked", [(0, 256, 17, 1), (128, 129, 255, 0), (0, 0, 0, 0)])
def test_masked_small(fg, dev, oracle, fmt, masked):
    case = _masked_case(4, 256, 256, 384, fmt, 2)
    out = _run_masked(fg, dev, case, masked, fmt)
    rc, bits = fg.check_status()
    assert rc == 0, hex(bits)
    ref, valid = oracle.grouped_masked(*case, np.asarray(masked, np.int32), fmt)
    o = out.float().cpu().numpy()
    v = valid.astype(bool)
    if v.any():
        gemm_close(o[v], ref[v], f"masked {masked}")
    assert np.isnan(o[~v]).all(), "rows beyond masked_m were written"


@pytest.mark.parametrize("fmt", FMTS)
def test_masked_full_size(fg, dev, oracle, fmt):
    """32 experts, Mmax=256, N=7168, K=2048, valid rows uniform in [0, 256]:
    every valid output element against the oracle, the other rows untouched."""
    G, Mmax, N, K = 32, 256, 7168, 2048
    masked = inputs.masked_rows(G, Mmax, seed=0).numpy()
    case = _masked_case(G, Mmax, N, K, fmt, 4)
    out = _run_masked(fg, dev, case, masked, fmt)
    rc, _ = fg.check_status()
    assert rc == 0
    aq, sfa, bq, sfb = case
    ref, valid = oracle.grouped_masked_dequant(aq, sfa, bq, sfb, masked, fmt)
    o = out.float().cpu().numpy()
    v = valid.astype(bool)
    gemm_close(o[v], ref[v], "masked full")
    assert np.isnan(o[~v]).all(), "rows beyond masked_m were written"
    rng = np.random.default_rng(2)
    gs = [g for g in range(G) if masked[g] > 0]
    g = rng.choice(gs, 200)
    m = np.array([rng.integers(0, masked[x]) for x in g])
    n = rng.integers(0, N, 200)
    loop = np.array([oracle.gemm_fp8_entries(aq[gg], sfa[gg], bq[gg], sfb[gg:gg + 1], fmt, [mm], [nn])[0]
                     for gg, mm, nn in zip(g, m, n)])
    gemm_close(o[g, m, n], loop, "masked full (triple loop)")


def test_masked_bad_count_is_reported(fg, dev):
    case = _masked_case(2, 128, 128, 256, 0, 5)
    out = _run_masked(fg, dev, case, (5, 1000), 0)
    rc, bits = fg.check_status()
    assert rc == 6 and bits & 2


@pytest.mark.parametrize("tile", ["2x224", "2x128", "1x224", "1x64", "1x48"])
def test_masked_ue8m0_every_tile(fg, dev, oracle, monkeypatch, tile):
    monkeypatch.setenv("FGF8_FORCE_TILE", tile)
    masked = (0, 256, 17, 200)
    case = _masked_case(4, 256, 448, 384, 1, 6)
    out = _run_masked(fg, dev, case, masked, 1)
    rc, bits = fg.check_status()
    assert rc == 0, hex(bits)
    ref, valid = oracle.grouped_masked(*case, np.asarray(masked, np.int32), 1)
    o = out.float().cpu().numpy()
    v = valid.astype(bool)
    gemm_close(o[v], ref[v], f"masked {tile}")
    assert np.isnan(o[~v]).all()


@pytest.mark.parametrize("tile", ["2x128", "1x256", "1x128", "1x128ws"])
def test_masked_f32scale_every_tile(fg, dev, oracle, monkeypatch, tile):
    monkeypatch.setenv("FGF8_FORCE_TILE", tile)
    masked = (0, 256, 17, 200)
    case = _masked_case(4, 256, 512, 384, 0, 7)
    out = _run_masked(fg, dev, case, masked, 0)
    rc, bits = fg.check_status()
    assert rc == 0, hex(bits)
    ref, valid = oracle.grouped_masked(*case, np.asarray(masked, np.int32), 0)
    o = out.float().cpu().numpy()
    v = valid.astype(bool)
    gemm_close(o[v], ref[v], f"masked f32 {tile}")
    assert np.isnan(o[~v]).all()


@pytest.mark.parametrize("fmt", FMTS)
def test_masked_maximum_expert_count(fg, dev, oracle, fmt):
    """G = 1024 experts, the largest the masked scheduler's per-expert table holds."""
    G, Mmax, N, K = 1024, 32, 128, 128
    masked = inputs.masked_rows(G, Mmax, seed=11).numpy()
    case = _masked_case(G, Mmax, N, K, fmt, 12)
    out = _run_masked(fg, dev, case, masked, fmt)
    rc, bits = fg.check_status()
    assert rc == 0, hex(bits)
    ref, valid = oracle.grouped_masked(*case, masked, fmt)
    o = out.float().cpu().numpy()
    v = valid.astype(bool)
    gemm_close(o[v], ref[v], "masked G=1024")
    assert np.isnan(o[~v]).all()


@pytest.mark.parametrize("counts,pairs", [((20000, 16000, 30000, 510), False),   # 521 blocks of 128 rows
                                          ((16384, 16384, 16384, 16384), True)])  # exactly 512
def test_contiguous_pair_table_limit(fg, dev, oracle, monkeypatch, counts, pairs):
    """A CTA-pair tile is asked for.  Beyond the pair scheduler's segment table
    (512 blocks of 128 rows) the launcher does not offer pairs and falls back to
    one-CTA tiles; at the limit it still runs the pair."""
    monkeypatch.setenv("FGF8_FORCE_TILE", "2x128")
    fmt = 1
    case = _contig_case(counts, 64, 128, fmt, 13)
    out = _run_contig(fg, dev, case, fmt)
    rc, bits = fg.check_status()
    assert rc == 0, hex(bits)
    ctas = int(fg.last_tile().split()[-1].split("x")[0])
    assert (ctas == 2) == pairs, fg.last_tile()
    m_idx, aq, sfa, bq, sfb = case
    ref, _ = oracle.grouped_contiguous(aq, sfa, bq, sfb, m_idx, fmt)
    o = out.float().cpu().numpy()
    rows = m_idx >= 0
    gemm_close(o[rows], ref[rows], f"contiguous {sum(counts)} rows")
    assert np.isnan(o[~rows]).all()


def test_masked_in_a_cuda_graph(fg, dev, oracle):
    """The masked layout reads its row counts on the device, so one captured call
    serves any counts: capture once, change masked_m in place, replay."""
    G, Mmax, N, K, fmt = 4, 256, 256, 384, 1
    case = _masked_case(G, Mmax, N, K, fmt, 14)
    aq, sfa, bq, sfb = (to_dev(a, dev) for a in case)
    counts = torch.zeros(G, dtype=torch.int32, device=dev)
    out = torch.empty((G, Mmax, N), dtype=torch.bfloat16, device=dev)
    fg.grouped_fp8_masked(aq, sfa, bq, sfb, counts, fmt, out=out)      # warm-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fg.grouped_fp8_masked(aq, sfa, bq, sfb, counts, fmt, out=out)
    for masked in [(0, 256, 17, 1), (128, 0, 255, 64)]:
        out.fill_(float("nan"))
        counts.copy_(torch.tensor(masked, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        rc, bits = fg.check_status()
        assert rc == 0, hex(bits)
        ref, valid = oracle.grouped_masked(*case, np.asarray(masked, np.int32), fmt)
        o = out.float().cpu().numpy()
        v = valid.astype(bool)
        gemm_close(o[v], ref[v], f"graph replay {masked}")
        assert np.isnan(o[~v]).all()


def test_masked_weight_stationary_full_size(fg, dev, oracle, monkeypatch):
    """The masked decode configuration (32 experts, Mmax = 256, N = 7168, K = 2048,
    FP32 scales) on the weight-stationary tile: every valid element against the
    oracle's dequantize-then-matmul form; rows past masked_m stay unwritten."""
    monkeypatch.setenv("FGF8_FORCE_TILE", "1x128ws")
    G, Mmax, N, K = 32, 256, 7168, 2048
    masked = inputs.masked_rows(G, Mmax, 10).numpy()
    case = _masked_case(G, Mmax, N, K, 0, 11)
    out = _run_masked(fg, dev, case, tuple(int(m) for m in masked), 0)
    assert fg.last_tile() == "f8f32 masked 1x128ws"
    ref, valid = oracle.grouped_masked_dequant(*case, masked.astype(np.int32), 0)
    o = out.float().cpu().numpy()
    v = valid.astype(bool)
    gemm_close(o[v], ref[v], "masked ws full size")
    assert np.isnan(o[~v]).all()
