"""Programmatic dependent launch keeps every data dependency.

With PDL each kernel starts its set-up while the previous kernel on the stream
is still running, so a read of a predecessor's output placed before the grid
dependency wait would see stale data.  These chains feed every GEMM the output of
the quantizer launched just before it, with inputs that change every iteration,
and compare against the oracle and against the same chain with PDL off.
"""
import pytest
import torch

from fine_grained_fp8_persistent_gb300 import inputs
from parity import gemm_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fg():
    from fine_grained_fp8_persistent_gb300 import binding
    return binding


def _chain(fg, xs, w, fmt):
    """quantize_128x128(w); then per x: quantize_1x128(x) -> GEMM, all back to back
    on one stream, reusing the same quantized buffers."""
    dev = xs[0].device
    M, K = xs[0].shape
    N = w.shape[0]
    xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sh, dt = fg.sfa_shape(M, K, fmt)
    sfa = torch.empty(sh, dtype=dt, device=dev)
    wq, sfb = fg.quantize_128x128(w, fmt)
    outs = []
    for x in xs:
        fg.quantize_1x128(x, fmt, xq, sfa)
        outs.append(fg.gemm_fp8_blockscaled(xq, sfa, wq, sfb, fmt))
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("fmt", [0, 1])
def test_dependent_chain_matches_oracle_and_pdl_off(fg, oracle, fmt):
    dev = torch.device("cuda:0")
    M, N, K = 256, 384, 2048
    xs_cpu = [inputs.normal_bf16((M, K), 700 + i, outliers=True) for i in range(6)]
    w_cpu = inputs.normal_bf16((N, K), 799, outliers=True)
    xs = [x.to(dev) for x in xs_cpu]
    w = w_cpu.to(dev)
    prev = fg.set_pdl(True)
    try:
        on = _chain(fg, xs, w, fmt)
        fg.set_pdl(False)
        off = _chain(fg, xs, w, fmt)
    finally:
        fg.set_pdl(prev)
    assert fg.check_status()[0] == 0
    for a, b in zip(on, off):
        assert torch.equal(a, b), "PDL changed a result"
    bq, sfb = oracle.quantize_128x128(w_cpu.float().numpy(), fmt)
    for i in (0, 3, 5):
        aq, sfa = oracle.quantize_1x128(xs_cpu[i].float().numpy(), fmt)
        gemm_close(on[i].float().cpu().numpy(), oracle.gemm_fp8(aq, sfa, bq, sfb, fmt), f"chain step {i}")
