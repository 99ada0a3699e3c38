"""Device-side failure detection without a GPU fault.

A kernel wait that nothing will ever satisfy must give up after the configured
limit, report FGF8_ERR_DEVICE_TIMEOUT through the status word (with the role
that gave up) and return, leaving the CUDA context usable: the next GEMM on the
same device runs and matches the oracle.  Host-side validation errors are
covered by test_abi.py and the device-input checks by test_gpu_grouped.py.
"""
import time

import pytest
import torch

from fine_grained_fp8_persistent_gb300 import inputs
from parity import gemm_close, to_dev

pytestmark = pytest.mark.gpu

TIMEOUT = 0x1
ROLE_SELFTEST = 0x800


@pytest.fixture(scope="module")
def fg():
    from fine_grained_fp8_persistent_gb300 import binding
    return binding


def test_wait_gives_up_reports_and_leaves_the_context_usable(fg, oracle):
    dev = torch.device("cuda:0")
    assert fg.check_status()[0] == 0                  # clean start
    prev = fg.set_wait_timeout_ms(20)
    try:
        t0 = time.perf_counter()
        fg.selftest_wait_timeout()
        rc, bits = fg.check_status()                  # synchronises the stream
        elapsed = time.perf_counter() - t0
    finally:
        fg.set_wait_timeout_ms(prev)
    assert rc == 5, (rc, hex(bits))                   # FGF8_ERR_DEVICE_TIMEOUT
    assert bits == TIMEOUT | ROLE_SELFTEST, hex(bits)
    assert 0.015 <= elapsed < 10.0                    # it waited its limit, then returned
    assert fg.check_status() == (0, 0)                # reading cleared the word

    # the context is still usable: a GEMM right after matches the oracle
    ue = fg.SCALE_UE8M0
    x = inputs.normal_bf16((128, 256), 31, outliers=True).float().numpy()
    w = inputs.normal_bf16((128, 256), 32, outliers=True).float().numpy()
    aq, sfa = oracle.quantize_1x128(x, ue)
    bq, sfb = oracle.quantize_128x128(w, ue)
    d = fg.gemm_fp8_blockscaled(to_dev(aq, dev), to_dev(sfa, dev), to_dev(bq, dev), to_dev(sfb, dev), ue)
    assert fg.check_status()[0] == 0
    gemm_close(d.float().cpu().numpy(), oracle.gemm_fp8(aq, sfa, bq, sfb, ue), "gemm after a timed-out wait")
