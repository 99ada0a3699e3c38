"""CPU checks of the Python binding's argument checks: every tensor handed to the
C ABI as a raw pointer must have the size the call will touch, and live on the
launch stream's device.  The library is replaced by a recorder, so nothing
reaches a GPU."""
from types import SimpleNamespace

import pytest
import torch


class _Recorder:
    """Stands in for the loaded library: records calls, returns success."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def f(*args):
            self.calls.append(name)
            return 0
        return f


@pytest.fixture()
def fg(monkeypatch):
    from fine_grained_fp8_persistent_gb300 import binding
    rec = _Recorder()
    monkeypatch.setattr(binding, "_lib", rec)
    monkeypatch.setattr(binding, "_ptr", lambda t: None if t is None else t.data_ptr())
    monkeypatch.setattr(binding, "_stream", lambda stream=None, **t: binding._Stream(0, None))
    monkeypatch.setattr(binding, "_call", lambda name, st, *args: rec.calls.append(name))
    binding.recorder = rec
    return binding


def _fp8(fg, M, N, K, fmt, G=1):
    aq = torch.zeros((M, K), dtype=torch.uint8)
    bq = torch.zeros((G, N, K), dtype=torch.uint8) if G > 1 else torch.zeros((N, K), dtype=torch.uint8)
    sa, da = fg.sfa_shape(M, K, fmt)
    sb, db = fg.sfb_shape(G, N, K, fmt)
    return aq, torch.zeros(sa, dtype=da), bq, torch.zeros(sb, dtype=db)


@pytest.mark.parametrize("fmt", [0, 1])
def test_well_formed_calls_reach_the_library(fg, fmt):
    aq, sfa, bq, sfb = _fp8(fg, 64, 256, 512, fmt)
    fg.gemm_fp8_blockscaled(aq, sfa, bq, sfb, fmt)
    dq, sfd = fg.gemm_fp8_blockscaled_quant(aq, sfa, bq, sfb, fmt, 1 - fmt)
    assert dq.shape == (64, 256) and sfd.shape == fg.sfa_shape(64, 256, 1 - fmt)[0]
    fg.quantize_1x128(torch.zeros((64, 512), dtype=torch.bfloat16), fmt)
    fg.quantize_128x128(torch.zeros((256, 512), dtype=torch.bfloat16), fmt)
    assert fg.recorder.calls == ["gemm_fp8_blockscaled", "gemm_fp8_blockscaled_quant", "quantize_1x128",
                                 "quantize_128x128"]


def test_short_scale_tables_are_rejected(fg):
    aq, sfa, bq, sfb = _fp8(fg, 64, 256, 512, 0)
    with pytest.raises(ValueError, match="sfa"):
        fg.gemm_fp8_blockscaled(aq, sfa[:, :32], bq, sfb, 0)
    with pytest.raises(ValueError, match="sfb"):
        fg.gemm_fp8_blockscaled(aq, sfa, bq, sfb[:, :1], 0)
    with pytest.raises(ValueError, match="sfa"):                       # FP32 table under UE8M0
        fg.gemm_fp8_blockscaled(aq, sfa, bq, _fp8(fg, 64, 256, 512, 1)[3], 1)
    assert fg.recorder.calls == []


def test_mismatched_operands_and_outputs_are_rejected(fg):
    aq, sfa, bq, sfb = _fp8(fg, 64, 256, 512, 1)
    with pytest.raises(ValueError, match="bq"):                        # B with another K
        fg.gemm_fp8_blockscaled(aq, sfa, torch.zeros((256, 384), dtype=torch.uint8), sfb, 1)
    with pytest.raises(ValueError, match="out"):
        fg.gemm_fp8_blockscaled(aq, sfa, bq, sfb, 1, out=torch.zeros((64, 255), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="out"):
        fg.gemm_fp8_blockscaled(aq, sfa, bq, sfb, 1, out=torch.zeros((64, 256), dtype=torch.float32))
    with pytest.raises(ValueError, match="sfd"):
        fg.gemm_fp8_blockscaled_quant(aq, sfa, bq, sfb, 1, 0, sfd=torch.zeros((2, 60), dtype=torch.float32))
    with pytest.raises(ValueError, match="xq"):
        fg.quantize_1x128(torch.zeros((64, 512), dtype=torch.bfloat16), 1, xq=torch.zeros((64, 256), dtype=torch.uint8))
    with pytest.raises(ValueError, match="bf16"):
        fg.quantize_1x128(torch.zeros((64, 512), dtype=torch.float32), 1)
    assert fg.recorder.calls == []


def test_grouped_checks(fg):
    G, Mmax, N, K, fmt = 4, 64, 256, 256, 0
    aq = torch.zeros((G, Mmax, K), dtype=torch.uint8)
    sa, da = fg.sfa_shape(Mmax, K, fmt)
    sfa = torch.zeros((G, *sa), dtype=da)
    bq = torch.zeros((G, N, K), dtype=torch.uint8)
    sb, db = fg.sfb_shape(G, N, K, fmt)
    sfb = torch.zeros(sb, dtype=db)
    fg.grouped_fp8_masked(aq, sfa, bq, sfb, torch.zeros(G, dtype=torch.int32), fmt)
    with pytest.raises(ValueError, match="masked_m"):
        fg.grouped_fp8_masked(aq, sfa, bq, sfb, torch.zeros(G - 1, dtype=torch.int32), fmt)
    with pytest.raises(ValueError, match="sfa"):
        fg.grouped_fp8_masked(aq, sfa[:2], bq, sfb, torch.zeros(G, dtype=torch.int32), fmt)
    M = 512
    a2, s2, b2, t2 = _fp8(fg, M, N, K, fmt, G=G)
    fg.grouped_fp8_contiguous(a2, s2, b2, t2, torch.zeros(M, dtype=torch.int32), fmt)
    with pytest.raises(ValueError, match="m_indices"):
        fg.grouped_fp8_contiguous(a2, s2, b2, t2, torch.zeros(M - 128, dtype=torch.int32), fmt)
    assert fg.recorder.calls == ["grouped_fp8_masked", "grouped_fp8_contiguous"]


def test_tensors_on_another_device_are_rejected():
    """Every tensor of a call must sit on the launch stream's device (a pointer
    into another GPU's memory would reach the kernel's tensor maps)."""
    from fine_grained_fp8_persistent_gb300 import binding
    d0, d1 = torch.device("cuda:0"), torch.device("cuda:1")
    on0, on1 = SimpleNamespace(device=d0), SimpleNamespace(device=d1)
    binding.same_device(d0, aq=on0, sfa=on0, out=None)
    with pytest.raises(ValueError, match="sfb is on cuda:1"):
        binding.same_device(d0, aq=on0, sfb=on1)
    with pytest.raises(ValueError, match="launch stream is on cuda:1"):
        binding.same_device(d1, x=on0)
