"""fine_grained_fp8_persistent_gb300 -- fine-grained FP8 NT GEMM engine for GB300.

The compute lives in libfgf8.so (hand-written sm_103a CUDA kernels behind the C
ABI in include/fgf8.h).  The names below come from ``binding`` and are loaded on
first use, so ``fine_grained_fp8_persistent_gb300.inputs`` (seeded synthetic
inputs) can be imported on machines where the library is not built.
"""
from __future__ import annotations

_EXPORTS = (
    "quantize_1x128", "quantize_128x128", "gemm_f16", "gemm_fp8_blockscaled", "gemm_fp8_blockscaled_quant",
    "grouped_fp8_contiguous", "grouped_fp8_masked", "check_status",
    "mk_alignment_for_contiguous", "sfa_bytes", "sfb_bytes", "sfa_shape", "sfb_shape",
    "set_wait_timeout_ms", "set_pdl", "selftest_wait_timeout", "last_error", "last_tile", "version", "FGF8Error", "SCALE_F32", "SCALE_UE8M0",
)


def __getattr__(name):
    if name in _EXPORTS:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)


__all__ = list(_EXPORTS)
