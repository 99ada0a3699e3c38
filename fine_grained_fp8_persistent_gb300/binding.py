"""ctypes binding of libfgf8.so (include/fgf8.h).

Argument marshalling only: shapes and raw device pointers go to the C ABI, the
caller's current torch CUDA stream is passed as the stream, and outputs are
allocated with torch.empty when the caller does not provide them.  Every step of
the computation runs in the library's CUDA kernels; there is no fallback.  If
the library has not been built, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfgf8.so")

SCALE_F32 = 0
SCALE_UE8M0 = 1
FP4_MX = 0     # MXFP4: E2M1 + E8M0 scale per 32 elements along K
FP4_NV = 1     # NVFP4: E2M1 + E4M3 scale per 16 elements along K
F16 = 0
BF16 = 1

OK = 0
ERR_DEVICE_TIMEOUT = 5
ERR_DEVICE_INPUT = 6


class FGF8Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} (fgf8 status {code})")
        self.code = code


if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)
_P = ctypes.c_void_p
_I = ctypes.c_int
_LL = ctypes.c_longlong

_SIGS = {
    "quantize_1x128": ([_P, _P, _P, _I, _I, _I, _P], _I),
    "quantize_128x128": ([_P, _P, _P, _I, _I, _I, _I, _P], _I),
    "gemm_f16": ([_P, _P, _P, _I, _I, _I, _I, _I, _P], _I),
    "gemm_fp8_blockscaled": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "gemm_fp8_blockscaled_quant": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P], _I),
    "grouped_fp8_contiguous": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P], _I),
    "grouped_fp8_masked": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P], _I),
    "quantize_fp4": ([_P, _P, _P, _I, _I, _I, _P], _I),
    "gemm_fp4_blockscaled": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "fgf8_fp4_sf_bytes": ([_I, _I, _I], _LL),
    "fgf8_mk_alignment_for_contiguous": ([], _I),
    "fgf8_sfa_bytes": ([_I, _I, _I], _LL),
    "fgf8_sfb_bytes": ([_I, _I, _I, _I], _LL),
    "fgf8_check_status": ([_P, ctypes.POINTER(ctypes.c_uint)], _I),
    "fgf8_last_error": ([], ctypes.c_char_p),
    "fgf8_last_tile": ([], ctypes.c_char_p),
    "fgf8_set_wait_timeout_ms": ([_I], _I),
    "fgf8_selftest_wait_timeout": ([_P], _I),
    "fgf8_set_pdl": ([_I], _I),
    "fgf8_set_scheduler": ([_I], _I),
    "fgf8_set_sm_cap": ([_I], _I),
    "fgf8_persistent_clusters": ([_LL, _I, _I, _I, _I], _LL),
    "fgf8_version": ([], _I),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


def lib() -> ctypes.CDLL:
    """The loaded shared library (for callers that pass raw pointers)."""
    return _lib


def last_error() -> str:
    return (_lib.fgf8_last_error() or b"").decode()


def _check(rc: int, name: str) -> None:
    if rc != OK:
        raise FGF8Error(rc, f"{name}: {last_error()}")


def _fmt(fmt) -> int:
    if isinstance(fmt, str):
        return {"f32": SCALE_F32, "fp32": SCALE_F32, "ue8m0": SCALE_UE8M0}[fmt.lower()]
    return int(fmt)


class _Stream:
    """The stream of one library call and its device."""

    def __init__(self, handle: int, device):
        self.handle = handle
        self.device = device


def same_device(device, **tensors) -> None:
    """Raise ValueError unless every given tensor lives on `device` (the launch
    stream's device).  The C ABI sees raw pointers only: a tensor of another GPU
    would put that GPU's memory under the kernel's tensor maps."""
    for name, t in tensors.items():
        if t is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device} but the launch stream is on {device}")


def _stream(stream=None, **tensors) -> _Stream:
    """The launch stream (the given one, else the current stream of the tensors'
    device), after checking that every tensor lives on its device."""
    if stream is None:
        first = next((t for t in tensors.values() if t is not None), None)
        stream = torch.cuda.current_stream(None if first is None else first.device)
    same_device(stream.device, **tensors)
    return _Stream(stream.cuda_stream, stream.device)


def _call(name: str, st: _Stream, *args) -> None:
    """Run one library entry point with the stream's device current (the library
    takes the device from cudaGetDevice) and raise FGF8Error on failure."""
    with torch.cuda.device(st.device):
        rc = getattr(_lib, name)(*args, st.handle)
    _check(rc, name)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _u8(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.uint8) if t.dtype != torch.uint8 else t


# The C ABI takes raw pointers and cannot see buffer sizes, so the binding checks
# every tensor it passes against the sizes the call will touch.
def _need(t: torch.Tensor, numel: int, itemsize: int, name: str) -> None:
    """An input or scale table: exactly `numel` elements of `itemsize` bytes."""
    if t.numel() != numel or t.element_size() != itemsize:
        raise ValueError(f"{name}: expected {numel} elements of {itemsize} bytes, "
                         f"got {t.numel()} of {t.element_size()} ({t.dtype}, {tuple(t.shape)})")


def _need_out(t: torch.Tensor, shape: tuple, dtypes: tuple, name: str) -> None:
    """An output: exactly this shape and one of these dtypes."""
    if tuple(t.shape) != tuple(shape) or t.dtype not in dtypes:
        raise ValueError(f"{name}: expected {dtypes[0]} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")


def _numel(shape) -> int:
    n = 1
    for d in shape:
        n *= d
    return n


def _need_fp8(aq, sfa, bq, sfb, fmt, rows: int, G: int, N: int, K: int) -> None:
    """E4M3 operands and their scale tables for `rows` activation rows and G
    experts of N x K weights."""
    _need(aq, rows * K, 1, "aq")
    _need(bq, G * N * K, 1, "bq")
    _need(sfa, _numel(sfa_shape(rows, K, fmt)[0]), 4, "sfa")
    _need(sfb, _numel(sfb_shape(G, N, K, fmt)[0]), 4, "sfb")


def align4(x: int) -> int:
    return (int(x) + 3) // 4 * 4


def sfa_shape(rows: int, K: int, fmt) -> tuple[tuple[int, ...], torch.dtype]:
    nkb = K // 128
    if _fmt(fmt) == SCALE_F32:
        return (nkb, align4(rows)), torch.float32
    return ((nkb + 3) // 4, align4(rows)), torch.int32


def sfb_shape(G: int, N: int, K: int, fmt) -> tuple[tuple[int, ...], torch.dtype]:
    nkb = K // 128
    if _fmt(fmt) == SCALE_F32:
        return (G, (N + 127) // 128, nkb), torch.float32
    return (G, (nkb + 3) // 4, align4(N)), torch.int32


# --------------------------------------------------------------------------- quantize
def quantize_1x128(x: torch.Tensor, fmt, xq: torch.Tensor | None = None,
                   sfa: torch.Tensor | None = None, stream=None):
    """bf16 (M, K) -> (E4M3 codes uint8 (M, K), activation scale table)."""
    M, K = x.shape
    if x.dtype != torch.bfloat16:
        raise ValueError("x must be bf16")
    shape, dt = sfa_shape(M, K, fmt)
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sfa is None:
        sfa = torch.empty(shape, dtype=dt, device=x.device)
    _need(xq, M * K, 1, "xq")
    _need(sfa, _numel(shape), 4, "sfa")
    st = _stream(stream, x=x, xq=xq, sfa=sfa)
    _call("quantize_1x128", st, _ptr(x), _ptr(_u8(xq)), _ptr(sfa), M, K, _fmt(fmt))
    return xq, sfa


def quantize_128x128(w: torch.Tensor, fmt, wq: torch.Tensor | None = None,
                     sfb: torch.Tensor | None = None, stream=None):
    """bf16 (N, K) or (G, N, K) -> (E4M3 codes, weight scale table with a G axis)."""
    G, N, K = (1, *w.shape) if w.dim() == 2 else w.shape
    if w.dtype != torch.bfloat16:
        raise ValueError("w must be bf16")
    shape, dt = sfb_shape(G, N, K, fmt)
    if wq is None:
        wq = torch.empty(tuple(w.shape), dtype=torch.uint8, device=w.device)
    if sfb is None:
        sfb = torch.empty(shape, dtype=dt, device=w.device)
    _need(wq, G * N * K, 1, "wq")
    _need(sfb, _numel(shape), 4, "sfb")
    st = _stream(stream, w=w, wq=wq, sfb=sfb)
    _call("quantize_128x128", st, _ptr(w), _ptr(_u8(wq)), _ptr(sfb), G, N, K, _fmt(fmt))
    return wq, sfb


# --------------------------------------------------------------------------- GEMM
def gemm_f16(a: torch.Tensor, b: torch.Tensor, out_dtype: torch.dtype | None = None,
             out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """D = A B^T for fp16/bf16 A (M, K), B (N, K); FP32 accumulation."""
    M, K = a.shape
    N = b.shape[0]
    if a.dtype != b.dtype or a.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("A and B must both be fp16 or both bf16")
    if tuple(b.shape) != (N, K):
        raise ValueError(f"b: expected {(N, K)}, got {tuple(b.shape)}")
    out_dtype = out_dtype or a.dtype
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    _need_out(out, (M, N), (torch.float16, torch.bfloat16), "out")
    in_code = BF16 if a.dtype == torch.bfloat16 else F16
    out_code = BF16 if out.dtype == torch.bfloat16 else F16
    st = _stream(stream, a=a, b=b, out=out)
    _call("gemm_f16", st, _ptr(a), _ptr(b), _ptr(out), M, N, K, in_code, out_code)
    return out


def gemm_fp8_blockscaled(aq, sfa, bq, sfb, fmt, out: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """D (bf16, M x N) from E4M3 A (M, K) / B (N, K) with fine-grained scales."""
    M, K = aq.shape
    N = bq.shape[-2]
    _need_fp8(aq, sfa, bq, sfb, fmt, M, 1, N, K)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=aq.device)
    _need_out(out, (M, N), (torch.bfloat16,), "out")
    st = _stream(stream, aq=aq, sfa=sfa, bq=bq, sfb=sfb, out=out)
    _call("gemm_fp8_blockscaled", st, _ptr(_u8(aq)), _ptr(sfa), _ptr(_u8(bq)), _ptr(sfb), _ptr(out),
          M, N, K, _fmt(fmt))
    return out


def gemm_fp8_blockscaled_quant(aq, sfa, bq, sfb, fmt, out_fmt, dq: torch.Tensor | None = None,
                               sfd: torch.Tensor | None = None, stream=None):
    """The block-scaled GEMM with its output quantized 1x128 in the epilogue:
    returns (Dq uint8 (M, N) E4M3 codes, SFD scale table in out_fmt), equal to
    quantize_1x128(gemm_fp8_blockscaled(...), out_fmt)."""
    M, K = aq.shape
    N = bq.shape[-2]
    _need_fp8(aq, sfa, bq, sfb, fmt, M, 1, N, K)
    shape, dt = sfa_shape(M, N, out_fmt)
    if dq is None:
        dq = torch.empty((M, N), dtype=torch.uint8, device=aq.device)
    if sfd is None:
        sfd = torch.empty(shape, dtype=dt, device=aq.device)
    _need(dq, M * N, 1, "dq")
    _need(sfd, _numel(shape), 4, "sfd")
    st = _stream(stream, aq=aq, sfa=sfa, bq=bq, sfb=sfb, dq=dq, sfd=sfd)
    _call("gemm_fp8_blockscaled_quant", st, _ptr(_u8(aq)), _ptr(sfa), _ptr(_u8(bq)), _ptr(sfb), _ptr(dq),
          _ptr(sfd), M, N, K, _fmt(fmt), _fmt(out_fmt))
    return dq, sfd


def grouped_fp8_contiguous(aq, sfa, bq, sfb, m_indices, fmt, out: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """Contiguous-layout MoE GEMM: rows of expert g use B[g]; m_indices -1 = padding."""
    M, K = aq.shape
    G, N, _ = bq.shape
    _need_fp8(aq, sfa, bq, sfb, fmt, M, G, N, K)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=aq.device)
    _need_out(out, (M, N), (torch.bfloat16,), "out")
    if m_indices.dtype != torch.int32 or m_indices.numel() != M:
        raise ValueError("m_indices must be int32 with one entry per row")
    st = _stream(stream, aq=aq, sfa=sfa, bq=bq, sfb=sfb, m_indices=m_indices, out=out)
    _call("grouped_fp8_contiguous", st, _ptr(_u8(aq)), _ptr(sfa), _ptr(_u8(bq)), _ptr(sfb),
          _ptr(m_indices), _ptr(out), M, N, K, G, _fmt(fmt))
    return out


def grouped_fp8_masked(aq, sfa, bq, sfb, masked_m, fmt, expected_m: int = 0,
                       out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Masked-layout MoE GEMM: A (G, Mmax, K); rows >= masked_m[g] are not computed."""
    G, Mmax, K = aq.shape
    N = bq.shape[1]
    _need(aq, G * Mmax * K, 1, "aq")
    _need(bq, G * N * K, 1, "bq")
    _need(sfa, G * _numel(sfa_shape(Mmax, K, fmt)[0]), 4, "sfa")
    _need(sfb, _numel(sfb_shape(G, N, K, fmt)[0]), 4, "sfb")
    if out is None:
        out = torch.empty((G, Mmax, N), dtype=torch.bfloat16, device=aq.device)
    _need_out(out, (G, Mmax, N), (torch.bfloat16,), "out")
    if masked_m.dtype != torch.int32 or masked_m.numel() != G:
        raise ValueError("masked_m must be int32 with one entry per expert")
    st = _stream(stream, aq=aq, sfa=sfa, bq=bq, sfb=sfb, masked_m=masked_m, out=out)
    _call("grouped_fp8_masked", st, _ptr(_u8(aq)), _ptr(sfa), _ptr(_u8(bq)), _ptr(sfb),
          _ptr(masked_m), _ptr(out), G, Mmax, N, K, int(expected_m), _fmt(fmt))
    return out


# --------------------------------------------------------------------------- 4-bit
def _fp4(fmt) -> int:
    if isinstance(fmt, str):
        return {"mx": FP4_MX, "mxfp4": FP4_MX, "nv": FP4_NV, "nvfp4": FP4_NV}[fmt.lower()]
    return int(fmt)


def fp4_sf_shape(rows: int, K: int, fmt) -> tuple[tuple[int, ...], torch.dtype]:
    """Scale table of quantize_fp4: int32 [ceil(K / SV / 4)][align4(rows)]."""
    sv = 32 if _fp4(fmt) == FP4_MX else 16
    return ((K // sv + 3) // 4, align4(rows)), torch.int32


def quantize_fp4(x: torch.Tensor, fmt, xq: torch.Tensor | None = None, sf: torch.Tensor | None = None,
                 stream=None):
    """bf16 (R, K) -> (packed E2M1 codes uint8 (R, K/2), scale table), MXFP4 or NVFP4."""
    R, K = x.shape
    if x.dtype != torch.bfloat16:
        raise ValueError("x must be bf16")
    shape, dt = fp4_sf_shape(R, K, fmt)
    if xq is None:
        xq = torch.empty((R, K // 2), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty(shape, dtype=dt, device=x.device)
    _need(xq, R * (K // 2), 1, "xq")
    _need(sf, _numel(shape), 4, "sf")
    st = _stream(stream, x=x, xq=xq, sf=sf)
    _call("quantize_fp4", st, _ptr(x), _ptr(xq), _ptr(sf), R, K, _fp4(fmt))
    return xq, sf


def gemm_fp4_blockscaled(aq, sfa, bq, sfb, fmt, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """D (bf16, M x N) from packed E2M1 A (M, K/2) / B (N, K/2) with MXFP4 or NVFP4 scales."""
    M, Kh = aq.shape
    N = bq.shape[0]
    K = 2 * Kh
    _need(aq, M * Kh, 1, "aq")
    _need(bq, N * Kh, 1, "bq")
    _need(sfa, _numel(fp4_sf_shape(M, K, fmt)[0]), 4, "sfa")
    _need(sfb, _numel(fp4_sf_shape(N, K, fmt)[0]), 4, "sfb")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=aq.device)
    _need_out(out, (M, N), (torch.bfloat16,), "out")
    st = _stream(stream, aq=aq, sfa=sfa, bq=bq, sfb=sfb, out=out)
    _call("gemm_fp4_blockscaled", st, _ptr(aq), _ptr(sfa), _ptr(bq), _ptr(sfb), _ptr(out), M, N, K, _fp4(fmt))
    return out


# --------------------------------------------------------------------------- utilities
def check_status(stream=None) -> tuple[int, int]:
    """Synchronise the stream; return (status code, raw device status bits)."""
    bits = ctypes.c_uint(0)
    s = torch.cuda.current_stream() if stream is None else stream
    rc = _lib.fgf8_check_status(s.cuda_stream, ctypes.byref(bits))
    return rc, bits.value


def mk_alignment_for_contiguous() -> int:
    return int(_lib.fgf8_mk_alignment_for_contiguous())


def sfa_bytes(rows: int, K: int, fmt) -> int:
    return int(_lib.fgf8_sfa_bytes(rows, K, _fmt(fmt)))


def sfb_bytes(G: int, N: int, K: int, fmt) -> int:
    return int(_lib.fgf8_sfb_bytes(G, N, K, _fmt(fmt)))


def last_tile() -> str:
    """Kernel configuration of the last GEMM this thread launched ("mxf8 dense 2x224")."""
    return (_lib.fgf8_last_tile() or b"").decode()


def selftest_wait_timeout(stream=None) -> None:
    """Run the bounded-wait self-test: a wait on a barrier nothing signals, which
    must give up after the current limit and leave FGF8_ERR_DEVICE_TIMEOUT (raw bits
    0x801) for the next check_status()."""
    s = torch.cuda.current_stream() if stream is None else stream
    _check(_lib.fgf8_selftest_wait_timeout(s.cuda_stream), "fgf8_selftest_wait_timeout")


def set_pdl(enable: bool) -> bool:
    """Turn programmatic dependent launch on or off; returns the previous setting."""
    return bool(_lib.fgf8_set_pdl(1 if enable else 0))


SCHED_STATIC = 0
SCHED_CLC = 1


def set_scheduler(mode: int) -> int:
    """Tile scheduler of the GEMMs: SCHED_STATIC (persistent grid, static round
    robin) or SCHED_CLC (one cluster per tile, cluster launch control hands out the
    tiles of clusters not yet launched); returns the previous mode."""
    return int(_lib.fgf8_set_scheduler(int(mode)))


def set_sm_cap(enable: bool) -> bool:
    """Wave-preserving SM cap of the static persistent grid; returns the previous setting."""
    return bool(_lib.fgf8_set_sm_cap(1 if enable else 0))


def persistent_clusters(tiles: int, cluster: int, sms: int, max_clusters: int, cap: bool) -> int:
    """Clusters of the static persistent grid the launcher picks (host arithmetic)."""
    return int(_lib.fgf8_persistent_clusters(int(tiles), int(cluster), int(sms), int(max_clusters), 1 if cap else 0))


def set_wait_timeout_ms(ms: int) -> int:
    return int(_lib.fgf8_set_wait_timeout_ms(int(ms)))


def version() -> int:
    return int(_lib.fgf8_version())
