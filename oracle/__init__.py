"""CPU oracle for the fine-grained FP8 GEMM path (TEST INFRASTRUCTURE ONLY).

The arithmetic lives in ``fgf8_oracle.c`` (plain C, fp64 accumulation).  This
module builds it with gcc and wraps it for numpy arrays.  It shares no code with
the CUDA library and never imports it.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline`` leg may use it.

Parity unpinned: none.  Every function is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

SCALE_F32 = 0
SCALE_UE8M0 = 1
FP4_MX = 0   # MXFP4: E2M1 elements, E8M0 scale per 32 along K
FP4_NV = 1   # NVFP4: E2M1 elements, E4M3 scale per 16 along K

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fgf8_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfgf8_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        L = ctypes.c_long
        I = ctypes.c_int
        lib.fgo_e4m3_decode.restype = ctypes.c_double
        lib.fgo_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.fgo_e4m3_encode.restype = ctypes.c_uint8
        lib.fgo_e4m3_encode.argtypes = [ctypes.c_double]
        lib.fgo_e4m3_encode_array.argtypes = [P, P, L]
        lib.fgo_e4m3_decode_array.argtypes = [P, P, L]
        lib.fgo_align4.restype = L
        lib.fgo_align4.argtypes = [L]
        lib.fgo_quantize_1x128.argtypes = [P, L, L, I, P, P]
        lib.fgo_quantize_128x128.argtypes = [P, L, L, L, I, P, P]
        lib.fgo_gemm_fp8.argtypes = [P, P, P, P, L, L, L, I, P]
        lib.fgo_gemm_fp8_entries.argtypes = [P, P, P, P, L, L, L, I, P, P, L, P]
        lib.fgo_grouped_contiguous.argtypes = [P, P, P, P, P, L, L, L, L, I, P, P]
        lib.fgo_grouped_masked.argtypes = [P, P, P, P, P, L, L, L, L, I, P, P]
        lib.fgo_gemm_f16.argtypes = [P, P, L, L, L, P]
        lib.fgo_gemm_f16_entries.argtypes = [P, P, L, L, L, P, P, L, P]
        lib.fgo_e2m1_decode.restype = ctypes.c_double
        lib.fgo_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.fgo_e2m1_encode.restype = ctypes.c_uint8
        lib.fgo_e2m1_encode.argtypes = [ctypes.c_double]
        lib.fgo_e2m1_encode_array.argtypes = [P, P, L]
        lib.fgo_e2m1_decode_array.argtypes = [P, P, L]
        lib.fgo_fp4_scale_value.restype = ctypes.c_double
        lib.fgo_fp4_scale_value.argtypes = [ctypes.c_uint8, I]
        lib.fgo_quantize_fp4.argtypes = [P, L, L, I, P, P]
        lib.fgo_gemm_fp4.argtypes = [P, P, P, P, L, L, L, I, P]
        lib.fgo_num_threads.restype = I
        lib.fgo_set_num_threads.argtypes = [I]
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _u8(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.uint8))


def _sf_buffer(sf) -> np.ndarray:
    """Scale tables travel as raw bytes (float32 or packed int32)."""
    a = np.ascontiguousarray(np.asarray(sf))
    return a


def align4(x: int) -> int:
    return (int(x) + 3) // 4 * 4


def num_threads() -> int:
    return int(_load().fgo_num_threads())


def set_num_threads(n: int) -> None:
    _load().fgo_set_num_threads(int(n))


# --------------------------------------------------------------------------- E4M3
def e4m3_decode(codes) -> np.ndarray:
    q = _u8(codes)
    out = np.empty(q.shape, dtype=np.float64)
    _load().fgo_e4m3_decode_array(_ptr(q), _ptr(out), q.size)
    return out


def e4m3_encode(values) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float64))
    out = np.empty(v.shape, dtype=np.uint8)
    _load().fgo_e4m3_encode_array(_ptr(v), _ptr(out), v.size)
    return out


# --------------------------------------------------------------------------- scales
def sfa_shape(M: int, K: int, fmt: int):
    """(rows, cols, dtype) of an activation scale table for M rows."""
    nkb = K // 128
    if fmt == SCALE_F32:
        return (nkb, align4(M)), np.float32
    return ((nkb + 3) // 4, align4(M)), np.int32


def sfb_shape(G: int, N: int, K: int, fmt: int):
    nkb = K // 128
    if fmt == SCALE_F32:
        return (G, (N + 127) // 128, nkb), np.float32
    return (G, (nkb + 3) // 4, align4(N)), np.int32


def quantize_1x128(X, fmt: int):
    """X: (M, K) float32 (bf16 values). Returns (Xq uint8 (M,K), SFA)."""
    x = _f32(X)
    M, K = x.shape
    assert K % 128 == 0
    q = np.empty((M, K), dtype=np.uint8)
    shape, dt = sfa_shape(M, K, fmt)
    sf = np.empty(shape, dtype=dt)
    _load().fgo_quantize_1x128(_ptr(x), M, K, fmt, _ptr(q), _ptr(sf))
    return q, sf


def quantize_128x128(W, fmt: int):
    """W: (G, N, K) or (N, K) float32. Returns (Wq, SFB) with a leading G axis."""
    w = _f32(W)
    if w.ndim == 2:
        w = w[None]
    G, N, K = w.shape
    assert K % 128 == 0
    q = np.empty((G, N, K), dtype=np.uint8)
    shape, dt = sfb_shape(G, N, K, fmt)
    sf = np.empty(shape, dtype=dt)
    _load().fgo_quantize_128x128(_ptr(w), G, N, K, fmt, _ptr(q), _ptr(sf))
    return q, sf


# --------------------------------------------------------------------------- GEMM
def gemm_fp8(Aq, SFA, Bq, SFB, fmt: int) -> np.ndarray:
    a = _u8(Aq)
    b = _u8(Bq)
    if b.ndim == 3:
        assert b.shape[0] == 1
        b = b[0]
    M, K = a.shape
    N = b.shape[0]
    sfa = _sf_buffer(SFA)
    sfb = _sf_buffer(SFB)
    D = np.empty((M, N), dtype=np.float64)
    _load().fgo_gemm_fp8(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), M, N, K, fmt, _ptr(D))
    return D


def gemm_fp8_entries(Aq, SFA, Bq, SFB, fmt: int, rows, cols) -> np.ndarray:
    a = _u8(Aq)
    b = _u8(Bq)
    if b.ndim == 3:
        assert b.shape[0] == 1
        b = b[0]
    M, K = a.shape
    N = b.shape[0]
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    c = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    assert r.shape == c.shape
    out = np.empty(r.shape, dtype=np.float64)
    _load().fgo_gemm_fp8_entries(_ptr(a), _ptr(_sf_buffer(SFA)), _ptr(b), _ptr(_sf_buffer(SFB)),
                                 M, N, K, fmt, _ptr(r), _ptr(c), r.size, _ptr(out))
    return out


def grouped_contiguous(Aq, SFA, Bq, SFB, m_indices, fmt: int):
    """Returns (D float64 (M,N), valid uint8 (M,N))."""
    a = _u8(Aq)
    b = _u8(Bq)
    G, N, K = b.shape
    M = a.shape[0]
    mi = np.ascontiguousarray(np.asarray(m_indices, dtype=np.int32))
    assert mi.shape == (M,)
    D = np.zeros((M, N), dtype=np.float64)
    valid = np.zeros((M, N), dtype=np.uint8)
    _load().fgo_grouped_contiguous(_ptr(a), _ptr(_sf_buffer(SFA)), _ptr(b), _ptr(_sf_buffer(SFB)),
                                   _ptr(mi), M, N, K, G, fmt, _ptr(D), _ptr(valid))
    return D, valid


def grouped_masked(Aq, SFA, Bq, SFB, masked_m, fmt: int):
    """Aq: (G, Mmax, K). Returns (D float64 (G,Mmax,N), valid uint8)."""
    a = _u8(Aq)
    b = _u8(Bq)
    G, Mmax, K = a.shape
    N = b.shape[1]
    mm = np.ascontiguousarray(np.asarray(masked_m, dtype=np.int32))
    assert mm.shape == (G,)
    D = np.zeros((G, Mmax, N), dtype=np.float64)
    valid = np.zeros((G, Mmax, N), dtype=np.uint8)
    _load().fgo_grouped_masked(_ptr(a), _ptr(_sf_buffer(SFA)), _ptr(b), _ptr(_sf_buffer(SFB)),
                               _ptr(mm), G, Mmax, N, K, fmt, _ptr(D), _ptr(valid))
    return D, valid


def gemm_f16(A, B) -> np.ndarray:
    a = _f32(A)
    b = _f32(B)
    M, K = a.shape
    N = b.shape[0]
    D = np.empty((M, N), dtype=np.float64)
    _load().fgo_gemm_f16(_ptr(a), _ptr(b), M, N, K, _ptr(D))
    return D


def gemm_f16_entries(A, B, rows, cols) -> np.ndarray:
    a = _f32(A)
    b = _f32(B)
    M, K = a.shape
    N = b.shape[0]
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    c = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    out = np.empty(r.shape, dtype=np.float64)
    _load().fgo_gemm_f16_entries(_ptr(a), _ptr(b), M, N, K, _ptr(r), _ptr(c), r.size, _ptr(out))
    return out


# --------------------------------------------------------------------------- dequantize, then one matmul
# The block-scaled GEMM is, by definition, the GEMM of the dequantized operands
# ("DeepGEMM dissected", section "fine-grained quantization": x = q * s per 1x128
# group of A and per 128x128 block of B; "GPU GEMM part 4: tcgen05 & Blackwell",
# section 6 block-scaling formula).  The functions below take that definition
# literally: decode every code, multiply by its group's scale (both exact in
# fp64), then one float64 matmul from numpy as the library step.  They reach the
# triple-loop functions above up to fp64 summation order, and are what the
# full-size parity tests compare every output element against.
def a_scales(SFA, M: int, K: int, fmt: int) -> np.ndarray:
    """The (M, K/128) array of activation scales held in an SFA table."""
    nkb = K // 128
    sf = np.asarray(SFA)
    if fmt == SCALE_F32:
        return sf.astype(np.float64).reshape(nkb, -1)[:, :M].T.copy()
    b = np.ascontiguousarray(sf).view(np.uint8).reshape((nkb + 3) // 4, -1, 4)[:, :M, :]
    e = b.transpose(1, 0, 2).reshape(M, -1)[:, :nkb].astype(np.int64) - 127   # byte kb % 4 of word kb // 4
    return np.ldexp(1.0, e)


def b_scales(SFB, G: int, N: int, K: int, fmt: int) -> np.ndarray:
    """The (G, N, K/128) array of weight scales (each row n carries the scale of
    its 128-row block) held in an SFB table."""
    nkb = K // 128
    sf = np.asarray(SFB)
    if fmt == SCALE_F32:
        blocks = sf.astype(np.float64).reshape(G, (N + 127) // 128, nkb)
        return np.repeat(blocks, 128, axis=1)[:, :N, :]
    b = np.ascontiguousarray(sf).view(np.uint8).reshape(G, (nkb + 3) // 4, -1, 4)[:, :, :N, :]
    e = b.transpose(0, 2, 1, 3).reshape(G, N, -1)[:, :, :nkb].astype(np.int64) - 127
    return np.ldexp(1.0, e)


def dequantize_a(Aq, SFA, fmt: int) -> np.ndarray:
    """fp64 (M, K): decode(Aq[m, k]) * sA[m, k // 128]."""
    a = _u8(Aq)
    M, K = a.shape
    return e4m3_decode(a) * np.repeat(a_scales(SFA, M, K, fmt), 128, axis=1)


def dequantize_b(Bq, SFB, fmt: int) -> np.ndarray:
    """fp64 (G, N, K): decode(Bq[g, n, k]) * sB[g, n // 128, k // 128]."""
    b = _u8(Bq)
    if b.ndim == 2:
        b = b[None]
    G, N, K = b.shape
    return e4m3_decode(b) * np.repeat(b_scales(SFB, G, N, K, fmt), 128, axis=2)


def gemm_fp8_dequant(Aq, SFA, Bq, SFB, fmt: int) -> np.ndarray:
    """D = dequant(A) @ dequant(B)^T in float64 (the dense block-scaled GEMM)."""
    B = dequantize_b(Bq, SFB, fmt)
    assert B.shape[0] == 1
    return dequantize_a(Aq, SFA, fmt) @ B[0].T


def grouped_contiguous_dequant(Aq, SFA, Bq, SFB, m_indices, fmt: int):
    """Contiguous layout by dequantize-then-matmul per expert: (D, valid) as
    grouped_contiguous returns them (rows of padding or of an out-of-range
    expert: D 0, valid 0)."""
    A = dequantize_a(Aq, SFA, fmt)
    B = dequantize_b(Bq, SFB, fmt)
    G, N, _ = B.shape
    mi = np.asarray(m_indices)
    D = np.zeros((A.shape[0], N), dtype=np.float64)
    valid = np.zeros((A.shape[0], N), dtype=np.uint8)
    for g in range(G):
        rows = np.nonzero(mi == g)[0]
        if rows.size:
            D[rows] = A[rows] @ B[g].T
            valid[rows] = 1
    return D, valid


def grouped_masked_dequant(Aq, SFA, Bq, SFB, masked_m, fmt: int):
    """Masked layout by dequantize-then-matmul per expert: (D, valid) as
    grouped_masked returns them (rows >= masked_m[g]: D 0, valid 0)."""
    a = _u8(Aq)
    G, Mmax, K = a.shape
    sfa = np.asarray(SFA).reshape(G, -1)
    B = dequantize_b(Bq, SFB, fmt)
    N = B.shape[1]
    D = np.zeros((G, Mmax, N), dtype=np.float64)
    valid = np.zeros((G, Mmax, N), dtype=np.uint8)
    for g in range(G):
        m = int(min(max(int(masked_m[g]), 0), Mmax))
        if m:
            D[g, :m] = dequantize_a(a[g], sfa[g], fmt)[:m] @ B[g].T
            valid[g, :m] = 1
    return D, valid


def gemm_f16_matmul(A, B) -> np.ndarray:
    """D = A B^T of 16-bit operands (given as float32 holding their values) by
    one float64 matmul: every product of two 16-bit floats is exact in fp64
    ("TIRx and high-performance GEMM (part 2)", problem statement of the FP16
    NT GEMM), so this is the plain definition, summed in another order than
    gemm_f16's loop."""
    return _f32(A).astype(np.float64) @ _f32(B).astype(np.float64).T



# --------------------------------------------------------------------------- 4-bit formats
# MXFP4 / NVFP4 ("GPU GEMM part 4: tcgen05 & Blackwell", sections 6.1 block-scaled
# GEMM formula, 6.3 the two formats, 7.1 packing two elements per byte along K).
def e2m1_decode(codes) -> np.ndarray:
    q = _u8(codes)
    out = np.empty(q.shape, dtype=np.float64)
    _load().fgo_e2m1_decode_array(_ptr(q), _ptr(out), q.size)
    return out


def e2m1_encode(values) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float64))
    out = np.empty(v.shape, dtype=np.uint8)
    _load().fgo_e2m1_encode_array(_ptr(v), _ptr(out), v.size)
    return out


def fp4_vec(fmt: int) -> int:
    """Elements per scale along K: 32 (MXFP4) or 16 (NVFP4)."""
    return 32 if fmt == FP4_MX else 16


def fp4_sf_shape(R: int, K: int, fmt: int):
    """Scale table of R rows: int32 [ceil(K / SV / 4)][align4(R)]."""
    return ((K // fp4_vec(fmt) + 3) // 4, align4(R)), np.int32


def quantize_fp4(X, fmt: int):
    """X: (R, K) float32 (bf16 values).  Returns (Xq uint8 (R, K/2) packed E2M1,
    SF int32 scale table)."""
    x = _f32(X)
    R, K = x.shape
    assert K % 64 == 0
    q = np.empty((R, K // 2), dtype=np.uint8)
    shape, dt = fp4_sf_shape(R, K, fmt)
    sf = np.empty(shape, dtype=dt)
    _load().fgo_quantize_fp4(_ptr(x), R, K, fmt, _ptr(q), _ptr(sf))
    return q, sf


def fp4_unpack(Xq) -> np.ndarray:
    """(R, K/2) packed bytes -> (R, K) 4-bit codes (low nibble first)."""
    q = _u8(Xq)
    out = np.empty((q.shape[0], q.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = q & 0xF
    out[:, 1::2] = q >> 4
    return out


def fp4_scales(SF, R: int, K: int, fmt: int) -> np.ndarray:
    """The (R, K / SV) array of scale values held in a scale table."""
    ng = K // fp4_vec(fmt)
    b = np.ascontiguousarray(np.asarray(SF)).view(np.uint8).reshape((ng + 3) // 4, -1, 4)[:, :R, :]
    b = b.transpose(1, 0, 2).reshape(R, -1)[:, :ng]
    if fmt == FP4_MX:
        return np.ldexp(1.0, b.astype(np.int64) - 127)
    return e4m3_decode(b)


def dequantize_fp4(Xq, SF, fmt: int) -> np.ndarray:
    """fp64 (R, K): decode(code[r, k]) * scale[r, k // SV]."""
    codes = fp4_unpack(Xq)
    R, K = codes.shape
    return e2m1_decode(codes) * np.repeat(fp4_scales(SF, R, K, fmt), fp4_vec(fmt), axis=1)


def gemm_fp4(Aq, SFA, Bq, SFB, fmt: int) -> np.ndarray:
    """The block-scaled 4-bit NT GEMM term by term in fp64 (C triple loop)."""
    a, b = _u8(Aq), _u8(Bq)
    M, N, K = a.shape[0], b.shape[0], a.shape[1] * 2
    D = np.empty((M, N), dtype=np.float64)
    _load().fgo_gemm_fp4(_ptr(a), _ptr(_sf_buffer(SFA)), _ptr(b), _ptr(_sf_buffer(SFB)), M, N, K, fmt, _ptr(D))
    return D


def gemm_fp4_dequant(Aq, SFA, Bq, SFB, fmt: int) -> np.ndarray:
    """The same GEMM as dequantize-then-one-float64-matmul (the full-size form)."""
    return dequantize_fp4(Aq, SFA, fmt) @ dequantize_fp4(Bq, SFB, fmt).T
