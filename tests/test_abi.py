"""CPU-only checks of the C ABI: the library builds, loads, exports every symbol
include/fgf8.h declares, and rejects invalid calls on the host (error codes and
messages) without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fgf8.h")


@pytest.fixture(scope="module")
def lib():
    from fine_grained_fp8_persistent_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"^FGF8_API\s[^(]*?([A-Za-z_0-9]+)\(", text, flags=re.M)


def test_header_declares_the_entry_points():
    names = set(declared_symbols())
    for n in ("gemm_f16", "gemm_fp8_blockscaled", "grouped_fp8_contiguous", "grouped_fp8_masked",
              "quantize_1x128", "quantize_128x128", "fgf8_check_status", "fgf8_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_only_declared_symbols_are_exported():
    import subprocess
    from fine_grained_fp8_persistent_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm not available")
    exported = {l.split()[-1] for l in out.stdout.splitlines() if l.strip()}
    assert exported == set(declared_symbols())


def _err(lib):
    lib.fgf8_last_error.restype = ctypes.c_char_p
    return lib.fgf8_last_error().decode()


def test_host_validation(lib):
    P = ctypes.c_void_p
    al = P(0x10000)           # 16-byte aligned, never dereferenced (validation fails first)
    mis = P(0x10001)
    f = lib.quantize_1x128
    f.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
    assert f(al, al, al, 4, 100, 0, None) == 2 and "multiple of 128" in _err(lib)
    assert f(al, al, al, -1, 128, 0, None) == 1
    assert f(al, al, al, 4, 128, 7, None) == 1
    assert f(None, al, al, 4, 128, 0, None) == 1
    assert f(mis, al, al, 4, 128, 0, None) == 3
    assert f(None, None, None, 0, 128, 0, None) == 0          # empty problem: no-op
    g = lib.gemm_f16
    g.argtypes = [P, P, P] + [ctypes.c_int] * 5 + [P]
    assert g(al, al, al, 16, 12, 16, 0, 0, None) == 2        # N % 8
    assert g(al, al, al, 16, 16, 16, 3, 0, None) == 1        # dtype
    assert g(al, mis, al, 16, 16, 16, 0, 0, None) == 3
    h = lib.grouped_fp8_masked
    h.argtypes = [P] * 6 + [ctypes.c_int] * 6 + [P]
    assert h(al, al, al, al, al, al, 2000, 64, 128, 128, 0, 0, None) == 2   # G > 1024
    assert h(al, al, al, al, al, al, 4, 64, 128, 100, 0, 0, None) == 2      # K % 128
    c = lib.grouped_fp8_contiguous
    c.argtypes = [P] * 6 + [ctypes.c_int] * 5 + [P]
    assert c(al, al, al, al, al, al, 100, 128, 128, 2, 0, None) == 2        # M % 128
    q = lib.gemm_fp8_blockscaled_quant
    q.argtypes = [P] * 6 + [ctypes.c_int] * 5 + [P]
    assert q(al, al, al, al, al, al, 64, 256, 256, 2, 0, None) == 1         # input format
    assert q(al, al, al, al, al, al, 64, 200, 256, 1, 0, None) == 2         # N % 128
    assert q(al, al, al, al, al, al, 64, 256, 256, 1, 5, None) == 1         # output format
    assert q(al, al, al, al, mis, al, 64, 256, 256, 1, 0, None) == 3
    assert q(al, al, al, al, al, None, 64, 256, 256, 1, 1, None) == 1
    assert q(None, None, None, None, None, None, 0, 256, 256, 1, 1, None) == 0


def test_host_validation_fp4(lib):
    P = ctypes.c_void_p
    al = P(0x10000)
    q = lib.quantize_fp4
    q.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
    assert q(al, al, al, 4, 96, 0, None) == 2 and "multiple of 64" in _err(lib)
    assert q(al, al, al, 4, 128, 2, None) == 1
    assert q(al, al, al, -1, 128, 0, None) == 1
    assert q(None, None, None, 0, 128, 1, None) == 0
    g = lib.gemm_fp4_blockscaled
    g.argtypes = [P] * 5 + [ctypes.c_int] * 4 + [P]
    assert g(al, al, al, al, al, 16, 64, 128, 0, None) == 2 and "multiple of 256" in _err(lib)
    assert g(al, al, al, al, al, 16, 48, 256, 0, None) == 2 and "multiple of 32" in _err(lib)
    assert g(al, al, al, al, al, 16, 64, 256, 3, None) == 1
    assert g(al, P(0x10004), al, al, al, 16, 64, 256, 1, None) == 3
    assert g(None, None, None, None, None, 0, 64, 256, 1, None) == 0
    lib.fgf8_fp4_sf_bytes.restype = ctypes.c_longlong
    assert lib.fgf8_fp4_sf_bytes(4096, 7168, 0) == 56 * 4096 * 4      # 224 groups of 32
    assert lib.fgf8_fp4_sf_bytes(37, 7168, 1) == 112 * 40 * 4         # 448 groups of 16
    assert lib.fgf8_fp4_sf_bytes(8, 64, 0) == 1 * 8 * 4               # 2 groups: half a word
    assert lib.fgf8_fp4_sf_bytes(8, 100, 0) == -1


def test_size_helpers(lib):
    lib.fgf8_sfa_bytes.restype = ctypes.c_longlong
    lib.fgf8_sfb_bytes.restype = ctypes.c_longlong
    assert lib.fgf8_mk_alignment_for_contiguous() == 128
    assert lib.fgf8_sfa_bytes(4096, 7168, 0) == 56 * 4096 * 4
    assert lib.fgf8_sfa_bytes(37, 640, 1) == 2 * 40 * 4
    assert lib.fgf8_sfb_bytes(8, 4096, 7168, 0) == 8 * 32 * 56 * 4
    assert lib.fgf8_sfb_bytes(1, 300, 512, 1) == 1 * 1 * 300 * 4
    assert lib.fgf8_sfa_bytes(4, 100, 0) == -1
    assert lib.fgf8_version() >= 100
