"""CPU-side checks of the C ABI: the library builds and loads, exports every declared entry
point, and validates arguments on the host (no GPU call is made by these tests)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from gemm_uq_gb300.build import build
    build()
    import gemm_uq_gb300 as uq
    return uq.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "uq.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|uq_status)\s+(uq_\w+)\s*\(", src, re.M)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/uq.h but not exported by libuq.so"
    import gemm_uq_gb300 as uq
    assert set(names) == set(uq.SIGNATURES), "binding signatures out of sync with include/uq.h"


def test_status_strings(L):
    assert L.uq_status_string(0) == b"UQ_OK"
    assert L.uq_status_string(3) == b"UQ_ERR_ALIGN"
    assert L.uq_status_string(99) == b"UQ_ERR_UNKNOWN"


def test_packed_size(L):
    import gemm_uq_gb300 as uq
    assert uq.packed_size(4096, 4096, 128, "INT4_ASYM") == (4096 * 2048, 4096 * 32 * 2, 4096 * 16)
    assert uq.packed_size(8192, 8192, 64, "INT2_ASYM") == (8192 * 2048, 8192 * 128 * 2, 8192 * 128 * 2)
    assert uq.packed_size(8192, 8192, 128, "INT8_SYM") == (8192 * 8192, 8192 * 64 * 2, 0)
    assert uq.packed_size(8192, 8192, 64, "NF4") == (8192 * 4096, 8192 * 128 * 2, 64)
    assert uq.packed_size(1024, 8192, 256, "K4") == (1024 * 4096, 1024 * 32 * 16, 0)
    assert uq.packed_size(256, 256, 32, "INT4_SYM") == (256 * 128, 256 * 8 * 2, 0)


@pytest.mark.parametrize("N,K,group,fmt,status", [
    (16, 100, 32, 1, 1),      # K not a multiple of the group
    (16, 256, 48, 1, 2),      # unsupported group
    (16, 96, 32, 3, 2),       # INT2 needs K % 64
    (16, 512, 128, 5, 2),     # K4 needs group 256
    (16, 384, 256, 5, 1),     # K4 needs K % 256
    (-1, 256, 32, 0, 1),      # negative size
    (16, 256, 32, 9, 1),      # unknown format
])
def test_packed_size_rejects(L, N, K, group, fmt, status):
    a = ctypes.c_size_t()
    assert L.uq_packed_size(N, K, group, fmt, ctypes.byref(a), None, None) == status
    assert len(L.uq_last_error()) > 0


def test_gemm_host_validation_needs_no_gpu(L):
    # argument errors are caught on the host before any CUDA call
    P = ctypes.c_void_p
    buf = (ctypes.c_uint8 * 64)()
    base = ctypes.addressof(buf)
    al = P(base + (-base) % 16)
    assert L.uq_gemm(al, al, al, None, al, -1, 8, 256, 32, 0, None) == 1            # M < 0
    assert L.uq_gemm(al, al, al, None, al, 0, 8, 256, 32, 0, None) == 0             # M == 0: no-op
    assert L.uq_gemm(al, al, al, None, al, 4, 0, 256, 32, 0, None) == 0             # N == 0: no-op
    assert L.uq_gemm(None, al, al, None, al, 1, 8, 256, 32, 0, None) == 1           # x NULL
    assert L.uq_gemm(al, al, al, None, None, 1, 8, 256, 32, 0, None) == 1           # y NULL
    assert L.uq_gemm(al, al, al, al, al, 1, 8, 256, 32, 0, None) == 1               # zeros given for INT4_SYM
    assert L.uq_gemm(al, al, al, None, al, 1, 8, 256, 128, 1, None) == 1            # zeros missing for ASYM
    mis = P(al.value + 2)
    assert L.uq_gemm(mis, al, al, None, al, 1, 8, 256, 32, 0, None) == 3            # misaligned x
    assert L.uq_gemm(al, al, al, None, mis, 1, 8, 256, 32, 0, None) == 3            # misaligned y


def test_kernel_count_host_validation(L):
    # shape errors and empty calls are answered on the host, before any CUDA call
    n = ctypes.c_int(-1)
    assert L.uq_gemm_kernel_count(1, 8, 256, 48, 0, ctypes.byref(n)) == 2   # group 48
    assert L.uq_gemm_kernel_count(-1, 8, 256, 32, 0, ctypes.byref(n)) == 1  # M < 0
    assert L.uq_gemm_kernel_count(0, 8, 256, 32, 0, ctypes.byref(n)) == 0 and n.value == 0
    assert L.uq_gemm_kernel_count(1, 8, 256, 32, 0, None) == 1              # no output pointer
