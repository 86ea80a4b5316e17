"""Python binding of the uq C-ABI library (include/uq.h): argument marshalling only.

Every function here forwards torch tensors' device pointers, sizes and the current CUDA
stream to the same-named ``extern "C"`` entry point of ``libuq.so`` and raises
``UqError`` on a non-OK status.  No step of the computation runs in Python or in
PyTorch: if the library is missing, importing the ops raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libuq.so")

FORMATS = {"INT4_SYM": 0, "INT4_ASYM": 1, "INT8_SYM": 2, "INT2_ASYM": 3, "NF4": 4, "K4": 5}
BITS = {"INT4_SYM": 4, "INT4_ASYM": 4, "INT8_SYM": 8, "INT2_ASYM": 2, "NF4": 4, "K4": 4}

# every entry point declared in include/uq.h: name -> (restype, argtypes)
_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)
SIGNATURES = {
    "uq_status_string": (ctypes.c_char_p, [_I]),
    "uq_last_error": (ctypes.c_char_p, []),
    "uq_packed_size": (_I, [_I, _I, _I, _I, _SZ, _SZ, _SZ]),
    "uq_pack_layout": (_I, [_P, _P, _I, _I, _I, _I, _P]),
    "uq_pack_kmeta": (_I, [_P, _P, _P, _P, _P, _I, _I, _P]),
    "uq_gemm": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "uq_unpack_codes": (_I, [_P, _P, _I, _I, _I, _I, _P]),
    "uq_dequant": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "uq_quantize": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "uq_quantize_k4": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _P]),
    "uq_pack_zeros": (_I, [_P, _P, _I, _I, _P]),
    "uq_device_fault": (_I, [ctypes.POINTER(ctypes.c_uint)]),
    "uq_gemm_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "uq_gemm_noalloc_scratch": (_I, [_I, _I, _I, _I, _I, _SZ, _SZ]),
    "uq_set_launch_overlap": (_I, [_I]),
    "uq_set_gemm_path": (_I, [_I]),
    "uq_gemm_kernel_count": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_I)]),
    "uq_gemm_gated": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "uq_gemm_gated_kernel_count": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_I)]),
    "uq_pack_gguf": (_I, [_P, _I, _P, _P, _I, _I, _P]),
    "uq_gemm_w4a8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "uq_gemm_w4a8_kernel_count": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_I)]),
    "uq_rope_table": (_I, [_P, _I, _I, ctypes.c_double, _P]),
    "uq_rmsnorm_rope": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_float, _P]),
}

_lib = None


class UqError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: status {status} ({msg})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded libuq.so (raises if it has not been built: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with `python -m gemm_uq_gb300.build` "
                              "(the quantized GEMV has no non-CUDA implementation)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != 0:
        L = lib()
        raise UqError(status, where, f"{L.uq_status_string(status).decode()}: {L.uq_last_error().decode()}")


def _ptr(t):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "tensors passed to uq must be contiguous CUDA tensors"
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def packed_size(N: int, K: int, group: int, fmt: str):
    """(wq_bytes, scales_bytes, zeros_bytes) -- host only."""
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().uq_packed_size(N, K, group, FORMATS[fmt], ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
           "uq_packed_size")
    return a.value, b.value, c.value


def pack_layout(codes: torch.Tensor, group: int, fmt: str, stream=None) -> torch.Tensor:
    """int8 codes [N][K] (device) -> packed uint8 plane (synchronizes the stream)."""
    N, K = codes.shape
    wq_bytes, _, _ = packed_size(N, K, group, fmt)
    wq = torch.empty(max(wq_bytes, 16), dtype=torch.uint8, device=codes.device)
    _check(lib().uq_pack_layout(_ptr(codes), _ptr(wq), N, K, group, FORMATS[fmt], _stream(stream)),
           "uq_pack_layout")
    return wq


GGUF_TYPES = {"Q4_0": (0, "INT4_SYM"), "Q8_0": (1, "INT8_SYM")}


def pack_gguf(blocks: torch.Tensor, qtype: str, N: int, K: int, stream=None):
    """uq_pack_gguf: GGUF Q4_0 / Q8_0 block bytes (device uint8) -> (wq, scales) of INT4_SYM / INT8_SYM, group 32."""
    t, fmt = GGUF_TYPES[qtype]
    wq_bytes, sc_bytes, _ = packed_size(N, K, 32, fmt)
    wq = torch.empty(max(wq_bytes, 16), dtype=torch.uint8, device=blocks.device)
    scales = torch.empty((N, K // 32), dtype=torch.int16, device=blocks.device)
    assert blocks.is_cuda and blocks.is_contiguous()
    _check(lib().uq_pack_gguf(ctypes.c_void_p(blocks.data_ptr()), t, _ptr(wq), _ptr(scales), N, K, _stream(stream)),
           "uq_pack_gguf")
    return wq, scales


def pack_kmeta(d, dmin, sc, m, stream=None) -> torch.Tensor:
    """K4 fp16 d, dmin [N][S] (as int16/uint16/float16 tensors), uint8 sc, m [N][S][8] -> records [N][S][16]."""
    N, S = d.shape
    meta = torch.empty((N, S, 16), dtype=torch.uint8, device=d.device)
    _check(lib().uq_pack_kmeta(_ptr(d), _ptr(dmin), _ptr(sc), _ptr(m), _ptr(meta), N, S * 256, _stream(stream)),
           "uq_pack_kmeta")
    return meta


def pack_zeros(z: torch.Tensor, stream=None) -> torch.Tensor:
    """INT4_ASYM zeros, one per byte [N][G] -> two per byte [N][ceil(G/2)]."""
    N, G = z.shape
    out = torch.empty((N, (G + 1) // 2), dtype=torch.uint8, device=z.device)
    _check(lib().uq_pack_zeros(_ptr(z), _ptr(out), N, G, _stream(stream)), "uq_pack_zeros")
    return out


def gemm(x: torch.Tensor, wq: torch.Tensor, scales: torch.Tensor, zc, N: int, group: int, fmt: str,
         y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = x . W_hat^T (bf16 [M][N]) with W_hat dequantized on the fly."""
    M, K = x.shape
    assert x.dtype == torch.bfloat16
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(lib().uq_gemm(_ptr(x), _ptr(wq), _ptr(scales), _ptr(zc), _ptr(y), M, N, K, group, FORMATS[fmt],
                         _stream(stream)), "uq_gemm")
    return y


def gemm_gated(x: torch.Tensor, gate: tuple, up: tuple, N: int, group: int, fmt: str,
               h: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """h = silu(x . W_gate_hat^T) * (x . W_up_hat^T) (bf16 [M][N]); gate and up are (wq, scales, zc)."""
    M, K = x.shape
    assert x.dtype == torch.bfloat16
    if h is None:
        h = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    (wg, sg, zg), (wu, su, zu) = gate, up
    _check(lib().uq_gemm_gated(_ptr(x), _ptr(wg), _ptr(sg), _ptr(zg), _ptr(wu), _ptr(su), _ptr(zu), _ptr(h),
                               M, N, K, group, FORMATS[fmt], _stream(stream)), "uq_gemm_gated")
    return h


def gemm_gated_ptrs(x_ptr: int, gate: tuple, up: tuple, h_ptr: int, M: int, N: int, K: int, group: int, fmt: str,
                    stream_handle: int) -> None:
    """Raw-pointer form of uq_gemm_gated; gate and up are (wq_ptr, scales_ptr, zc_ptr or 0)."""
    P = ctypes.c_void_p
    _check(lib().uq_gemm_gated(P(x_ptr), P(gate[0]), P(gate[1]), P(gate[2]) if gate[2] else None, P(up[0]),
                               P(up[1]), P(up[2]) if up[2] else None, P(h_ptr), M, N, K, group, FORMATS[fmt],
                               P(stream_handle)), "uq_gemm_gated")


def gemm_gated_kernel_count(M: int, N: int, K: int, group: int, fmt: str) -> int:
    v = ctypes.c_int(0)
    _check(lib().uq_gemm_gated_kernel_count(M, N, K, group, FORMATS[fmt], ctypes.byref(v)),
           "uq_gemm_gated_kernel_count")
    return v.value


def rope_table(max_pos: int, head_dim: int, base: float, device=None, stream=None) -> torch.Tensor:
    """uq_rope_table: fp32 [max_pos][head_dim/2][2] (cos, sin) on the device."""
    t = torch.empty((max_pos, head_dim // 2, 2), dtype=torch.float32, device=device or "cuda")
    _check(lib().uq_rope_table(_ptr(t), max_pos, head_dim, float(base), _stream(stream)), "uq_rope_table")
    return t


def rmsnorm_rope(x: torch.Tensor, gamma: torch.Tensor, pos: torch.Tensor, table: torch.Tensor, head_dim: int,
                 eps: float, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """uq_rmsnorm_rope: y = RoPE(RMSNorm(x) * gamma, pos) (bf16 [M][D]); y may be x."""
    M, D = x.shape
    assert x.dtype == torch.bfloat16 and gamma.dtype == torch.bfloat16 and pos.dtype == torch.int32
    if y is None:
        y = torch.empty_like(x)
    _check(lib().uq_rmsnorm_rope(_ptr(x), _ptr(gamma), _ptr(pos), _ptr(table), _ptr(y), M, D, head_dim,
                                 table.shape[0], float(eps), _stream(stream)), "uq_rmsnorm_rope")
    return y


def gemm_w4a8(x: torch.Tensor, wq: torch.Tensor, scales: torch.Tensor, zc, N: int, group: int, fmt: str,
              y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """uq_gemm_w4a8: y with x quantized per row to int8 and integer dot products (bf16 [M][N])."""
    M, K = x.shape
    assert x.dtype == torch.bfloat16
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(lib().uq_gemm_w4a8(_ptr(x), _ptr(wq), _ptr(scales), _ptr(zc), _ptr(y), M, N, K, group, FORMATS[fmt],
                              _stream(stream)), "uq_gemm_w4a8")
    return y


def gemm_w4a8_ptrs(x_ptr: int, wq_ptr: int, scales_ptr: int, zc_ptr, y_ptr: int, M: int, N: int, K: int, group: int,
                   fmt: str, stream_handle: int) -> None:
    P = ctypes.c_void_p
    _check(lib().uq_gemm_w4a8(P(x_ptr), P(wq_ptr), P(scales_ptr), P(zc_ptr) if zc_ptr else None, P(y_ptr), M, N, K,
                              group, FORMATS[fmt], P(stream_handle)), "uq_gemm_w4a8")


def gemm_w4a8_kernel_count(M: int, N: int, K: int, group: int, fmt: str) -> int:
    v = ctypes.c_int(0)
    _check(lib().uq_gemm_w4a8_kernel_count(M, N, K, group, FORMATS[fmt], ctypes.byref(v)), "uq_gemm_w4a8_kernel_count")
    return v.value


def gemm_noalloc(x: torch.Tensor, wq: torch.Tensor, scales: torch.Tensor, zc, N: int, group: int, fmt: str,
                 y: torch.Tensor, stream=None) -> torch.Tensor:
    """uq_gemm_noalloc: the GEMV with the library's static scratch (y must be given: nothing is allocated)."""
    M, K = x.shape
    _check(lib().uq_gemm_noalloc(_ptr(x), _ptr(wq), _ptr(scales), _ptr(zc), _ptr(y), M, N, K, group, FORMATS[fmt],
                                 _stream(stream)), "uq_gemm_noalloc")
    return y


def gemm_noalloc_scratch(M: int, N: int, K: int, group: int, fmt: str):
    """uq_gemm_noalloc_scratch: (ticket_bytes, partial_bytes) of the static scratch the call would use
    (host only; 0, 0 when every worker owns whole row blocks)."""
    t, p = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().uq_gemm_noalloc_scratch(M, N, K, group, FORMATS[fmt], ctypes.byref(t), ctypes.byref(p)),
           "uq_gemm_noalloc_scratch")
    return t.value, p.value


def gemm_ptrs(x_ptr: int, wq_ptr: int, scales_ptr: int, zc_ptr, y_ptr: int, M: int, N: int, K: int, group: int,
              fmt: str, stream_handle: int) -> None:
    """Raw-pointer form of uq_gemm (for graph capture loops that pre-compute pointers)."""
    _check(lib().uq_gemm(ctypes.c_void_p(x_ptr), ctypes.c_void_p(wq_ptr), ctypes.c_void_p(scales_ptr),
                         ctypes.c_void_p(zc_ptr) if zc_ptr else None, ctypes.c_void_p(y_ptr), M, N, K, group,
                         FORMATS[fmt], ctypes.c_void_p(stream_handle)), "uq_gemm")


def unpack_codes(wq: torch.Tensor, N: int, K: int, group: int, fmt: str, stream=None) -> torch.Tensor:
    codes = torch.empty((N, K), dtype=torch.int8, device=wq.device)
    _check(lib().uq_unpack_codes(_ptr(wq), _ptr(codes), N, K, group, FORMATS[fmt], _stream(stream)),
           "uq_unpack_codes")
    return codes


def dequant(wq: torch.Tensor, scales: torch.Tensor, zc, N: int, K: int, group: int, fmt: str,
            stream=None) -> torch.Tensor:
    w = torch.empty((N, K), dtype=torch.float32, device=wq.device)
    _check(lib().uq_dequant(_ptr(wq), _ptr(scales), _ptr(zc), _ptr(w), N, K, group, FORMATS[fmt],
                            _stream(stream)), "uq_dequant")
    return w


def quantize(w: torch.Tensor, group: int, fmt: str, codebook: torch.Tensor | None = None, stream=None):
    """GPU quantizer for the flat formats: returns (codes int8 [N][K], scales fp16 bits [N][G], zeros)."""
    N, K = w.shape
    G = K // group if group else 0
    codes = torch.empty((N, K), dtype=torch.int8, device=w.device)
    scales = torch.empty((N, G), dtype=torch.int16, device=w.device)
    zeros = None
    if fmt == "INT4_ASYM":
        zeros = torch.empty((N, G), dtype=torch.uint8, device=w.device)
    elif fmt == "INT2_ASYM":
        zeros = torch.empty((N, G), dtype=torch.int16, device=w.device)
    _check(lib().uq_quantize(_ptr(w), _ptr(codes), _ptr(scales), _ptr(zeros), _ptr(codebook), N, K, group,
                             FORMATS[fmt], _stream(stream)), "uq_quantize")
    return codes, scales, zeros


def quantize_k4(w: torch.Tensor, stream=None):
    """GPU K4 quantizer: returns (codes, d, dmin, sc, m)."""
    N, K = w.shape
    S = K // 256
    dev = w.device
    codes = torch.empty((N, K), dtype=torch.int8, device=dev)
    d = torch.empty((N, S), dtype=torch.int16, device=dev)
    dmin = torch.empty((N, S), dtype=torch.int16, device=dev)
    sc = torch.empty((N, S, 8), dtype=torch.uint8, device=dev)
    m = torch.empty((N, S, 8), dtype=torch.uint8, device=dev)
    _check(lib().uq_quantize_k4(_ptr(w), _ptr(codes), _ptr(d), _ptr(dmin), _ptr(sc), _ptr(m), N, K,
                                _stream(stream)), "uq_quantize_k4")
    return codes, d, dmin, sc, m


def set_launch_overlap(enable: bool) -> None:
    """uq_set_launch_overlap: let GEMV launches prefetch their (constant) weights early."""
    _check(lib().uq_set_launch_overlap(1 if enable else 0), "uq_set_launch_overlap")


GEMM_PATHS = {"auto": 0, "tensor_cores": 1, "mma": 2}


def set_gemm_path(path: str) -> None:
    """uq_set_gemm_path: "auto" (default), "tensor_cores" (the tcgen05 kernel for every block of 16..64
    rows it supports) or "mma" (the mma.sync GEMM for every block of 9..64 rows of a 4-bit / 2-bit format)."""
    _check(lib().uq_set_gemm_path(GEMM_PATHS[path]), "uq_set_gemm_path")


def gemm_kernel_count(M: int, N: int, K: int, group: int, fmt: str) -> int:
    """uq_gemm_kernel_count: kernels one gemm() call of this shape launches on the current device."""
    v = ctypes.c_int(0)
    _check(lib().uq_gemm_kernel_count(M, N, K, group, FORMATS[fmt], ctypes.byref(v)), "uq_gemm_kernel_count")
    return v.value


def device_fault() -> int:
    v = ctypes.c_uint(0)
    _check(lib().uq_device_fault(ctypes.byref(v)), "uq_device_fault")
    return v.value
