"""Seeded synthetic inputs shared by the oracle-side tests and the GPU-side tests/bench.

This module holds NO arithmetic of the quantization method: it only draws random
numbers (NumPy PCG64 through ``numpy.random.default_rng``), rounds activations to
bf16 (input preparation: the activations of the decode path are bf16), and
describes the workloads by their shapes.  Both the CPU oracle and the CUDA path
receive exactly the arrays produced here.

Workloads follow the decode-step linears that the "Ultra LLM Engine" page names
(section "Fused Kernels": dequantized weight GEMV for single-token decode and
dequantized weight GEMM for batched decode; section "Quantization": group-wise
INT-N and NF4).  The concrete shapes are those of an 8B-class and a 70B-class
decoder (hidden 4096 / 8192, intermediate 14336 / 28672, GQA k/v width 1024).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "bf16_round",
    "bf16_bits",
    "bf16_from_bits",
    "normal_weights",
    "activations",
    "Linear",
    "Workload",
    "WORKLOADS",
    "seed_for",
    "gguf_blocks",
]


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32 holding bf16 values.

    NaN/Inf are not expected in synthetic inputs and are not handled specially.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of bf16-representable float32 values (asserts representability)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value is not bf16-representable"
    return (u >> 16).astype(np.uint16)


def bf16_from_bits(b: np.ndarray) -> np.ndarray:
    """float32 values of uint16 bf16 bit patterns."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_weights(seed: int, n: int, k: int, sigma: float,
                   outlier_p: float = 0.0, outlier_mult: float = 1.0) -> np.ndarray:
    """W (n x k, float32) ~ N(0, sigma^2); with probability ``outlier_p`` an element is multiplied by ``outlier_mult``.

    Two independent PCG64 streams: [seed, 0] for the normals, [seed, 2] for the outlier mask.
    """
    rng = np.random.default_rng([seed, 0])
    w = rng.standard_normal((n, k), dtype=np.float32) * np.float32(sigma)
    if outlier_p > 0.0:
        mask = np.random.default_rng([seed, 2]).random((n, k)) < outlier_p
        w[mask] *= np.float32(outlier_mult)
    return w


def activations(seed: int, m: int, k: int) -> np.ndarray:
    """x (m x k) ~ N(0, 1) drawn in float32 from stream [seed, 1], rounded to bf16 (float32 array of bf16 values)."""
    rng = np.random.default_rng([seed, 1])
    return bf16_round(rng.standard_normal((m, k), dtype=np.float32))


def gguf_blocks(seed: int, n: int, k: int, qtype: str, sigma: float = 0.01) -> np.ndarray:
    """Random GGUF blocks (uint8 [n][k/32][block bytes]) of type "Q4_0" (18 bytes) or "Q8_0" (34 bytes):
    uniform random code bytes and an fp16 d ~ N(0, sigma) in the first two bytes (little endian).
    Every such byte pattern is a valid block; nothing here quantizes anything."""
    nbytes = {"Q4_0": 18, "Q8_0": 34}[qtype]
    rng = np.random.default_rng([seed, 3])
    raw = rng.integers(0, 256, (n, k // 32, nbytes)).astype(np.uint8)
    d = (rng.normal(0.0, sigma, (n, k // 32)).astype(np.float16)).view(np.uint16)
    raw[..., 0] = (d & 0xFF).astype(np.uint8)
    raw[..., 1] = (d >> 8).astype(np.uint8)
    return raw


def seed_for(workload: int, index: int) -> int:
    """Seed of linear ``index`` of workload ``workload``: the tiny INT4 case uses seed 0, others 1000*w + index."""
    return 0 if workload == 1 else 1000 * workload + index


@dataclass(frozen=True)
class Linear:
    name: str
    n: int          # output features (rows of W)
    k: int          # input features (columns of W)


@dataclass(frozen=True)
class Workload:
    """A named set of decode linears in one weight format, run at the listed batch sizes M."""
    key: int
    title: str
    fmt: str
    group: int
    sigma: float
    linears: tuple
    ms: tuple
    outlier_p: float = 0.0
    outlier_mult: float = 1.0
    layers: int = 1
    extra: dict = field(default_factory=dict)


_L3_8B = (Linear("q", 4096, 4096), Linear("k", 1024, 4096), Linear("v", 1024, 4096),
          Linear("o", 4096, 4096), Linear("gate", 14336, 4096), Linear("up", 14336, 4096),
          Linear("down", 4096, 14336))
_L3_70B = (Linear("q", 8192, 8192), Linear("k", 1024, 8192), Linear("v", 1024, 8192),
           Linear("o", 8192, 8192), Linear("gate", 28672, 8192), Linear("up", 28672, 8192),
           Linear("down", 8192, 28672))

WORKLOADS = {
    1: Workload(1, "tiny INT4 GEMV 256x256", "INT4_SYM", 32, 0.02,
                (Linear("w", 256, 256),), (1,)),
    2: Workload(2, "8B-shaped decode linears, INT4 asym g128, M=1", "INT4_ASYM", 128, 0.02,
                _L3_8B, (1,), outlier_p=0.001, outlier_mult=20.0, layers=32),
    3: Workload(3, "batched decode sweep, INT4 asym g128", "INT4_ASYM", 128, 0.02,
                (Linear("gate", 14336, 4096), Linear("down", 4096, 14336)),
                (1, 2, 4, 8, 16, 32, 64)),
    4: Workload(4, "format sweep 8192x8192", "INT8_SYM|INT2_ASYM|NF4", 0, 0.02,
                (Linear("w", 8192, 8192),), (1, 16),
                extra={"formats": (("INT8_SYM", 128), ("INT2_ASYM", 64), ("NF4", 64))}),
    5: Workload(5, "70B-shaped decode linear stack, two-level INT4", "K4", 256, 0.015,
                _L3_70B, (1, 8, 32), layers=8),
}
