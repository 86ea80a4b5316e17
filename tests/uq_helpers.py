"""Test helpers: move oracle-quantized weights to the device in the uq_gemm caller layout."""
from __future__ import annotations

import numpy as np
import torch

import gemm_uq_gb300 as uq
from oracle import quant as oquant

KT = {"INT4_SYM": 1024, "INT4_ASYM": 1024, "INT8_SYM": 512, "INT2_ASYM": 2048, "NF4": 1024, "K4": 1024}


def h16(a: np.ndarray, dev) -> torch.Tensor:
    """fp16 numpy array -> int16 device tensor holding the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16).view(np.int16)).to(dev)


def device_weights(qz: "oquant.Quantized", dev):
    """(wq, scales, zc) device tensors for uq_gemm from an oracle Quantized."""
    codes = torch.from_numpy(np.ascontiguousarray(qz.codes)).to(dev)
    wq = uq.pack_layout(codes, qz.group, qz.fmt)
    zc = None
    if qz.fmt == "K4":
        scales = uq.pack_kmeta(h16(qz.d, dev), h16(qz.dmin, dev),
                               torch.from_numpy(np.ascontiguousarray(qz.sc)).to(dev),
                               torch.from_numpy(np.ascontiguousarray(qz.m)).to(dev))
    else:
        scales = h16(qz.scale, dev)
        if qz.fmt == "INT4_ASYM":
            zc = torch.from_numpy(oquant.pack_zero_nibbles(qz.zero)).to(dev)
        elif qz.fmt == "INT2_ASYM":
            zc = h16(qz.zero, dev)
        elif qz.fmt == "NF4":
            zc = torch.from_numpy(np.ascontiguousarray(qz.codebook, dtype=np.float32)).to(dev)
    return wq, scales, zc


def device_x(x: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev).to(torch.bfloat16)


def y_to_f64(y: torch.Tensor) -> np.ndarray:
    return y.float().cpu().numpy().astype(np.float64)


def mma_gemm_launches(fmt, N, K, sms):
    """Launches of one block of 9..64 rows on the mma.sync GEMM, by the library's split rule: the k
    units of a row group (128 rows) are split over the fewest CTAs that minimise the units of the
    busiest SM; a split adds the second pass, K4 its x column-sum pre-kernel."""
    kc = 128 if fmt == "INT2_ASYM" else 64
    kp = -(-K // kc) * kc
    ub = -(-kp // (4 * kc))
    rg = -(-(-(-N // 16)) // 8)
    best, best_load = 1, None
    for ks in range(1, min(ub, 64) + 1):
        load = -(-(rg * ks) // sms) * -(-ub // ks)
        if best_load is None or load < best_load:
            best, best_load = ks, load
    return 1 + (1 if best > 1 else 0) + (1 if fmt == "K4" else 0)
