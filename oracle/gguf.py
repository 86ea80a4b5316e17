"""Decoding of GGUF-style block-quantized weights (Q4_0, Q8_0) to W_hat, in float64.

Source: "Ultra LLM Engine", section "Checkpoint Loading" (GGUF k-quant and block formats such as Q4_0 are
detected there but not dequantized) and the "lollm" page, section on shared infrastructure (GGUF parse +
dequant of the block formats).  The block layouts are the GGUF file format's own:

  Q4_0  32 weights per block, 18 bytes: fp16 d (little endian), then 16 bytes qs; weight j (j < 16) is
        the low nibble of qs[j], weight j + 16 its high nibble; w = d * (nibble - 8).
  Q8_0  32 weights per block, 34 bytes: fp16 d, then 32 signed bytes q; w = d * q.

A weight row of K values (K a multiple of 32) is K / 32 consecutive blocks; rows follow each other.
W_hat is d * q, exact in float32 (11-bit d times a small integer), returned as float32.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).
"""
from __future__ import annotations

import numpy as np

BLOCK = 32
BLOCK_BYTES = {"Q4_0": 18, "Q8_0": 34}


def split_blocks(raw: np.ndarray, qtype: str, n: int, k: int):
    """(d fp16 [n][k/32], codes int8 [n][k]) of raw GGUF block bytes (uint8 [n][k/32][block bytes])."""
    assert k % BLOCK == 0
    nb = k // BLOCK
    b = np.asarray(raw, dtype=np.uint8).reshape(n, nb, BLOCK_BYTES[qtype])
    d = b[..., 0:2].copy().view("<f2").reshape(n, nb)
    if qtype == "Q4_0":
        qs = b[..., 2:18].astype(np.int16)
        lo = (qs & 0x0F) - 8                                 # weights 0 .. 15 of the block
        hi = (qs >> 4) - 8                                   # weights 16 .. 31
        codes = np.concatenate([lo, hi], axis=-1)
    elif qtype == "Q8_0":
        codes = b[..., 2:34].copy().view(np.int8).astype(np.int16)
    else:
        raise ValueError(qtype)
    return d.astype(np.float16), codes.reshape(n, k).astype(np.int8)


def dequant(raw: np.ndarray, qtype: str, n: int, k: int) -> np.ndarray:
    """W_hat (float32 [n][k]) = d * q of every block (exact)."""
    d, codes = split_blocks(raw, qtype, n, k)
    w = d.astype(np.float64).repeat(BLOCK, axis=1) * codes.astype(np.float64)
    return w.astype(np.float32)
