"""Pins of the GGUF block decoder (oracle/gguf.py): hand-built blocks with known bytes, the agreement of
Q4_0 / Q8_0 with the INT4_SYM / INT8_SYM group-32 definitions, and planted layout mistakes."""
import numpy as np

from oracle import gguf, quant


def _q4_block(d_bits, qs):
    return np.array([d_bits & 0xFF, d_bits >> 8] + list(qs), dtype=np.uint8)


def test_q4_0_hand_built_block():
    # d = 0.5 (fp16 0x3800); byte j holds weight j (low nibble) and weight j + 16 (high nibble)
    qs = [(j & 0xF) | ((15 - j) << 4) for j in range(16)]
    w = gguf.dequant(_q4_block(0x3800, qs), "Q4_0", 1, 32)[0]
    want = [0.5 * (j - 8) for j in range(16)] + [0.5 * ((15 - j) - 8) for j in range(16)]
    assert w.tolist() == want
    # planted: nibbles taken as consecutive weights (2j, 2j + 1) give a different row
    inter = [0.5 * ((qs[j // 2] >> (4 * (j % 2))) & 0xF) - 4.0 for j in range(32)]
    assert inter != want


def test_q8_0_hand_built_block_and_byte_order():
    q = list(range(-128, -112)) + list(range(112, 128))
    raw = np.array([0x00, 0xB4] + [v & 0xFF for v in q], dtype=np.uint8)     # d = -0.25
    w = gguf.dequant(raw, "Q8_0", 1, 32)[0]
    assert w.tolist() == [-0.25 * v for v in q]
    one = np.array([0x00, 0x3C] + [1] * 32, dtype=np.uint8)                   # little-endian d = 1.0
    assert gguf.dequant(one, "Q8_0", 1, 32)[0].tolist() == [1.0] * 32


def test_q4_0_and_q8_0_agree_with_the_symmetric_group_32_formats():
    rng = np.random.default_rng(11)
    n, k = 5, 256
    for qtype, fmt in (("Q4_0", "INT4_SYM"), ("Q8_0", "INT8_SYM")):
        nbytes = gguf.BLOCK_BYTES[qtype]
        raw = rng.integers(0, 256, (n, k // 32, nbytes)).astype(np.uint8)
        d = (rng.normal(0, 0.01, (n, k // 32)).astype(np.float16)).view(np.uint16)
        raw[..., 0] = d & 0xFF
        raw[..., 1] = d >> 8
        dd, codes = gguf.split_blocks(raw, qtype, n, k)
        qz = quant.Quantized(fmt, 32, codes, scale=dd)
        assert np.array_equal(quant.dequant(qz).view(np.uint32), gguf.dequant(raw, qtype, n, k).view(np.uint32))
        lo, hi = (-8, 7) if qtype == "Q4_0" else (-128, 127)
        assert codes.min() >= lo and codes.max() <= hi
