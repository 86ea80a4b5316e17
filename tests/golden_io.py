"""Reader for the text fixtures under tests/golden/ (hand-worked values)."""
from __future__ import annotations

import os
from fractions import Fraction

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _expand(tokens):
    out = []
    for t in tokens:
        if "*" in t:
            v, n = t.rsplit("*", 1)
            out.extend([Fraction(v)] * int(n))
        else:
            out.append(Fraction(t))
    return out


def read_blocks(name: str) -> dict:
    """{section: {key: [Fraction, ...]}} from an INI-like fixture with 'v*n' repetition."""
    blocks, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("[") and line.endswith("]"):
                cur = blocks.setdefault(line[1:-1], {})
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            cur[key] = _expand(val.split())
    return blocks
