"""Writes the stored inputs under tests/golden/ that are computed (not hand-worked): calls only oracle/.

    python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle.nf4 import nf4_codebook  # noqa: E402


def main():
    c = nf4_codebook()
    with open(os.path.join(HERE, "nf4_codebook.txt"), "w") as f:
        f.write("# NF4 codebook (float32, ascending), written by tests/golden/make_golden.py from oracle.nf4\n")
        for v in c:
            f.write(f"{float(v):.9g}\n")


if __name__ == "__main__":
    main()
