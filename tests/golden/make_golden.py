"""Write tests/golden/b1h1n256d64_rows.txt from the CPU oracle.

The fixture pins two things across machines and time: the seeded input
generator (a SHA-256 of the Q, K, V bytes it produces) and the oracle's output
on sampled rows of the tiny B=1, H=1, N=256, D=64 non-causal problem (seed 1001,
scale 1/8).  It calls only ``oracle`` and the input generator; nothing here
comes from the CUDA path.  Run from the repository root:

    python tests/golden/make_golden.py
"""
import hashlib
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from tiled_attention_forward_fa2_gb300.inputs import WORKLOADS  # noqa: E402

ROWS = [0, 1, 63, 64, 127, 128, 200, 255]
OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "b1h1n256d64_rows.txt")


def digest(q, k, v):
    h = hashlib.sha256()
    for a in (q, k, v):
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def main():
    w = WORKLOADS["b1h1n256d64"]
    q, k, v = w.qkv()
    o, lse = oracle.attn_rows(q, k, v, w.causal, w.scale, np.zeros(len(ROWS), np.int64), np.array(ROWS))
    with open(OUT, "w") as f:
        f.write("# oracle output on sampled rows of the b1h1n256d64 problem (seed 1001, scale 1/8, non-causal)\n")
        f.write("# written by tests/golden/make_golden.py, which calls only oracle/ and the input generator\n")
        f.write(f"sha256_qkv {digest(q, k, v)}\n")
        for r, orow, l in zip(ROWS, o, lse):
            f.write(f"row {r} lse {float(l)!r} o " + " ".join(repr(float(x)) for x in orow) + "\n")
    print("wrote", OUT)


if __name__ == "__main__":
    main()
