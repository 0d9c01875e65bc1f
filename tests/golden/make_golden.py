"""Writes tests/golden/oracle_tables_sha256.txt: the sha256 of the oracle's
axis tables for every workload in synthetic.WORKLOADS, followed by its NeoX
cache of 131,072 x 256 rows (base 10000). Calls only oracle/ (and the shapes
in synthetic/). The fixture pins the tables across machines: the host C
library's pow, cos and sin feed them, and x86-64 and aarch64 must agree.

    python tests/golden/make_golden.py
"""
from __future__ import annotations

import hashlib
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synthetic  # noqa: E402


def tables_digest() -> str:
    h = hashlib.sha256()
    for _, w in sorted(synthetic.WORKLOADS.items()):
        for c, s in oracle.tables(w.T, w.H, w.W, w.split, w.base):
            h.update(c.tobytes())
            h.update(s.tobytes())
    h.update(oracle.neox_cache(131072, 256, 10000.0).tobytes())
    return h.hexdigest()


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_tables_sha256.txt"), "w") as f:
        f.write(tables_digest() + "\n")
