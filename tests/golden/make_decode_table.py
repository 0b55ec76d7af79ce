"""Writes decode_table.txt from the oracle alone: the SHA-256 of the fp16
weights of all 65536 16-bit states (little-endian uint16, state order), a
few sample states, the number of states whose fp32 half-sum is an exact
fp16 tie, and summary statistics. Run from the repository root:

    python tests/golden/make_decode_table.py
"""
import hashlib
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402

SAMPLES = (0x0000, 0x0001, 0x0002, 0x1234, 0x8000, 0xFFFF)


def table_facts():
    t = oracle.decode_table()
    f = t.view(np.float16).astype(np.float64)
    ties = 0
    for s in range(65536):
        u = oracle.lcg_masked(s)
        exact = oracle.half_to_float(u & 0xFFFF) + oracle.half_to_float(u >> 16)
        below = float(np.float16(exact))
        # an exact tie sits halfway between two adjacent fp16 values
        lo = np.float16(exact)
        nxt = np.nextafter(lo, np.float16(np.inf if exact > float(lo) else -np.inf))
        if exact != below and abs(exact - float(lo)) == abs(float(nxt) - exact):
            ties += 1
    return {
        "sha256": hashlib.sha256(t.astype("<u2").tobytes()).hexdigest(),
        "samples": {s: int(t[s]) for s in SAMPLES},
        "ties": ties,
        "sum": float(f.sum()),
        "min": float(f.min()),
        "max": float(f.max()),
    }


def main():
    d = table_facts()
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "decode_table.txt")
    with open(out, "w") as fh:
        fh.write("# fp16 weights of all 65536 trellis states, written by make_decode_table.py from the oracle\n")
        fh.write(f"sha256 {d['sha256']}\n")
        for s, v in d["samples"].items():
            fh.write(f"state 0x{s:04X} 0x{v:04X}\n")
        fh.write(f"ties {d['ties']}\n")
        fh.write(f"sum {d['sum']!r}\nmin {d['min']!r}\nmax {d['max']!r}\n")
    print(open(out).read())


if __name__ == "__main__":
    main()
