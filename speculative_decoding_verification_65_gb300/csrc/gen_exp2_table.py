"""Write exp2_table.h: 2^(i/256) for i = 0..255 as pairs of floats.

Each value is computed with Python's decimal module at 60 significant digits,
then split into hi = the nearest float and lo = the nearest float to the
remainder, so hi + lo carries about 48 bits.  The exact-draw kernels use the
table for 2^x to about 1e-13 relative error.  Run from anywhere:
    python gen_exp2_table.py
"""
from __future__ import annotations

import decimal
import os
import struct

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "exp2_table.h")


def f32(x: decimal.Decimal) -> float:
    """x rounded to float64, then to float32 (the check in main() confirms
    that the two roundings gave the float32 nearest to x)."""
    return struct.unpack("<f", struct.pack("<f", float(x)))[0]


def main() -> None:
    decimal.getcontext().prec = 60
    two = decimal.Decimal(2)
    ln2 = two.ln()
    rows = []
    for i in range(256):
        v = (ln2 * decimal.Decimal(i) / 256).exp()
        hi = f32(v)
        lo = f32(v - decimal.Decimal(hi))
        # hi must be the float nearest v (no double-rounding tie in the
        # float64 step): |v - hi| <= half an ulp of hi
        ulp = decimal.Decimal(2) ** (-23)  # hi is in [1, 2)
        assert abs(v - decimal.Decimal(hi)) <= ulp / 2, i
        assert abs(v - decimal.Decimal(hi) - decimal.Decimal(lo)) < decimal.Decimal(2) ** -47, i
        rows.append((hi, lo))
    with open(OUT, "w") as f:
        f.write("// exp2_table.h -- written by gen_exp2_table.py; do not edit.\n")
        f.write("// Entry i holds 2^(i/256) as hi + lo (hi the nearest float, lo the\n")
        f.write("// nearest float to the remainder).\n")
        f.write("#pragma once\n\n")
        f.write("// Device code only (included by resolve.cuh).\n")
        f.write("static __device__ const float kExp2Tab[256][2] = {\n")
        for i, (hi, lo) in enumerate(rows):
            f.write(f"    {{{hi.hex()}f, {lo.hex()}f}},  // {i}\n")
        f.write("};\n")


if __name__ == "__main__":
    main()
