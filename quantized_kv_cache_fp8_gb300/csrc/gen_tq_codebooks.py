"""Write kvq_tq_codebooks.cuh: the N(0,1) Lloyd-Max codebooks of the rotated tiers at
3 and 6 bits (8 and 64 levels) as binary16 bit patterns.

The quantizer is the fixed point of two conditions (colibri PR #399, "Why rotated-int4
for the 4-bit tier": a fixed N(0,1)-optimal Lloyd-Max codebook): every threshold is the
midpoint of its two neighbouring outputs, and every output is the mean of N(0,1) over
its cell.  It is solved here by Newton's method on T(c) - c = 0, where T maps outputs to
cell means; T_k depends on c_{k-1}, c_k, c_{k+1} only, so each step is a banded solve.
Cell masses are taken from the tail that keeps them accurate.  Each output is then
rounded to the nearest binary16 value.

Run: python gen_tq_codebooks.py   (rewrites kvq_tq_codebooks.cuh next to this file)
"""
import os

import numpy as np
from scipy.linalg import solve_banded
from scipy.special import erfc

SQRT1_2 = 0.7071067811865476


def _pdf(t):
    return np.where(np.isinf(t), 0.0, np.exp(-0.5 * np.square(np.where(np.isinf(t), 0.0, t)))) \
        / np.sqrt(2.0 * np.pi)


def _mass(a, b):
    """P(a < X < b) for X ~ N(0,1), from the upper tail above 0 and the lower tail below."""
    up = 0.5 * (erfc(a * SQRT1_2) - erfc(b * SQRT1_2))
    lo = 0.5 * (erfc(-b * SQRT1_2) - erfc(-a * SQRT1_2))
    mid = 1.0 - 0.5 * erfc(b * SQRT1_2) - 0.5 * erfc(-a * SQRT1_2)
    return np.where(a >= 0, up, np.where(b <= 0, lo, mid))


def lloyd_max(levels: int, steps: int = 200) -> np.ndarray:
    # start from the cell means of an equal-probability partition (near the fixed point)
    c = np.sqrt(2.0) * np.array([_probit((k + 0.5) / levels) for k in range(levels)])
    for _ in range(steps):
        t = np.concatenate([[-np.inf], 0.5 * (c[1:] + c[:-1]), [np.inf]])
        pa, pb = _pdf(t[:-1]), _pdf(t[1:])
        m = _mass(t[:-1], t[1:])
        T = (pa - pb) / m
        dA = np.where(np.isinf(t[:-1]), 0.0, pa * (T - np.where(np.isinf(t[:-1]), 0.0, t[:-1])) / m)
        dB = np.where(np.isinf(t[1:]), 0.0, pb * (np.where(np.isinf(t[1:]), 0.0, t[1:]) - T) / m)
        # Jacobian of T - c: row k has 0.5 dA_k (col k-1), 0.5 (dA_k + dB_k) - 1, 0.5 dB_k
        ab = np.zeros((3, levels))
        ab[0, 1:] = 0.5 * dB[:-1]
        ab[1, :] = 0.5 * (dA + dB) - 1.0
        ab[2, :-1] = 0.5 * dA[1:]
        delta = solve_banded((1, 1), ab, -(T - c))
        c = c + delta
        if np.max(np.abs(delta)) < 1e-16:
            break
    return c


def _probit(p: float) -> float:
    """erf^-1(2p - 1) by bisection on erfc (p in (0, 1))."""
    lo, hi = -10.0, 10.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if 0.5 * erfc(-mid) < p:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def main():
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "kvq_tq_codebooks.cuh")
    lines = ["// kvq_tq_codebooks.cuh — written by gen_tq_codebooks.py; do not edit.",
             "// N(0,1) Lloyd-Max outputs of the rotated tiers at 3 and 6 bits, each rounded to",
             "// the nearest binary16 value, ascending (bit patterns).",
             "#pragma once", "", "#include <cstdint>", "", "namespace kvq {", ""]
    for bits in (3, 6):
        c = lloyd_max(1 << bits)
        h = c.astype(np.float16).view(np.uint16)
        assert np.all(np.diff(c) > 0) and np.allclose(c, -c[::-1], atol=1e-13)
        lines.append(f"constexpr uint16_t kTq{bits}CentroidBits[{1 << bits}] = {{")
        for i in range(0, len(h), 8):
            lines.append("    " + ", ".join(f"0x{int(v):04X}" for v in h[i:i + 8]) + ",")
        lines.append("};")
        lines.append("")
    lines += ["}  // namespace kvq", ""]
    open(out, "w").write("\n".join(lines))
    print(out)


if __name__ == "__main__":
    main()
