"""Fits the odd polynomials tanh(y) ~= y * P(y^2), |y| <= Y0, that the 16-bit
row kernels evaluate on the FMA pipe for the softcap transform, and writes
hl_tanh_poly.h.

Three fits are emitted:
  POLY  degree 6 on |y| <= 0.8   (resident kernel)
  A     degree 3 on |y| <= 0.45  (streaming kernel, narrow tier)
  B     degree 5 on |y| <= 0.8   (streaming kernel, wide tier)
Each P has P(0) = 1 and minimises the maximum relative error of P(u) against
tanh(sqrt(u)) / sqrt(u) on a dense grid (iteratively reweighted least
squares).  Run this file to regenerate the header.
"""
import os

import numpy as np

FITS = (("POLY", 0.8, 6), ("A", 0.45, 3), ("B", 0.8, 5))


def fit(y0, deg, iters=60):
    u = np.linspace(0.0, y0 * y0, 20001)
    y = np.sqrt(u)
    f = np.where(u > 0, np.tanh(y) / np.where(y > 0, y, 1.0), 1.0)
    A = np.vander(u, deg + 1, increasing=True)
    w = np.ones_like(u)
    for _ in range(iters):
        c, *_ = np.linalg.lstsq(A * w[:, None], f * w, rcond=None)
        err = (A @ c - f) / f
        w = w * (1 + 10 * np.abs(err) / np.abs(err).max())
        w /= w.mean()
    return c, float(np.abs(err).max())


def main():
    here = os.path.dirname(os.path.abspath(__file__))
    lines = [
        "// hl_tanh_poly.h -- written by fit_tanh_poly.py; do not edit.",
        "// tanh(y) ~= y * P(y^2) for |y| <= Y0, P(0) = 1 (coefficients C0 .. Cdeg).",
        "#pragma once",
    ]
    for name, y0, deg in FITS:
        c, err = fit(y0, deg)
        c32 = [float(np.float32(v)) for v in c]
        c32[0] = 1.0
        tag = "HL_TANH_POLY" if name == "POLY" else f"HL_TANH_{name}"
        lines.append(f"// {tag}: degree {deg} on |y| <= {y0}; max relative error of the "
                     f"real-valued fit {err:.2e}")
        lines.append(f"#define {tag}_Y0 {y0}f")
        for k, v in enumerate(c32):
            lines.append(f"#define {tag}_C{k} {v!r}f")
    with open(os.path.join(here, "hl_tanh_poly.h"), "w") as fh:
        fh.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
