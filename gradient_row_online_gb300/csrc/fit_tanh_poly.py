"""Fits the odd polynomial tanh(y) ~= y * P(y^2), |y| <= Y0, used by the
16-bit row kernel for the softcap transform on the FMA pipe (hl_tanh_poly.h).

P has degree 6 in u = y^2 with P(0) = 1.  The fit minimises the maximum
relative error of P(u) against tanh(sqrt(u)) / sqrt(u) on a dense grid by
iteratively reweighted least squares.  Run it to regenerate the header.
"""
import os

import numpy as np

Y0 = 0.8
DEG = 6


def fit(y0=Y0, deg=DEG, iters=60):
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
    c, err = fit()
    c32 = [float(np.float32(v)) for v in c]
    c32[0] = 1.0
    here = os.path.dirname(os.path.abspath(__file__))
    lines = [
        "// hl_tanh_poly.h -- written by fit_tanh_poly.py; do not edit.",
        f"// tanh(y) ~= y * P(y^2) for |y| <= {Y0}; P of degree {DEG} in u = y^2, P(0) = 1.",
        f"// Max relative error of the real-valued fit: {err:.2e}.",
        "#pragma once",
        f"#define HL_TANH_POLY_Y0 {Y0}f",
    ]
    for k, v in enumerate(c32):
        lines.append(f"#define HL_TANH_POLY_C{k} {v!r}f")
    with open(os.path.join(here, "hl_tanh_poly.h"), "w") as fh:
        fh.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
