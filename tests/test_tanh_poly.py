"""CPU check of the softcap tanh polynomial the 16-bit kernel evaluates on
the FMA pipe: fp32 Horner evaluation (each step an fp32-rounded fma) against
numpy's tanh over its whole range, including the odd symmetry and y = 0."""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "gradient_row_online_gb300", "csrc", "hl_tanh_poly.h")


def coeffs():
    txt = open(HDR).read()
    y0 = float(re.search(r"HL_TANH_POLY_Y0 ([0-9.eE+-]+)f", txt).group(1))
    c = {int(k): float(v) for k, v in re.findall(r"HL_TANH_POLY_C(\d) ([0-9.eE+-]+)f", txt)}
    return y0, [np.float32(c[k]) for k in sorted(c)]


def fma32(a, b, c):
    # the product of two fp32 values is exact in fp64; one rounding to fp32
    return (a.astype(np.float64) * b.astype(np.float64) + np.float64(c)).astype(np.float32)


def tanh_poly32(y):
    y0, c = coeffs()
    y = y.astype(np.float32)
    u = (y * y).astype(np.float32)
    p = np.full_like(u, c[-1])
    for ck in reversed(c[:-1]):
        p = fma32(p, u, ck)
    return (y * p).astype(np.float32)


def test_polynomial_matches_tanh_on_its_range():
    y0, c = coeffs()
    assert c[0] == 1.0 and len(c) == 7
    y = np.linspace(-y0, y0, 400001).astype(np.float32)
    err = np.abs(tanh_poly32(y).astype(np.float64) - np.tanh(y.astype(np.float64)))
    assert err.max() < 1.2e-7
    # error relative to tanh itself stays at fp32 rounding level away from 0
    far = np.abs(y) > 1e-3
    rel = err[far] / np.abs(np.tanh(y[far].astype(np.float64)))
    assert rel.max() < 4e-7


def test_polynomial_is_odd_and_exact_at_zero():
    y = np.linspace(0, 0.8, 1001).astype(np.float32)
    assert np.array_equal(tanh_poly32(y), -tanh_poly32(-y))
    assert tanh_poly32(np.zeros(1, np.float32))[0] == 0.0
