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


def tier_coeffs(tag):
    txt = open(HDR).read()
    y0 = float(re.search(rf"HL_TANH_{tag}_Y0 ([0-9.eE+-]+)f", txt).group(1))
    c = {int(k): float(v) for k, v in re.findall(rf"HL_TANH_{tag}_C(\d) ([0-9.eE+-]+)f", txt)}
    return y0, [np.float64(np.float32(c[k])) for k in sorted(c)]


def folded_zs32(x, tag, s, c):
    """The streaming kernel's softcap transform in base 2, zs = x * Q(x^2),
    with Q_k = s * log2(e) * C_k / c^(2k) formed in fp64 and rounded to fp32,
    Horner in fp32 fmas, and 1 - tanh^2 as 1 - zs^2 / Kc^2."""
    _, cc = tier_coeffs(tag)
    f = s * 1.4426950408889634
    q = []
    for ck in cc:
        q.append(np.float32(ck * f))
        f /= c * c
    x = x.astype(np.float32)
    u = (x * x).astype(np.float32)
    p = np.full_like(u, q[-1])
    for qk in reversed(q[:-1]):
        p = fma32(p, u, qk)
    zs = (x * p).astype(np.float32)
    kc = np.float32(np.float32(s) * np.float32(c) * np.float32(1.4426950408889634))
    m = np.float32(-1.0) / (kc * kc)
    omt = fma32(zs, (zs * m).astype(np.float32), np.float32(1.0))
    return zs, omt


def test_folded_tiers_match_scaled_tanh():
    # (tier, bound on the relative error of zs)
    for tag, tol in (("A", 6e-7), ("B", 4e-7)):
        y0, cc = tier_coeffs(tag)
        assert cc[0] == 1.0
        for s, c in ((0.5, 30.0), (1.0, 3.0), (1.0, 20.0), (2.0, 50.0), (0.7, 1.0)):
            x = np.linspace(-y0 * c, y0 * c, 200001).astype(np.float32)
            zs, omt = folded_zs32(x, tag, s, c)
            ref = s * c * np.log2(np.e) * np.tanh(x.astype(np.float64) / c)
            far = np.abs(x) > 1e-3 * c
            rel = np.abs(zs[far] - ref[far]) / np.abs(ref[far])
            assert rel.max() < tol, (tag, s, c, rel.max())
            # 1 - tanh^2 against 1 / cosh^2 (no cancellation on these ranges)
            ref_omt = 1.0 / np.cosh(x.astype(np.float64) / c) ** 2
            assert np.abs(omt - ref_omt).max() < 1e-6, (tag, s, c)
            assert np.array_equal(zs, -folded_zs32(-x, tag, s, c)[0])
