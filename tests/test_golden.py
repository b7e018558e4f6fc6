"""The stored two-class rows (tests/golden/two_class_rows.json).

CPU: the oracle reproduces the stored values, and the stored values agree
with two-class closed forms.  With V = 2 every softmax is a logistic sigmoid
of the logit difference, so each loss, statistic and derivative has a form in
sigmoid / softplus of that difference, written here independently of the
oracle's log-sum-exp code (the loss definitions follow issue #507 Problem and
PR #549 Loss coverage; the softcap and scale follow PR #549 Approach).

GPU: the library reproduces the stored values under the parity tolerances,
for fp32, bf16 and fp16 logits (every stored logit is exact in all three).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as orc
from gradient_row_online_gb300 import workloads as W
from tests import _harness as H

FIXTURE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                       "two_class_rows.json")

with open(FIXTURE) as fh:
    DOC = json.load(fh)
CASES = {c["name"]: c for c in DOC["cases"]}


def f32(v):
    return float(np.float32(v))


def oracle_cfg(c):
    flags = 0
    for name in c["losses"]:
        flags |= H.ORACLE_BITS[name]
    return orc.make_cfg(flags, {k: f32(v) for k, v in c["weights"].items()},
                        temperature=f32(c["temperature"]), clip_eps=f32(c["clip_eps"]),
                        softcap=f32(c["softcap"]), logits_scale=f32(c["logits_scale"]),
                        grad_scale=f32(c["grad_scale"]))


def arrays(c):
    x = np.array(c["logits"], np.float64)
    lab = np.array(c["labels"], np.int64)
    t = np.array(c["teacher"], np.float64) if "teacher" in c else None
    o = np.array(c["old_logprobs"], np.float32).astype(np.float64) if "old_logprobs" in c else None
    a = np.array(c["advantages"], np.float32).astype(np.float64) if "advantages" in c else None
    return x, lab, t, o, a


# ------------------------------------------------------------ two-class closed forms

def softplus(v):
    return np.maximum(v, 0.0) + np.log1p(np.exp(-np.abs(v)))


def sigmoid(v):
    return np.where(v >= 0, 1.0 / (1.0 + np.exp(-v)), np.exp(v) / (1.0 + np.exp(v)))


def two_class(c):
    """Scalars[16] and gradient (n x 2) from the logistic forms."""
    x, lab, t, o, a = arrays(c)
    w = {k: f32(v) for k, v in c["weights"].items()}
    get = lambda k: w.get(k, 0.0)
    T, eps = f32(c["temperature"]), f32(c["clip_eps"])
    cap, s, gs = f32(c["softcap"]), f32(c["logits_scale"]), f32(c["grad_scale"])
    L = set(c["losses"])
    if cap > 0:
        th = np.tanh(x / cap)
        z, dzdx = s * cap * th, s * (1.0 - th * th)
    else:
        z, dzdx = s * x, np.full_like(x, s)
    valid = lab >= 0
    n = int(valid.sum())
    d = z[:, 1] - z[:, 0]                    # logit difference; p1 = sigmoid(d)
    p1, p0 = sigmoid(d), sigmoid(-d)
    lse = z[:, 0] + softplus(d)
    y = np.where(valid, lab, 0)
    sgn = np.where(y == 1, 1.0, -1.0)        # d(z_y - z_other) / d(d)
    ce = softplus(-sgn * d)                   # -log p_y
    dce = np.where(y == 1, -p0, p1)           # d ce / d(d)
    out = np.zeros(16)
    rows = {}
    gd = np.zeros(x.shape[0])                 # d(row loss) / d(d), weighted
    g0_extra = np.zeros(x.shape[0])           # the part of dL/dz0 + dL/dz1 (z-loss only)
    if "ce" in L:
        rows["ce"] = ce
        gd += get("ce") * dce
    if "z" in L:
        rows["z"] = lse ** 2
        # z-loss is not a function of d alone: d/dz_j (lse^2) = 2 lse p_j
        g0_extra += get("z") * 2.0 * lse
    if L & {"dist_ce", "fkl", "rkl"}:
        dT = d / T
        du = (t[:, 1] - t[:, 0]) / T
        pT1, pT0 = sigmoid(dT), sigmoid(-dT)
        q1, q0 = sigmoid(du), sigmoid(-du)
        lpT1, lpT0 = -softplus(-dT), -softplus(dT)
        lq1, lq0 = -softplus(-du), -softplus(du)
        if "dist_ce" in L:
            rows["dist_ce"] = -(q0 * lpT0 + q1 * lpT1)
            gd += get("dist_ce") * (pT1 - q1) / T
        if "fkl" in L:
            rows["fkl"] = q0 * (lq0 - lpT0) + q1 * (lq1 - lpT1)
            gd += get("fkl") * (pT1 - q1) / T
        if "rkl" in L:
            rows["rkl"] = pT0 * (lpT0 - lq0) + pT1 * (lpT1 - lq1)
            gd += get("rkl") * pT1 * pT0 * (dT - du) / T
    if L & {"grpo", "grpo_stats"}:
        lp = -ce
        rho = np.exp(lp - o)
        clipped_rho = np.clip(rho, 1.0 - eps, 1.0 + eps)
        grpo = -np.minimum(rho * a, clipped_rho * a)
        act = ~(((a > 0) & (rho > 1.0 + eps)) | ((a < 0) & (rho < 1.0 - eps)))
        if "grpo" in L:
            rows["grpo"] = grpo
            gd += get("grpo") * (-a * rho * act) * (-dce)
        if "grpo_stats" in L:
            m = lambda v: float(np.sum(np.where(valid, v, 0.0))) / n
            out[7], out[8] = m(lp), m(rho)
            clip = valid & (np.abs(rho - 1.0) > eps)
            out[9], out[15] = clip.sum() / n, float(clip.sum())
            out[10] = m(rho - 1.0 - np.log(rho))
            out[11] = m(a)
            out[12] = np.sqrt(max(m(a * a) - out[11] ** 2, 0.0))
    if "entropy" in L:
        ent = p0 * softplus(d) + p1 * softplus(-d)    # -p0 log p0 - p1 log p1
        rows["entropy"] = ent
        gd += get("entropy") * (-d * p1 * p0)
    slot = dict(ce=1, z=2, dist_ce=3, fkl=4, rkl=5, grpo=6, entropy=13)
    for k, v in rows.items():
        out[slot[k]] = float(np.sum(np.where(valid, v, 0.0))) / n
    out[0] = sum(get(k) * out[slot[k]] for k in rows)
    out[14] = n
    # dL/dz1 = gd + extra * p1, dL/dz0 = -gd + extra * p0; then the chain rule
    g = np.stack([-gd + g0_extra * p0, gd + g0_extra * p1], axis=1)
    g = np.where(valid[:, None], gs / n * g * dzdx, 0.0)
    return out, g


@pytest.mark.parametrize("name", sorted(CASES))
def test_oracle_reproduces_stored_values(name):
    c = CASES[name]
    x, lab, t, o, a = arrays(c)
    sc, rec, grad, gmag = orc.forward_backward(oracle_cfg(c), x, lab, t, o, a, want_grad=True,
                                               want_gmag=True, n_threads=1)
    e = c["expected"]
    np.testing.assert_allclose(sc, e["scalars"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(rec, e["records"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(grad, e["grad"], rtol=1e-13, atol=1e-17)
    np.testing.assert_allclose(gmag, e["gmag"], rtol=1e-13, atol=1e-17)


@pytest.mark.parametrize("name", sorted(CASES))
def test_stored_values_match_two_class_closed_forms(name):
    c = CASES[name]
    want_s, want_g = two_class(c)
    e = c["expected"]
    np.testing.assert_allclose(e["scalars"], want_s, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(e["grad"], want_g, rtol=1e-11, atol=1e-16)


def test_fixture_covers_the_grpo_branches():
    """The GRPO rows put the ratio outside both bounds with either advantage
    sign, and inside them, none within reach of a bound."""
    rf = DOC["record_fields"]
    seen = set()
    for c in CASES.values():
        if "advantages" not in c:
            continue
        for r, a in zip(c["expected"]["records"], c["advantages"]):
            if not r[rf["valid"]]:
                continue
            assert r[rf["ambiguous"]] == 0.0
            rho = r[rf["ratio"]]
            seen.add((rho > 1.2, rho < 0.8, a > 0, bool(r[rf["act"]])))
    assert (True, False, True, False) in seen      # rho > 1+eps, A > 0: clipped branch
    assert (True, False, False, True) in seen      # rho > 1+eps, A < 0: unclipped branch
    assert (False, True, False, False) in seen     # rho < 1-eps, A < 0: clipped branch
    assert (False, True, True, True) in seen       # rho < 1-eps, A > 0: unclipped branch
    assert (False, False, True, True) in seen      # inside the bounds


# ------------------------------------------------------------------------ GPU

@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("name", sorted(CASES))
def test_library_reproduces_stored_values(name, dtype):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    c = CASES[name]
    x, lab, t, o, a = arrays(c)
    weights = dict(ce=0.0, z=0.0, dist_ce=0.0, fkl=0.0, rkl=0.0, grpo=0.0, entropy=0.0)
    weights.update(c["weights"])
    weights["grad_scale"] = c["grad_scale"]
    wl = W.Workload(name, x.shape[0], x.shape[1], dtype, tuple(c["losses"]), weights,
                    temperature=c["temperature"], clip_eps=c["clip_eps"], softcap=c["softcap"],
                    logits_scale=c["logits_scale"])
    dev = "cuda"
    inp = dict(logits=torch.tensor(x, dtype=dtype, device=dev),
               labels=torch.tensor(lab, device=dev),
               teacher=None if t is None else torch.tensor(t, dtype=dtype, device=dev),
               old_logprobs=None if o is None else torch.tensor(o, dtype=torch.float32, device=dev),
               advantages=None if a is None else torch.tensor(a, dtype=torch.float32, device=dev))
    assert np.array_equal(inp["logits"].double().cpu().numpy(), x)    # exact in dtype
    got, g, _ = H.run_gpu(wl, inp)
    e = c["expected"]
    rec = np.array(e["records"])
    ref = H.check_scalars(wl, got, oracle_cfg(c), rec)
    np.testing.assert_allclose(ref, e["scalars"], rtol=1e-13, atol=1e-15)
    H.check_grad(wl, g, np.array(e["grad"]), np.array(e["gmag"]), rec)
