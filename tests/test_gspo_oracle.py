"""Pins of the GSPO oracle (oracle.gspo_forward_backward) against what the
method and the mathematics fix, none of it a retyping of the oracle:

- segments of one token are GRPO, token for token: loss, clip fraction, ratio
  mean and gradient equal the (separately pinned) GRPO row oracle's;
- central finite differences of the loss in every logit;
- at the old policy every sequence ratio is 1: the loss is minus the mean
  sequence advantage and each token's coefficient has a closed form;
- without clipping the loss is -(1/G) sum_i s_i A_i, with s_i the geometric
  mean of the token ratios (a product, not the oracle's log-sum);
- clipped sequences with a positive advantage carry no gradient.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as orc


def _lp(x, labels, softcap=0.0, scale=1.0):
    """Label log-prob by torch.log_softmax of the capped, scaled logits."""
    z = scale * (softcap * np.tanh(x / softcap) if softcap > 0 else x)
    lp = F.log_softmax(torch.from_numpy(z), -1)
    safe = torch.from_numpy(np.where(labels >= 0, labels, 0))
    out = lp.gather(1, safe[:, None])[:, 0].numpy().copy()
    out[labels < 0] = 0.0
    return out


def _problem(seed, n=18, V=11, mask_frac=0.2):
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 2.0, (n, V))
    labels = rng.integers(0, V, n).astype(np.int64)
    labels[rng.random(n) < mask_frac] = -100
    adv = rng.normal(0.0, 1.0, n)
    return rng, x, labels, adv


@pytest.mark.parametrize("softcap,scale", [(0.0, 1.0), (4.0, 0.8)])
def test_one_token_segments_are_grpo(softcap, scale):
    rng, x, labels, adv = _problem(1)
    n = x.shape[0]
    old = _lp(x, labels, softcap, scale) + rng.normal(0, 0.3, n)
    off = np.arange(n + 1)
    eps, w, gs = 0.2, 0.7, 1.3
    s, coeff, g = orc.gspo_forward_backward(x, labels, old, adv, off, eps, weight=w,
                                            grad_scale=gs, softcap=softcap, logits_scale=scale)
    cfg = orc.make_cfg(orc.GRPO | orc.GRPO_STATS, dict(ce=0.0, grpo=w), clip_eps=eps,
                       softcap=softcap, logits_scale=scale, grad_scale=gs)
    sr, rec, gr, _ = orc.forward_backward(cfg, x, labels, old_logprobs=old, advantages=adv)
    assert abs(s[0] - sr[6]) < 1e-12
    assert abs(s[1] - sr[8]) < 1e-12
    assert abs(s[2] - sr[9]) < 1e-12
    assert s[3] == sr[14]
    assert np.abs(g - gr).max() < 1e-12


def test_gradient_matches_central_finite_differences():
    rng, x, labels, adv = _problem(2, n=9, V=6, mask_frac=0.0)
    labels[4] = -100
    off = np.array([0, 3, 4, 9])  # the middle segment holds one masked token only
    old = _lp(x, labels, 3.0, 0.9) + rng.normal(0, 0.25, x.shape[0])
    eps, w, gs = 0.15, 0.6, 1.1

    def loss(xx):
        return w * gs * orc.gspo_forward_backward(xx, labels, old, adv, off, eps, softcap=3.0,
                                                  logits_scale=0.9)[0][0]

    _, _, g = orc.gspo_forward_backward(x, labels, old, adv, off, eps, weight=w, grad_scale=gs,
                                        softcap=3.0, logits_scale=0.9)
    h = 1e-5
    fd = np.zeros_like(x)
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            xp = x.copy(); xp[i, j] += h
            xm = x.copy(); xm[i, j] -= h
            fd[i, j] = (loss(xp) - loss(xm)) / (2 * h)
    assert np.abs(fd - g).max() < 1e-8 * max(1.0, np.abs(g).max())
    assert np.abs(g[4]).max() == 0.0


def test_at_the_old_policy():
    _, x, labels, adv = _problem(3, n=20)
    old = _lp(x, labels)
    off = np.array([0, 5, 5, 12, 20])  # an empty segment too
    s, coeff, _ = orc.gspo_forward_backward(x, labels, old, adv, off, 0.2, weight=1.0)
    segs = [np.arange(a, b) for a, b in zip(off[:-1], off[1:])]
    segs = [t[labels[t] >= 0] for t in segs]
    segs = [t for t in segs if t.size]
    G = len(segs)
    A = [adv[t].mean() for t in segs]
    assert abs(s[0] + np.mean(A)) < 1e-12
    assert abs(s[1] - 1.0) < 1e-12 and s[2] == 0.0 and s[3] == G
    ref = np.zeros_like(coeff)
    for t, a in zip(segs, A):
        ref[t] = -a / (G * t.size)
    assert np.abs(coeff - ref).max() < 1e-15


def test_without_clipping_is_the_geometric_mean_ratio():
    rng, x, labels, adv = _problem(4, n=16)
    lp = _lp(x, labels)
    old = lp + rng.normal(0, 0.5, x.shape[0])
    off = np.array([0, 4, 9, 16])
    s, _, _ = orc.gspo_forward_backward(x, labels, old, adv, off, 1e9)
    objs, ratios = [], []
    for a, b in zip(off[:-1], off[1:]):
        t = np.arange(a, b)
        t = t[labels[t] >= 0]
        r = float(np.prod(np.exp(lp[t] - old[t]))) ** (1.0 / t.size)
        objs.append(r * adv[t].mean())
        ratios.append(r)
    assert abs(s[0] + np.mean(objs)) < 1e-12
    assert abs(s[1] - np.mean(ratios)) < 1e-12


def test_clipped_sequences_with_positive_advantage_carry_no_gradient():
    _, x, labels, _ = _problem(5, n=12, mask_frac=0.0)
    lp = _lp(x, labels)
    eps = 0.2
    old = lp - 0.5  # every sequence ratio e^0.5 > 1 + eps
    adv = np.full(x.shape[0], 0.8)
    off = np.array([0, 6, 12])
    s, coeff, g = orc.gspo_forward_backward(x, labels, old, adv, off, eps)
    assert abs(s[0] + (1 + eps) * 0.8) < 1e-12
    assert s[2] == 1.0
    assert np.abs(coeff).max() == 0.0 and np.abs(g).max() == 0.0
    # a negative advantage takes the unclipped branch: gradient flows
    s2, coeff2, _ = orc.gspo_forward_backward(x, labels, old, -adv, off, eps)
    assert abs(s2[0] - math.exp(0.5) * 0.8) < 1e-12
    assert np.abs(coeff2).min() > 0.0


def test_rejects_bad_offsets():
    _, x, labels, adv = _problem(6, n=5)
    old = np.zeros(5)
    for off in ([1, 5], [0, 3, 2, 5], [0, 4]):
        with pytest.raises(ValueError):
            orc.gspo_forward_backward(x, labels, old, adv, np.array(off), 0.2)
