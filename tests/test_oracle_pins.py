"""Pins for the fp64 oracle, against things other than itself (CPU only).

Closed forms, invariants, library special cases and central finite
differences.  Each pin is chosen so that a plausible slip in the oracle (a
dropped term, a wrong sign or temperature factor, KL arguments swapped, min
taken as max) fails at least one of them.
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as orc

ALL_FLAGS = (orc.CE, orc.Z, orc.DIST_CE, orc.FKL, orc.RKL, orc.GRPO, orc.GRPO_STATS, orc.ENTROPY)
ALL = sum(ALL_FLAGS)


def _slots(s):
    return dict(zip(orc.SLOTS, s))


def _rand_problem(rng, n, V, sigma=2.0, mask_frac=0.25, teacher_noise=1.0):
    x = rng.normal(0.0, sigma, (n, V))
    labels = rng.integers(0, V, n).astype(np.int64)
    labels[rng.random(n) < mask_frac] = -100
    t = x + rng.normal(0.0, teacher_noise, (n, V))
    adv = rng.normal(0.0, 1.0, n)
    return x, labels, t, adv


def _torch_lp(z, labels):
    """Label log-prob by torch.log_softmax (a library routine), 0 on masked rows."""
    lp = F.log_softmax(torch.from_numpy(z), -1)
    safe = torch.from_numpy(np.where(labels >= 0, labels, 0))
    out = lp.gather(1, safe[:, None])[:, 0].numpy().copy()
    out[labels < 0] = 0.0
    return out


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("V", [1, 2, 7, 1000])
@pytest.mark.parametrize("softcap,scale", [(0.0, 1.0), (30.0, 0.5), (5.0, 2.0)])
def test_uniform_row_ce_and_entropy_are_log_v(V, softcap, scale):
    x = np.full((3, V), 1.7)
    labels = np.array([0, V - 1, V // 2], np.int64)
    cfg = orc.make_cfg(orc.CE | orc.ENTROPY, softcap=softcap, logits_scale=scale)
    s, _, _, _ = orc.forward_backward(cfg, x, labels)
    assert abs(s[1] - math.log(V)) < 1e-12
    assert abs(s[13] - math.log(V)) < 1e-12
    assert s[14] == 3


@pytest.mark.parametrize("V", [1, 5, 1024])
def test_uniform_row_z_loss_is_square_of_shifted_log_v(V):
    c0 = -0.8
    x = np.full((4, V), c0)
    cfg = orc.make_cfg(orc.Z, weights=dict(ce=0.0, z=1.0))
    s, _, _, _ = orc.forward_backward(cfg, x, None)
    assert abs(s[2] - (c0 + math.log(V)) ** 2) < 1e-12


@pytest.mark.parametrize("T", [1.0, 2.0, 0.7])
def test_distillation_against_itself_has_zero_kl_and_no_gradient(T):
    rng = np.random.default_rng(1)
    x = rng.normal(0, 3, (4, 33))
    flags = orc.DIST_CE | orc.FKL | orc.RKL
    cfg = orc.make_cfg(flags, weights=dict(ce=0.0, fkl=0.7, rkl=1.3, dist_ce=0.0), temperature=T)
    s, _, g, _ = orc.forward_backward(cfg, x, None, teacher=x)
    assert abs(s[4]) < 1e-13 and abs(s[5]) < 1e-13
    assert np.abs(g).max() < 1e-15
    # from-distribution CE of a distribution against itself is its entropy
    H = torch.distributions.Categorical(logits=torch.from_numpy(x / T)).entropy().mean().item()
    assert abs(s[3] - H) < 1e-12


# ----------------------------------------------------------- library routines

def test_ce_matches_torch_cross_entropy_with_ignore_index():
    rng = np.random.default_rng(2)
    x, labels, _, _ = _rand_problem(rng, 40, 97, sigma=3.0)
    cfg = orc.make_cfg(orc.CE)
    s, rec, _, _ = orc.forward_backward(cfg, x, labels)
    ref = F.cross_entropy(torch.from_numpy(x), torch.from_numpy(labels), ignore_index=-100)
    assert abs(s[1] - ref.item()) < 1e-12
    assert s[14] == int((labels >= 0).sum())


def test_ce_gradient_matches_torch_autograd():
    rng = np.random.default_rng(3)
    x, labels, _, _ = _rand_problem(rng, 12, 31)
    cfg = orc.make_cfg(orc.CE, grad_scale=0.37)
    _, _, g, _ = orc.forward_backward(cfg, x, labels)
    xt = torch.from_numpy(x).requires_grad_()
    (0.37 * F.cross_entropy(xt, torch.from_numpy(labels), ignore_index=-100)).backward()
    assert np.abs(g - xt.grad.numpy()).max() < 1e-15


def test_softcapped_ce_matches_torch_on_capped_logits():
    rng = np.random.default_rng(4)
    x, labels, _, _ = _rand_problem(rng, 16, 50, sigma=20.0)
    c, s_ = 7.0, 0.5
    cfg = orc.make_cfg(orc.CE, softcap=c, logits_scale=s_)
    s, _, _, _ = orc.forward_backward(cfg, x, labels)
    z = s_ * c * torch.tanh(torch.from_numpy(x) / c)
    ref = F.cross_entropy(z, torch.from_numpy(labels), ignore_index=-100)
    assert abs(s[1] - ref.item()) < 1e-12


def test_z_loss_is_mean_square_logsumexp():
    rng = np.random.default_rng(5)
    x, labels, _, _ = _rand_problem(rng, 30, 64)
    cfg = orc.make_cfg(orc.Z | orc.CE, weights=dict(z=0.1))
    s, _, _, _ = orc.forward_backward(cfg, x, labels)
    keep = labels >= 0
    lse = torch.logsumexp(torch.from_numpy(x[keep]), -1)
    assert abs(s[2] - (lse ** 2).mean().item()) < 1e-12
    assert abs(s[0] - (s[1] + 0.1 * s[2])) < 1e-12


def test_entropy_matches_torch_categorical():
    rng = np.random.default_rng(6)
    x, labels, _, _ = _rand_problem(rng, 25, 40, sigma=4.0)
    cfg = orc.make_cfg(orc.ENTROPY, weights=dict(ce=0.0))
    s, _, _, _ = orc.forward_backward(cfg, x, labels)
    keep = labels >= 0
    H = torch.distributions.Categorical(logits=torch.from_numpy(x[keep])).entropy().mean()
    assert abs(s[13] - H.item()) < 1e-12


@pytest.mark.parametrize("T", [1.0, 1.5, 2.0])
def test_distillation_losses_match_torch_kl_div_and_soft_cross_entropy(T):
    rng = np.random.default_rng(7)
    x, labels, t, _ = _rand_problem(rng, 20, 45, sigma=3.0)
    flags = orc.DIST_CE | orc.FKL | orc.RKL
    cfg = orc.make_cfg(flags, weights=dict(ce=0.0), temperature=T)
    s, _, _, _ = orc.forward_backward(cfg, x, labels, teacher=t)
    keep = labels >= 0
    log_pT = F.log_softmax(torch.from_numpy(x[keep] / T), -1)
    log_q = F.log_softmax(torch.from_numpy(t[keep] / T), -1)
    n = int(keep.sum())
    fkl = F.kl_div(log_pT, log_q, reduction="sum", log_target=True).item() / n
    rkl = F.kl_div(log_q, log_pT, reduction="sum", log_target=True).item() / n
    dce = F.cross_entropy(torch.from_numpy(x[keep] / T), log_q.exp()).item()
    assert abs(s[4] - fkl) < 1e-12
    assert abs(s[5] - rkl) < 1e-12
    assert abs(s[3] - dce) < 1e-12


# ------------------------------------------------------------------- GRPO

def _grpo_setup(rng, n=24, V=19):
    x, labels, _, _ = _rand_problem(rng, n, V)
    lp = _torch_lp(x, labels)
    return x, labels, lp


def test_grpo_at_the_old_policy():
    rng = np.random.default_rng(8)
    x, labels, lp = _grpo_setup(rng)
    adv = rng.normal(0, 1, x.shape[0])
    cfg = orc.make_cfg(orc.GRPO | orc.GRPO_STATS, weights=dict(ce=0.0))
    s, _, _, _ = orc.forward_backward(cfg, x, labels, old_logprobs=lp, advantages=adv)
    keep = labels >= 0
    d = _slots(s)
    assert abs(d["ratio_mean"] - 1.0) < 1e-12
    assert d["clip_frac"] == 0.0 and d["n_clipped"] == 0.0
    assert abs(d["kl_k3"]) < 1e-12
    assert abs(d["grpo_loss"] + adv[keep].mean()) < 1e-12
    assert abs(d["new_logprob_mean"] - lp[keep].mean()) < 1e-12
    assert abs(d["adv_mean"] - adv[keep].mean()) < 1e-13
    assert abs(d["adv_std"] - adv[keep].std()) < 1e-12


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_grpo_clipping_takes_the_minimum(sign):
    rng = np.random.default_rng(9)
    x, labels, lp = _grpo_setup(rng)
    keep = labels >= 0
    eps, shift = 0.2, 0.5  # rho = e^0.5 > 1 + eps on every row
    adv = sign * (0.5 + rng.random(x.shape[0]))
    cfg = orc.make_cfg(orc.GRPO | orc.GRPO_STATS, weights=dict(ce=0.0), clip_eps=eps)
    s, _, g, _ = orc.forward_backward(cfg, x, labels, old_logprobs=lp - shift, advantages=adv)
    d = _slots(s)
    rho = math.exp(shift)
    assert abs(d["ratio_mean"] - rho) < 1e-12
    assert d["n_clipped"] == keep.sum() and d["clip_frac"] == 1.0
    assert abs(d["kl_k3"] - (rho - 1 - shift)) < 1e-12
    if sign > 0:  # the clipped surrogate is the smaller one: no gradient
        assert abs(d["grpo_loss"] + (1 + eps) * adv[keep].mean()) < 1e-12
        assert np.abs(g).max() == 0.0
    else:  # negative advantage: the unclipped surrogate is the smaller one
        assert abs(d["grpo_loss"] + rho * adv[keep].mean()) < 1e-12
        assert np.abs(g[keep]).max() > 1e-3


def test_grpo_without_clipping_is_plain_policy_gradient():
    rng = np.random.default_rng(10)
    x, labels, lp = _grpo_setup(rng)
    old = lp + rng.normal(0, 0.7, x.shape[0])
    adv = rng.normal(0, 1, x.shape[0])
    cfg = orc.make_cfg(orc.GRPO, weights=dict(ce=0.0), clip_eps=1e9)
    s, _, _, _ = orc.forward_backward(cfg, x, labels, old_logprobs=old, advantages=adv)
    keep = labels >= 0
    ref = -(np.exp(lp - old) * adv)[keep].mean()
    assert abs(s[6] - ref) < 1e-12


# ----------------------------------------------------- masking / invariances

def test_masked_rows_have_exact_zero_gradient_and_are_not_counted():
    rng = np.random.default_rng(11)
    x, labels, t, adv = _rand_problem(rng, 10, 23, mask_frac=0.5)
    lp = _torch_lp(x, labels)
    cfg = orc.make_cfg(ALL, weights=dict(z=0.1, fkl=0.5, rkl=0.5, dist_ce=0.2, entropy=0.3),
                       temperature=1.5, softcap=10.0, logits_scale=0.5)
    s, rec, g, _ = orc.forward_backward(cfg, x, labels, t, lp + 0.1, adv)
    m = labels < 0
    assert m.any()
    assert np.all(g[m] == 0.0) and not np.signbit(g[m]).any()
    assert s[14] == (~m).sum()
    assert np.all(rec[m] == 0.0)


def test_all_rows_masked_gives_zeros():
    rng = np.random.default_rng(12)
    x, _, t, adv = _rand_problem(rng, 5, 9)
    labels = np.full(5, -100, np.int64)
    cfg = orc.make_cfg(ALL, weights=dict(z=0.1, fkl=0.5))
    s, _, g, _ = orc.forward_backward(cfg, x, labels, t, np.zeros(5), adv)
    assert np.all(s == 0.0) and np.all(g == 0.0)


@pytest.mark.parametrize("seed", range(4))
def test_gradient_row_sums_to_z_loss_term(seed):
    """Every loss but z-loss has a zero-sum gradient over the vocabulary."""
    rng = np.random.default_rng(20 + seed)
    x, labels, t, adv = _rand_problem(rng, 8, 29)
    lp = _torch_lp(x, labels)
    wz, s_, gs = 0.3, 0.75, 1.7
    cfg = orc.make_cfg(ALL, weights=dict(z=wz, fkl=0.5, rkl=0.25, dist_ce=0.2, entropy=0.1),
                       temperature=1.3, logits_scale=s_, grad_scale=gs)
    s, rec, g, _ = orc.forward_backward(cfg, x, labels, t, lp + 0.05, adv)
    n = s[14]
    keep = labels >= 0
    lse = torch.logsumexp(torch.from_numpy(s_ * x), -1).numpy()
    expect = s_ * 2.0 * (gs / n) * wz * lse
    assert np.allclose(g.sum(1)[keep], expect[keep], rtol=1e-11, atol=1e-14)


def test_logits_scale_is_the_chain_rule():
    rng = np.random.default_rng(13)
    x, labels, t, adv = _rand_problem(rng, 6, 17)
    s_ = 0.37
    lp = _torch_lp(s_ * x, labels)
    flags = orc.CE | orc.Z | orc.GRPO | orc.ENTROPY
    w = dict(z=0.2, entropy=0.4)
    a = orc.forward_backward(orc.make_cfg(flags, w, logits_scale=s_), x, labels, None, lp + .1, adv)
    b = orc.forward_backward(orc.make_cfg(flags, w, logits_scale=1.0), s_ * x, labels, None,
                             lp + .1, adv)
    assert np.allclose(a[0], b[0], rtol=1e-12, atol=1e-14)
    assert np.allclose(a[2], s_ * b[2], rtol=1e-11, atol=1e-16)


@pytest.mark.parametrize("y", [0.3, 4.0, 12.0, 25.0])
def test_saturated_softcap_gradient_keeps_relative_accuracy(y):
    """Two classes, label 0, softcap c, logits (c*y, 0): dCE/dx_0 = (p_0 - 1) * s * sech^2(y),
    with sech^2(y) = 4 e^{-2y} / (1 + e^{-2y})^2 written out independently of cosh / tanh."""
    c, s_ = 3.0, 0.7
    x = np.array([[c * y, 0.0]])
    cfg = orc.make_cfg(orc.CE, softcap=c, logits_scale=s_)
    _, _, g, _ = orc.forward_backward(cfg, x, np.array([0], np.int64))
    e = math.exp(-2.0 * y)
    sech2 = 4.0 * e / (1.0 + e) ** 2
    z0 = s_ * c * math.tanh(y)
    p0 = 1.0 / (1.0 + math.exp(-z0))
    expect = (p0 - 1.0) * s_ * sech2
    assert abs(g[0, 0] - expect) <= 1e-12 * abs(expect)


def test_softcap_limit_is_no_softcap():
    rng = np.random.default_rng(14)
    x, labels, t, adv = _rand_problem(rng, 6, 17)
    lp = _torch_lp(x, labels)
    w = dict(z=0.2, fkl=0.3, rkl=0.3, entropy=0.1)
    a = orc.forward_backward(orc.make_cfg(ALL, w, softcap=1e7), x, labels, t, lp + .1, adv)
    b = orc.forward_backward(orc.make_cfg(ALL, w, softcap=0.0), x, labels, t, lp + .1, adv)
    assert np.allclose(a[0], b[0], rtol=1e-9, atol=1e-12)
    assert np.allclose(a[2], b[2], rtol=1e-9, atol=1e-14)


# -------------------------------------------------------- finite differences

def _fd_problem(seed):
    rng = np.random.default_rng(100 + seed)
    n, V = 3, 6
    x, labels, t, adv = _rand_problem(rng, n, V, mask_frac=0.0)
    labels[1] = -100
    lp = _torch_lp(0.8 * 4.0 * np.tanh(x / 4.0), labels)
    eps = 0.2
    # old log-probs: some rows inside the clip band, some outside, none near a kink
    while True:
        old = lp + rng.normal(0, 0.3, n)
        lr = lp - old
        if np.all(np.abs(np.abs(lr) - np.log(1 + eps)) > 0.02) and np.all(
                np.abs(lr - np.log(1 - eps)) > 0.02):
            break
    return x, labels, t, old, adv


SUBSETS = [sum(c) for r in range(1, 9) for c in itertools.combinations(ALL_FLAGS, r)]


@pytest.mark.parametrize("seed", range(2))
def test_gradient_matches_central_finite_differences_for_every_flag_subset(seed):
    x, labels, t, old, adv = _fd_problem(seed)
    w = dict(ce=0.9, z=0.3, dist_ce=0.4, fkl=0.6, rkl=0.7, grpo=1.1, entropy=0.5)
    h = 1e-5
    for flags in SUBSETS:
        cfg = orc.make_cfg(flags, w, temperature=1.7, clip_eps=0.2, softcap=4.0,
                           logits_scale=0.8, grad_scale=1.3)
        s, _, g, _ = orc.forward_backward(cfg, x, labels, t, old, adv)

        def loss(xx):
            return 1.3 * orc.forward_backward(cfg, xx, labels, t, old, adv, want_grad=False)[0][0]

        fd = np.zeros_like(x)
        for i in range(x.shape[0]):
            for j in range(x.shape[1]):
                xp = x.copy(); xp[i, j] += h
                xm = x.copy(); xm[i, j] -= h
                fd[i, j] = (loss(xp) - loss(xm)) / (2 * h)
        err = np.abs(fd - g).max()
        assert err < 1e-8 * max(1.0, np.abs(g).max()), (flags, err)


def test_rejects_missing_inputs():
    x = np.zeros((2, 4))
    with pytest.raises(ValueError):
        orc.forward_backward(orc.make_cfg(orc.CE), x, None)
    with pytest.raises(ValueError):
        orc.forward_backward(orc.make_cfg(orc.FKL), x, np.zeros(2, np.int64))
    with pytest.raises(ValueError):
        orc.forward_backward(orc.make_cfg(orc.GRPO), x, np.zeros(2, np.int64))
    with pytest.raises(ValueError):
        orc.forward_backward(orc.make_cfg(orc.CE), x, np.array([0, 4], np.int64))


# ------------------------------------------------- LM head in front of the loss

def _lm_head_problem(seed, n=3, D=4, V=5):
    rng = np.random.default_rng(300 + seed)
    hid = rng.normal(0.0, 1.0, (n, D))
    wt = rng.normal(0.0, 0.8, (V, D))
    labels = rng.integers(0, V, n).astype(np.int64)
    labels[1] = -100
    t = hid @ wt.T + rng.normal(0.0, 1.0, (n, V))
    adv = rng.normal(0.0, 1.0, n)
    x = hid @ wt.T
    lp = _torch_lp(0.8 * 4.0 * np.tanh(x / 4.0), labels)
    while True:  # old log-probs away from the clip kinks
        old = lp + rng.normal(0, 0.3, n)
        lr = lp - old
        if np.all(np.abs(np.abs(lr) - np.log(1.2)) > 0.02) and np.all(
                np.abs(lr - np.log(0.8)) > 0.02):
            break
    return hid, wt, labels, t, old, adv


@pytest.mark.parametrize("flags", [orc.CE | orc.Z, orc.FKL | orc.RKL | orc.DIST_CE,
                                   orc.GRPO | orc.GRPO_STATS | orc.ENTROPY, ALL])
def test_lm_head_gradients_match_finite_differences(flags):
    """dH and dW against central differences of grad_scale * total in every entry
    of hidden and weight (a transposed or misplaced matmul operand fails)."""
    hid, wt, labels, t, old, adv = _lm_head_problem(0)
    cfg = orc.make_cfg(flags, dict(ce=0.9, z=0.3, dist_ce=0.4, fkl=0.6, rkl=0.7, grpo=1.1,
                                   entropy=0.5),
                       temperature=1.7, clip_eps=0.2, softcap=4.0, logits_scale=0.8,
                       grad_scale=1.3)
    _, _, dH, dW, _, _ = orc.lm_head_forward_backward(cfg, hid, wt, labels, t, old, adv)

    def loss(hh, ww):
        x = hh @ ww.T
        return 1.3 * orc.forward_backward(cfg, x, labels, t, old, adv, want_grad=False)[0][0]

    step = 1e-5
    for a, d in ((hid, dH), (wt, dW)):
        fd = np.zeros_like(a)
        for idx in np.ndindex(*a.shape):
            ap = a.copy(); ap[idx] += step
            am = a.copy(); am[idx] -= step
            args_p = (ap, wt) if a is hid else (hid, ap)
            args_m = (am, wt) if a is hid else (hid, am)
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * step)
        assert np.abs(fd - d).max() < 1e-8 * max(1.0, np.abs(d).max()), (flags, a.shape)


def test_lm_head_with_identity_weight_is_the_row_loss():
    """weight = I (D = V): the logits are the hidden states, dH is the logits
    gradient and dW = G^T hidden."""
    rng = np.random.default_rng(7)
    n, V = 4, 6
    x, labels, t, adv = _rand_problem(rng, n, V)
    old = rng.normal(-2.0, 0.5, n)
    cfg = orc.make_cfg(ALL, dict(z=0.2, dist_ce=0.3, fkl=0.4, rkl=0.5, entropy=0.1),
                       temperature=1.3, softcap=5.0, logits_scale=0.7)
    s, rec, dH, dW, logits, g = orc.lm_head_forward_backward(cfg, x, np.eye(V), labels, t,
                                                             old, adv)
    s2, rec2, g2, _ = orc.forward_backward(cfg, x, labels, t, old, adv)
    np.testing.assert_array_equal(logits, x)
    np.testing.assert_array_equal(s, s2)
    np.testing.assert_array_equal(dH, g2)
    np.testing.assert_allclose(dW, g2.T @ x, rtol=0, atol=0)


def test_lm_head_scaling_identities():
    """Scaling the weight by a: d/da total(H, aW) at a = 1 equals sum(dW * W) and
    equals sum(dH * H) (both are the derivative along the logits themselves)."""
    hid, wt, labels, t, old, adv = _lm_head_problem(1, n=4, D=3, V=7)
    cfg = orc.make_cfg(orc.CE | orc.Z | orc.FKL | orc.ENTROPY,
                       dict(z=0.1, fkl=0.5, entropy=0.2), temperature=1.5)
    _, _, dH, dW, _, _ = orc.lm_head_forward_backward(cfg, hid, wt, labels, t, old, adv)
    step = 1e-6
    tot = lambda a: orc.forward_backward(cfg, hid @ (a * wt).T, labels, t, old, adv,
                                         want_grad=False)[0][0]
    dda = (tot(1 + step) - tot(1 - step)) / (2 * step)
    assert abs(dda - np.sum(dW * wt)) < 1e-7 * max(1.0, abs(dda))
    assert abs(dda - np.sum(dH * hid)) < 1e-7 * max(1.0, abs(dda))


# ------------------------------------------------- per-tile first-pass records

def _merge_records(rec):
    """Merge a row's tile records by their maxima (the block-wise online form)."""
    M = rec[:, 0].max()
    al = np.exp2(rec[:, 0] - M)
    S = np.sum(al * rec[:, 1])
    E = np.sum(al * (rec[:, 2] + (rec[:, 0] - M) * rec[:, 1]))
    return M, S, E


@pytest.mark.parametrize("softcap,scale", [(0.0, 1.0), (30.0, 0.5), (3.0, 0.7)])
def test_tile_records_merge_to_the_row_oracle_lse_and_entropy(softcap, scale):
    """Merged over a row's tiles, the records give the C row oracle's log-sum-exp
    (ln 2 (m2 + log2 S)) and entropy (ln 2 (log2 S - E / S))."""
    rng = np.random.default_rng(3)
    n, V = 5, 1024
    x = rng.normal(0.0, 3.0, (n, V))
    labels = rng.integers(0, V, n).astype(np.int64)
    rec = orc.tile_records(x, softcap, scale)
    assert rec.shape == (n, 4, 4)
    cfg = orc.make_cfg(orc.CE | orc.ENTROPY, dict(entropy=1.0), softcap=softcap,
                       logits_scale=scale)
    rr, _, _ = orc.rows(cfg, x, labels, want_grad=False)
    for i in range(n):
        M, S, E = _merge_records(rec[i])
        assert abs(math.log(2) * (M + math.log2(S)) - rr[i, orc.RF["lse"]]) < 1e-12
        H = math.log(2) * (math.log2(S) - E / S)
        assert abs(H - rr[i, orc.RF["entropy"]]) < 1e-12


def test_tile_records_closed_forms():
    """A constant tile: S = 256, E = 0; a zero tile with one value b > 0 at
    scale s (no softcap): m2 = s b log2 e, S = 1 + 255 2^-m2, E = -255 m2 2^-m2;
    X is the largest magnitude, whatever its sign."""
    x = np.zeros((2, 512))
    x[0, :256] = -1.5
    x[0, 256:] = 0.0
    x[1, 7] = 2.0
    x[1, 300] = -4.0
    rec = orc.tile_records(x, 0.0, 0.5)
    l2e = 1.0 / math.log(2.0)
    np.testing.assert_allclose(rec[0, 0], [-0.75 * l2e, 256.0, 0.0, 1.5], rtol=1e-15, atol=0)
    m2 = 1.0 * l2e
    np.testing.assert_allclose(rec[1, 0], [m2, 1 + 255 * 2 ** -m2, -255 * m2 * 2 ** -m2, 2.0],
                               rtol=1e-14)
    assert rec[1, 1, 3] == 4.0
    assert rec[1, 1, 0] == 0.0  # the largest zs of tile 1 is a zero logit


@pytest.mark.parametrize("T", [1.0, 1.5, 0.5])
def test_tile_records_at_temperature(T):
    """S_T merged over a row's tiles (weights 2^((m2_k - M) / T)) is the base-2
    sum of 2^(zs / T) (scipy's logsumexp); at T = 1 it is S; a constant tile
    gives 256 and a one-spike tile 1 + 255 2^(-m2 / T)."""
    from scipy.special import logsumexp
    rng = np.random.default_rng(5)
    x = rng.normal(0.0, 3.0, (3, 768))
    x[0, 256:512] = 0.0
    x[0, 300] = 4.0
    rec = orc.tile_records(x, 30.0, 0.5, temperature=T)
    assert rec.shape == (3, 3, 5)
    zs = 0.5 * 30.0 * np.tanh(x / 30.0) / math.log(2.0)
    for i in range(3):
        M = rec[i, :, 0].max()
        tot = np.sum(np.exp2((rec[i, :, 0] - M) / T) * rec[i, :, 4])
        ref = logsumexp(zs[i] * math.log(2.0) / T) / math.log(2.0)
        assert abs(M / T + math.log2(tot) - ref) < 1e-12
    if T == 1.0:
        np.testing.assert_allclose(rec[..., 4], rec[..., 1], rtol=1e-15)
    m2 = rec[0, 1, 0]
    assert abs(rec[0, 1, 4] - (1 + 255 * 2 ** (-m2 / T))) < 1e-12
    c = orc.tile_records(np.full((1, 256), -2.0), 0.0, 1.0, temperature=T)
    assert c[0, 0, 4] == 256.0
