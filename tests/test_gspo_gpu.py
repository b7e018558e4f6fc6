"""GPU parity of GSPO's three steps against the oracle (oracle.gspo_forward_backward
for GSPO, the row oracle for the losses computed beside it):

  1. headloss_forward_backward_ext with new_logprobs (metrics only);
  2. headloss_gspo_seam: sequence ratios, clipped objective, per-token
     coefficients;
  3. headloss_forward_backward_ext with token_coeff: the coefficient
     superposed on the label column with CE + z-loss (or with a CE of weight
     0, i.e. GSPO's gradient alone).

Old log-probs are the synthetic inputs' (the label log-prob by torch plus
noise) with a per-segment shift, so that some sequences sit beyond either clip
bound and others inside; no sequence ratio lies near a bound.  Segments
include an empty one, a one-row one and rows masked inside segments.
Tolerances are the library's: scalars 1e-3 (16-bit logits) / 1e-5 (fp32),
gradients within 2 ulp or the cancellation bound, masked rows exactly 0."""
import numpy as np
import pytest
import torch

import oracle as orc
import gradient_row_online_gb300 as pkg
from gradient_row_online_gb300 import headloss as hlb
from gradient_row_online_gb300 import workloads as W
from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hlb.load_library()


def _case(N, V, dtype, offs, softcap, scale, seed, shifts):
    wl = W.Workload("gspo", N, V, dtype, ("ce", "z", "grpo_stats"),
                    dict(ce=1.0, z=0.05, dist_ce=0.0, fkl=0.0, rkl=0.0, grpo=0.0, entropy=0.0,
                         grad_scale=1.0), mask_frac=0.15, softcap=softcap, logits_scale=scale,
                    seed=seed, adv_block=max(1, N // 4))
    inp = W.make_inputs(wl, "cuda")
    old = inp["old_logprobs"].clone()
    for i, (a, b) in enumerate(zip(offs[:-1], offs[1:])):
        old[a:b] += shifts[i % len(shifts)]
    inp["old_logprobs"] = old
    return wl, inp


def _pipeline(wl, inp, offs, eps, w_gspo, gs, w_ce=1.0, w_z=0.05):
    N, V = wl.N, wl.V
    dev = inp["logits"].device
    dcode = hlb.dtype_code(wl.dtype)
    h = pkg.HeadLoss(pkg.flags_of(("ce", "z")), hlb.make_weights(ce=w_ce, z=w_z, grad_scale=gs),
                     1.0, eps, wl.softcap, wl.logits_scale)
    lp = torch.empty(N, dtype=torch.float32, device=dev)
    s1 = torch.empty(16, dtype=torch.float32, device=dev)
    hlb.headloss_forward_backward_ext(h.h, inp["logits"], N, V, dcode, inp["labels"], None, None,
                                      None, None, s1, new_logprobs=lp)
    off_d = torch.as_tensor(offs, dtype=torch.int64, device=dev)
    coeff = torch.full((N,), float("nan"), dtype=torch.float32, device=dev)
    sg = torch.empty(4, dtype=torch.float32, device=dev)
    hlb.headloss_gspo_seam(lp, inp["old_logprobs"], inp["advantages"], inp["labels"], N, V, off_d,
                           len(offs) - 1, eps, w_gspo, gs, coeff, sg)
    g = torch.empty_like(inp["logits"])
    s2 = torch.empty(16, dtype=torch.float32, device=dev)
    hlb.headloss_forward_backward_ext(h.h, inp["logits"], N, V, dcode, inp["labels"], None, None,
                                      None, g, s2, token_coeff=coeff)
    torch.cuda.synchronize()
    assert h.device_error() == hlb.HEADLOSS_OK
    h.close()
    return (s2.double().cpu().numpy(), sg.double().cpu().numpy(), coeff.double().cpu().numpy(),
            g)


def _gspo_term_bound(dtype):
    """Weight of the GSPO term in the per-element cancellation bound
    (H.TAU[dtype] * gmag).  The term reaches the kernel through fp32 values
    by the call's types -- the forward's log-probs and the seam's coefficient
    -- so its relative precision is about 2^-20 whatever the logits' dtype;
    for 16-bit logits the library's own bound is already coarser."""
    return max(2.0, 2.0 ** -20 / H.TAU[dtype])


def _check(wl, inp, offs, eps, w_gspo, gs, got, w_ce=1.0, w_z=0.05):
    s2, sg, coeff, g = got
    tol = H.SCALAR_TOL[wl.dtype]
    x = H.host64(inp["logits"])
    lab = H.host_i64(inp["labels"])
    old = H.host64(inp["old_logprobs"])
    adv = H.host64(inp["advantages"])
    rs, rcoeff, rgrad = orc.gspo_forward_backward(x, lab, old, adv, np.asarray(offs), eps,
                                                  weight=w_gspo, grad_scale=gs,
                                                  softcap=wl.softcap, logits_scale=wl.logits_scale)
    # both branches of the clip are exercised, and no ratio is near a bound
    assert 0.0 < rs[2] < 1.0
    assert abs(sg[0] - rs[0]) <= tol * max(abs(rs[0]), 1e-3), (sg[0], rs[0])
    assert abs(sg[1] - rs[1]) <= tol * rs[1]
    assert sg[2] == np.float32(rs[2]) and sg[3] == rs[3]  # stored as fp32
    scale_c = np.abs(rcoeff).max()
    assert np.abs(coeff - rcoeff).max() <= tol * scale_c, (coeff[:8], rcoeff[:8])
    # the losses beside GSPO, and the superposed gradient
    cfg = orc.make_cfg(orc.CE | orc.Z, dict(ce=w_ce, z=w_z), softcap=wl.softcap,
                       logits_scale=wl.logits_scale, grad_scale=gs)
    rec, ref, gmag = orc.rows(cfg, x, lab, want_grad=True, want_gmag=True)
    ref_s = orc.reduce(cfg, rec)
    for slot in (1, 2):
        if w_ce == 0.0 and slot == 1:
            continue
        assert abs(s2[slot] - ref_s[slot]) <= tol * abs(ref_s[slot]), (slot, s2[slot], ref_s[slot])
    ref = ref + rgrad
    gmag = gmag + np.abs(rgrad) * _gspo_term_bound(wl.dtype)
    wl_chk = wl.replace(losses=("ce", "z"))
    H.check_grad(wl_chk, g, ref, gmag, rec)


SEGS = [0, 10, 10, 33, 34, 60, 96]
SHIFTS = [0.0, 0.35, -0.35, 0.02, 0.5, -0.6]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("softcap,scale", [(0.0, 1.0), (30.0, 0.5)])
def test_gspo_with_ce_and_z(dtype, softcap, scale):
    wl, inp = _case(96, 1031, dtype, SEGS, softcap, scale, seed=3, shifts=SHIFTS)
    got = _pipeline(wl, inp, SEGS, 0.2, 0.8, 1.3)
    _check(wl, inp, SEGS, 0.2, 0.8, 1.3, got)


def test_gspo_alone():
    wl, inp = _case(96, 4096, torch.bfloat16, SEGS, 0.0, 1.0, seed=4, shifts=SHIFTS)
    got = _pipeline(wl, inp, SEGS, 0.2, 1.0, 1.0, w_ce=0.0, w_z=0.0)
    _check(wl, inp, SEGS, 0.2, 1.0, 1.0, got, w_ce=0.0, w_z=0.0)


def test_gspo_sequences_of_1024_tokens():
    offs = [0, 1024, 2048]
    wl, inp = _case(2048, 32000, torch.bfloat16, offs, 0.0, 1.0, seed=5, shifts=[0.3, -0.3])
    got = _pipeline(wl, inp, offs, 0.2, 1.0, 1.0)
    s2, sg, coeff, g = got
    x = H.host64(inp["logits"])
    lab = H.host_i64(inp["labels"])
    rs, rcoeff, rg = orc.gspo_forward_backward(x, lab, H.host64(inp["old_logprobs"]),
                                               H.host64(inp["advantages"]), np.asarray(offs), 0.2)
    assert abs(sg[0] - rs[0]) <= 1e-3 * max(abs(rs[0]), 1e-3)
    assert np.abs(coeff - rcoeff).max() <= 1e-3 * np.abs(rcoeff).max()
    # the gradient on sampled rows
    rows = np.array([0, 1, 500, 1023, 1024, 1500, 2047])
    sel = torch.as_tensor(rows, device="cuda")
    cfg = orc.make_cfg(orc.CE | orc.Z, dict(ce=1.0, z=0.05))
    n_valid = orc.count_valid(lab, lab.shape[0])
    rec, ref, gmag = orc.rows(cfg, x[rows], lab[rows], n_valid_total=n_valid, want_grad=True,
                              want_gmag=True)
    H.check_grad(wl.replace(losses=("ce", "z")), g.index_select(0, sel), ref + rg[rows],
                 gmag + _gspo_term_bound(wl.dtype) * np.abs(rg[rows]), rec)


def test_seam_host_checks():
    x = torch.zeros(4, dtype=torch.float32, device="cuda")
    lab = torch.zeros(4, dtype=torch.int64, device="cuda")
    off = torch.tensor([0, 4], dtype=torch.int64, device="cuda")
    out = torch.empty(4, device="cuda")
    seam = hlb.headloss_gspo_seam
    for args, status in [((x, x, x, lab, 4, 8, off, 0, 0.2, 1.0, 1.0, x, out), hlb.HEADLOSS_ERR_ARG),
                         ((x, x, x, lab, 4, 8, off, 1, -0.1, 1.0, 1.0, x, out), hlb.HEADLOSS_ERR_ARG),
                         ((x, x, x, lab, 4, 8, None, 1, 0.2, 1.0, 1.0, x, out), hlb.HEADLOSS_ERR_ARG),
                         ((x, x, x, lab.data_ptr() + 4, 4, 8, off, 1, 0.2, 1.0, 1.0, x, out),
                          hlb.HEADLOSS_ERR_ALIGN)]:
        with pytest.raises(hlb.HeadlossError) as e:
            seam(*args)
        assert e.value.status == status
