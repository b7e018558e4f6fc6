"""GPU parity of headloss_forward_backward_ext's extras against the oracle:
per-row log p(label) and total loss, gradient accumulation into existing
values, and a batch split over calls that share one divisor."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as orc
import gradient_row_online_gb300 as pkg
from gradient_row_online_gb300 import headloss as hlb
from gradient_row_online_gb300 import workloads as W
from tests import _harness as H

pytestmark = pytest.mark.gpu

FULL_W = dict(ce=0.9, z=0.3, dist_ce=0.4, fkl=0.6, rkl=0.7, grpo=1.1, entropy=0.5,
              grad_scale=1.3)
RESIDENT, STREAM = hlb.HEADLOSS_KERNEL_RESIDENT, hlb.HEADLOSS_KERNEL_STREAM
WEIGHT_FIELD = dict(ce="ce", z="z", dist_ce="dist_ce", fkl="fkl", rkl="rkl", grpo="grpo",
                    entropy="entropy")

CASES = [
    # (losses, dtype, softcap, plan)
    (("ce", "z", "grpo", "grpo_stats", "entropy"), torch.bfloat16, 0.0, None),
    (("ce", "z", "fkl", "grpo", "grpo_stats", "entropy"), torch.bfloat16, 30.0,
     dict(kernel=STREAM, stages=3, threads=256, chunk_words=1)),
    (("ce", "dist_ce", "fkl", "rkl"), torch.bfloat16, 0.0,
     dict(kernel=RESIDENT, cluster=2, stages=1, threads=256)),
    (("ce", "z", "entropy"), torch.float16, 15.0, None),
    (("ce", "grpo", "grpo_stats", "dist_ce", "rkl", "entropy"), torch.float32, 20.0, None),
    (("ce", "z", "fkl", "rkl", "entropy"), torch.float16, 30.0,
     dict(kernel=STREAM, stages=2, threads=512, chunk_words=1)),
    # fp32 without teacher, softcap or entropy: the double-float kernel
    (("ce", "z", "grpo", "grpo_stats"), torch.float32, 0.0, None),
    (("ce", "grpo"), torch.float32, 0.0, dict(kernel=RESIDENT, cluster=2, stages=1, threads=256)),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hlb.load_library()


def small(losses, dtype, softcap, N=36, V=4104, **kw):
    return W.Workload("ext", N, V, dtype, tuple(losses), dict(FULL_W), sigma=3.0, mask_frac=0.2,
                      teacher_noise=1.0, temperature=1.7, clip_eps=0.2, softcap=softcap,
                      logits_scale=0.6, **kw)


def handle(wl, plan):
    h = pkg.headloss_for(wl)
    if plan is not None:
        h.force_plan(**plan)
    return h


def expected_rows(wl, rec):
    """Per-row log p(label) and weighted total loss from the oracle's records."""
    lp = rec[:, orc.RF["logprob"]] if "grpo" in wl.losses or "grpo_stats" in wl.losses \
        else -rec[:, orc.RF["ce"]]
    tot = np.zeros(rec.shape[0])
    for name, field in WEIGHT_FIELD.items():
        if name in wl.losses:
            tot += np.float32(wl.weights[name]) * rec[:, orc.RF[field]]
    return lp, tot


def close_rows(got, ref, valid, tol):
    scale = max(float(np.abs(ref[valid]).mean()), 1e-30)
    err = np.abs(got[valid] - ref[valid]) / np.maximum(np.abs(ref[valid]), scale)
    assert err.max() <= tol, err.max()
    assert np.all(got[~valid] == 0.0)


@pytest.mark.parametrize("losses,dtype,softcap,plan", CASES)
def test_per_token_outputs(losses, dtype, softcap, plan):
    wl = small(losses, dtype, softcap)
    inp = W.make_inputs(wl, "cuda")
    h = handle(wl, plan)
    lp = torch.full((wl.N,), float("nan"), device="cuda")
    rl = torch.full((wl.N,), float("nan"), device="cuda")
    g = torch.empty_like(inp["logits"])
    out = h(inp["logits"], inp["labels"], inp["teacher"], inp["old_logprobs"],
            inp["advantages"], g, new_logprobs=lp, row_loss=rl)
    torch.cuda.synchronize()
    assert h.device_error() == hlb.HEADLOSS_OK
    cfg, rec, ref, gmag = H.oracle_rows(wl, inp)
    valid = rec[:, orc.RF["valid"]] > 0
    lp_ref, rl_ref = expected_rows(wl, rec)
    tol = H.SCALAR_TOL[dtype]
    close_rows(lp.double().cpu().numpy(), lp_ref, valid, tol)
    close_rows(rl.double().cpu().numpy(), rl_ref, valid, tol)
    # the mean of the per-row totals is the TOTAL slot; the gradient is unchanged
    o = out.double().cpu().numpy()
    n = valid.sum()
    assert abs(rl.double().cpu().numpy().sum() / n - o[0]) <= tol * max(1.0, abs(o[0]))
    H.check_grad(wl, g, ref, gmag, rec)


@pytest.mark.parametrize("losses,dtype,softcap,plan", CASES)
def test_accumulate_adds_to_existing_gradient(losses, dtype, softcap, plan):
    wl = small(losses, dtype, softcap)
    inp = W.make_inputs(wl, "cuda")
    h = handle(wl, plan)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    g0 = (torch.randn(inp["logits"].shape, generator=gen, device="cuda") * 1e-4).to(dtype)
    g = g0.clone()
    h(inp["logits"], inp["labels"], inp["teacher"], inp["old_logprobs"], inp["advantages"], g,
      accumulate=True)
    torch.cuda.synchronize()
    assert h.device_error() == hlb.HEADLOSS_OK
    cfg, rec, ref, gmag = H.oracle_rows(wl, inp)
    valid = rec[:, orc.RF["valid"]] > 0
    g0h = g0.double().cpu().numpy()
    # masked rows keep their values bit for bit
    assert torch.equal(g[torch.from_numpy(~valid).cuda()], g0[torch.from_numpy(~valid).cuda()])
    # valid rows: the existing value plus the oracle gradient, one rounding
    sel = torch.from_numpy(np.nonzero(valid)[0]).cuda()
    H.check_grad(wl, g.index_select(0, sel), (g0h + ref)[valid],
                 (gmag + np.abs(g0h))[valid], rec[valid])


@pytest.mark.parametrize("losses,dtype,softcap,plan", CASES)
def test_split_batch_with_shared_divisor(losses, dtype, softcap, plan):
    wl = small(losses, dtype, softcap, N=40)
    inp = W.make_inputs(wl, "cuda")
    cfg, rec, ref, gmag = H.oracle_rows(wl, inp)   # normalised by the whole batch's count
    whole = orc.reduce(cfg, rec)
    n_total = float(whole[14])
    h = handle(wl, plan)
    parts = [slice(0, 13), slice(13, 40)]
    g = torch.empty_like(inp["logits"])
    sums = np.zeros(16)
    for sl in parts:
        pick = lambda t: None if t is None else t[sl].contiguous()
        gp = torch.empty_like(inp["logits"][sl])
        out = h(pick(inp["logits"]), pick(inp["labels"]), pick(inp["teacher"]),
                pick(inp["old_logprobs"]), pick(inp["advantages"]), gp, divisor=n_total)
        torch.cuda.synchronize()
        assert h.device_error() == hlb.HEADLOSS_OK
        g[sl] = gp
        o = out.double().cpu().numpy()
        sums += o
        # metric slots stay means over the call's own rows
        own = orc.reduce(cfg, rec[sl])
        assert o[14] == own[14]
        if "grpo_stats" in wl.losses and own[14] > 0:
            for slot in (7, 8, 10, 11):
                assert abs(o[slot] - own[slot]) <= H.SCALAR_TOL[dtype] * max(1.0, abs(own[slot]))
    # the split's loss slots add up to the whole batch's, and so do the gradients
    tol = H.SCALAR_TOL[dtype]
    for slot in (0, 1, 2, 3, 4, 5, 6, 13):
        assert abs(sums[slot] - whole[slot]) <= tol * max(1.0, abs(whole[slot])), (slot, sums, whole)
    H.check_grad(wl, g, ref, gmag, rec)


def test_ext_argument_errors():
    wl = small(("ce", "z"), torch.bfloat16, 0.0, N=4, V=64)
    inp = W.make_inputs(wl, "cuda")
    h = pkg.headloss_for(wl)
    x = inp["logits"]
    with pytest.raises(hlb.HeadlossError) as e:
        h(x, inp["labels"], grad_out=None, accumulate=True)
    assert e.value.status == hlb.HEADLOSS_ERR_ARG
    with pytest.raises(hlb.HeadlossError) as e:
        h(x, inp["labels"], grad_out=x, accumulate=True)  # accumulating into the logits
    assert e.value.status == hlb.HEADLOSS_ERR_ARG
    with pytest.raises(hlb.HeadlossError) as e:
        h(x, inp["labels"], grad_out=torch.empty_like(x), divisor=-1.0)
    assert e.value.status == hlb.HEADLOSS_ERR_ARG
    # a per-row output whose address is not 4-byte aligned
    lib = hlb.load_library()
    buf = torch.empty(wl.N + 1, device="cuda")
    ext = hlb.headloss_call_ext(buf.data_ptr() + 1, None, 0, 0.0)
    out = torch.empty(16, device="cuda")
    st = lib.headloss_forward_backward_ext(h.h, x.data_ptr(), wl.N, wl.V, hlb.dtype_code(x.dtype),
                                           inp["labels"].data_ptr(), None, None, None, None,
                                           out.data_ptr(), ctypes.byref(ext), None)
    assert st == hlb.HEADLOSS_ERR_ALIGN
    # new log-probs need labels
    ext = hlb.headloss_call_ext(buf.data_ptr(), None, 0, 0.0)
    h2 = pkg.headloss_for(small(("z",), torch.bfloat16, 0.0, N=4, V=64))
    st = lib.headloss_forward_backward_ext(h2.h, x.data_ptr(), wl.N, wl.V,
                                           hlb.dtype_code(x.dtype), None, None, None, None, None,
                                           out.data_ptr(), ctypes.byref(ext), None)
    assert st == hlb.HEADLOSS_ERR_MISSING_INPUT
