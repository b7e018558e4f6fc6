"""GPU parity of the fused LM head's single-pass loss with the call's extras
(headloss_forward_backward_rowstats with a headloss_call_ext): per-row
log p(label) and total loss, accumulation into an existing gradient, a batch
split over calls that share one divisor, and GSPO's three steps (forward with
new log-probs, the segment seam, backward with the per-token coefficient) on
the GEMM's row records, against the oracle.

As in the other single-pass tests, the logits come out of the LM-head GEMM
with an identity weight (bit for bit the seeded rows), so its epilogue's
per-tile records describe the very values the oracle sees.  Tolerances are the
library's: scalars 1e-3, gradients 2 ulp of bf16 or the cancellation bound,
masked rows exactly +0 (or their old value when accumulating)."""
import numpy as np
import pytest
import torch

import oracle as orc
import gradient_row_online_gb300 as pkg
from gradient_row_online_gb300 import headloss as hlb
from gradient_row_online_gb300 import workloads as W
from tests import _harness as H
from tests import test_call_ext_gpu as CX
from tests import test_gspo_gpu as GS
from tests import test_rowstats_gpu as RS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hlb.load_library()


def _gemm_rows(x, softcap, scale, temperature=None):
    """RS._gemm on the rows padded with zeros to the GEMM's 128-row multiple,
    cut back to the batch's own rows."""
    N = x.shape[0]
    xp = torch.zeros(((N + 127) // 128 * 128, x.shape[1]), dtype=x.dtype, device=x.device)
    xp[:N] = x
    cut = lambda t: None if t is None else t[:N].contiguous()
    return tuple(cut(t) for t in RS._gemm(xp, softcap, scale, temperature))


def _records(wl, x, teacher):
    """The student's logits and records (with its sums at the temperature
    when a teacher is present and T != 1) and the teacher's."""
    T = float(np.float32(wl.temperature))
    logits, rs, rsT = _gemm_rows(x, wl.softcap, wl.logits_scale,
                                 T if teacher is not None and T != 1.0 else None)
    tl, trs = None, None
    if teacher is not None:
        tl, trs, _ = _gemm_rows(teacher, 0.0, 1.0 / T)
    return logits, rs, rsT, tl, trs


def _call(h, wl, rows, logits, rs, rsT, tl, trs, inp, g, **ext):
    """One rowstats call over rows `rows` (a slice) of the records and inputs."""
    pick = lambda t: None if t is None else t[rows].contiguous()
    x = pick(logits)
    out = torch.full((16,), float("nan"), device="cuda")
    hlb.headloss_forward_backward_rowstats(
        h.h, x, x.shape[0], wl.V, hlb.HEADLOSS_BF16, pick(inp["labels"]),
        pick(inp["old_logprobs"]), pick(inp["advantages"]), pick(rs), g, out,
        teacher=pick(tl), row_stats_t=pick(rsT), teacher_stats=pick(trs), **ext)
    torch.cuda.synchronize()
    assert h.device_error() == hlb.HEADLOSS_OK
    return out.double().cpu().numpy()


EXT_SETS = [("ce", "z"), ("ce", "z", "grpo", "grpo_stats", "entropy"),
            ("ce", "z", "fkl", "grpo", "grpo_stats", "entropy"), ("ce", "dist_ce", "fkl")]
CAPS = [(0.0, 1.0), (30.0, 0.6)]


def _small(losses, softcap, scale, N=36, V=4096):
    return W.Workload("ext", N, V, torch.bfloat16, tuple(losses), dict(CX.FULL_W, rkl=0.0),
                      sigma=3.0, mask_frac=0.2, teacher_noise=1.0, temperature=1.7,
                      clip_eps=0.2, softcap=softcap, logits_scale=scale, seed=len(losses))


@pytest.mark.parametrize("softcap,scale", CAPS)
@pytest.mark.parametrize("losses", EXT_SETS)
def test_rowstats_per_token_outputs(losses, softcap, scale):
    wl = _small(losses, softcap, scale)
    inp = W.make_inputs(wl, "cuda")
    recs = _records(wl, inp["logits"], inp["teacher"])
    h = pkg.headloss_for(wl)
    lp = torch.full((wl.N,), float("nan"), device="cuda")
    rl = torch.full((wl.N,), float("nan"), device="cuda")
    g = torch.empty_like(inp["logits"])
    o = _call(h, wl, slice(None), *recs, inp, g, new_logprobs=lp, row_loss=rl)
    h.close()
    cfg, rec, ref, gmag = H.oracle_rows(wl, inp)
    valid = rec[:, orc.RF["valid"]] > 0
    lp_ref, rl_ref = CX.expected_rows(wl, rec)
    tol = H.SCALAR_TOL[wl.dtype]
    CX.close_rows(lp.double().cpu().numpy(), lp_ref, valid, tol)
    CX.close_rows(rl.double().cpu().numpy(), rl_ref, valid, tol)
    assert abs(rl.double().cpu().numpy().sum() / valid.sum() - o[0]) <= tol * max(1.0, abs(o[0]))
    H.check_scalars(wl, o, cfg, rec)
    H.check_grad(wl, g, ref, gmag, rec)


@pytest.mark.parametrize("losses", [EXT_SETS[1], EXT_SETS[2]])
def test_rowstats_accumulates_into_existing_gradient(losses):
    wl = _small(losses, 30.0, 0.6)
    inp = W.make_inputs(wl, "cuda")
    recs = _records(wl, inp["logits"], inp["teacher"])
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    g0 = (torch.randn(inp["logits"].shape, generator=gen, device="cuda") * 1e-4).to(wl.dtype)
    g = g0.clone()
    h = pkg.headloss_for(wl)
    _call(h, wl, slice(None), *recs, inp, g, accumulate=True)
    h.close()
    cfg, rec, ref, gmag = H.oracle_rows(wl, inp)
    valid = rec[:, orc.RF["valid"]] > 0
    inval = torch.from_numpy(~valid).cuda()
    assert torch.equal(g[inval], g0[inval])  # masked rows keep their values bit for bit
    sel = torch.from_numpy(np.nonzero(valid)[0]).cuda()
    g0h = g0.double().cpu().numpy()
    H.check_grad(wl, g.index_select(0, sel), (g0h + ref)[valid], (gmag + np.abs(g0h))[valid],
                 rec[valid])


@pytest.mark.parametrize("losses", [EXT_SETS[1], EXT_SETS[3]])
def test_rowstats_split_batch_with_shared_divisor(losses):
    wl = _small(losses, 0.0, 1.0, N=40)
    inp = W.make_inputs(wl, "cuda")
    recs = _records(wl, inp["logits"], inp["teacher"])
    cfg, rec, ref, gmag = H.oracle_rows(wl, inp)
    whole = orc.reduce(cfg, rec)
    n_total = float(whole[14])
    h = pkg.headloss_for(wl)
    g = torch.empty_like(inp["logits"])
    sums = np.zeros(16)
    tol = H.SCALAR_TOL[wl.dtype]
    for sl in (slice(0, 13), slice(13, 40)):
        gp = torch.empty_like(inp["logits"][sl])
        o = _call(h, wl, sl, *recs, inp, gp, divisor=n_total)
        g[sl] = gp
        sums += o
        own = orc.reduce(cfg, rec[sl])
        assert o[14] == own[14]  # metric slots stay over the call's own rows
    h.close()
    for slot in (0, 1, 2, 3, 4, 5, 6, 13):
        assert abs(sums[slot] - whole[slot]) <= tol * max(1.0, abs(whole[slot])), (slot, sums,
                                                                                   whole)
    H.check_grad(wl, g, ref, gmag, rec)


def _gspo_rowstats(wl, inp, offs, eps, w_gspo, gs, w_ce=1.0, w_z=0.05, inplace=False):
    """GSPO's three steps through the single pass on the GEMM's records."""
    N = wl.N
    logits, rs, rsT, tl, trs = _records(wl, inp["logits"], None)
    h = pkg.HeadLoss(pkg.flags_of(("ce", "z")), hlb.make_weights(ce=w_ce, z=w_z, grad_scale=gs),
                     1.0, eps, wl.softcap, wl.logits_scale)
    lp = torch.empty(N, dtype=torch.float32, device="cuda")
    _call(h, wl, slice(None), logits, rs, rsT, tl, trs, inp, None, new_logprobs=lp)
    off_d = torch.as_tensor(offs, dtype=torch.int64, device="cuda")
    coeff = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    sg = torch.empty(4, dtype=torch.float32, device="cuda")
    hlb.headloss_gspo_seam(lp, inp["old_logprobs"], inp["advantages"], inp["labels"], N, wl.V,
                           off_d, len(offs) - 1, eps, w_gspo, gs, coeff, sg)
    g = logits if inplace else torch.empty_like(logits)
    s2 = _call(h, wl, slice(None), logits, rs, rsT, tl, trs, inp, g, token_coeff=coeff)
    h.close()
    return s2, sg.double().cpu().numpy(), coeff.double().cpu().numpy(), g


@pytest.mark.parametrize("inplace", [False, True])
@pytest.mark.parametrize("softcap,scale", [(0.0, 1.0), (30.0, 0.5)])
def test_rowstats_gspo_with_ce_and_z(softcap, scale, inplace):
    wl, inp = GS._case(96, 4096, torch.bfloat16, GS.SEGS, softcap, scale, seed=3,
                       shifts=GS.SHIFTS)
    ref_inp = dict(inp, logits=inp["logits"].clone())
    got = _gspo_rowstats(wl, inp, GS.SEGS, 0.2, 0.8, 1.3, inplace=inplace)
    GS._check(wl, ref_inp, GS.SEGS, 0.2, 0.8, 1.3, got)


def test_rowstats_gspo_alone():
    wl, inp = GS._case(96, 4096, torch.bfloat16, GS.SEGS, 0.0, 1.0, seed=4, shifts=GS.SHIFTS)
    got = _gspo_rowstats(wl, inp, GS.SEGS, 0.2, 1.0, 1.0, w_ce=0.0, w_z=0.0)
    GS._check(wl, inp, GS.SEGS, 0.2, 1.0, 1.0, got, w_ce=0.0, w_z=0.0)


def test_rowstats_ext_argument_errors():
    wl = _small(("ce", "z"), 0.0, 1.0, N=4, V=512)
    inp = W.make_inputs(wl, "cuda")
    logits, rs, rsT, tl, trs = _records(wl, inp["logits"], None)
    h = pkg.headloss_for(wl)
    out = torch.empty(16, device="cuda")
    fb = hlb.headloss_forward_backward_rowstats
    base = (h.h, logits, wl.N, wl.V, hlb.HEADLOSS_BF16, inp["labels"], None, None, rs)
    buf = torch.empty(wl.N + 1, device="cuda")
    cases = [
        (dict(grad_out=None, accumulate=True), hlb.HEADLOSS_ERR_ARG),
        (dict(grad_out=logits, accumulate=True), hlb.HEADLOSS_ERR_ARG),  # into the logits
        (dict(grad_out=torch.empty_like(logits), divisor=-1.0), hlb.HEADLOSS_ERR_ARG),
        (dict(grad_out=torch.empty_like(logits), new_logprobs=buf.data_ptr() + 1),
         hlb.HEADLOSS_ERR_ALIGN),
    ]
    for kw, status in cases:
        g = kw.pop("grad_out")
        with pytest.raises(hlb.HeadlossError) as e:
            fb(*base, g, out, **kw)
        assert e.value.status == status, kw
    # per-row log-probs and the per-token coefficient need labels
    h2 = pkg.headloss_for(_small(("z",), 0.0, 1.0, N=4, V=512))
    for kw in (dict(new_logprobs=buf), dict(token_coeff=buf)):
        with pytest.raises(hlb.HeadlossError) as e:
            fb(h2.h, logits, wl.N, wl.V, hlb.HEADLOSS_BF16, None, None, None, rs,
               torch.empty_like(logits), out, **kw)
        assert e.value.status == hlb.HEADLOSS_ERR_MISSING_INPUT, kw
    h.close()
    h2.close()
