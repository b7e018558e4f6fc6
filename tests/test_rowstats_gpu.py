"""GPU parity of the fused LM head's single-pass loss: the GEMM epilogue's
per-tile row statistics (headloss_lmhead_logits_rowstats; with a teacher, the
student's sums at the temperature and the teacher GEMM's records) consumed by
the loss's gradient pass alone (headloss_forward_backward_rowstats), against
the fp64 row oracle on the same logits.

The logits are seeded synthetic rows (N(0, 3^2), bf16), fed to the GEMM as
its hidden states with an identity weight: every logit is then a product
with 1.0 and a sum of one nonzero term, so the GEMM reproduces the seeded
logits exactly (checked bit for bit) while its epilogue computes their row
statistics, and the oracle sees the very same values.  Tolerances are the
library's (harness): scalars 1e-3 relative, gradient 2 ulp of bf16 or the
cancellation bound, masked rows exactly +0."""
import numpy as np
import pytest
import torch

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


def _gemm(x, softcap, scale, temperature=None):
    """Identity-weight GEMM: the logits reproduced bit for bit, with their
    per-tile records (and sums at the temperature)."""
    N, V = x.shape
    eye = torch.eye(V, dtype=torch.bfloat16, device="cuda")
    logits = torch.empty_like(x)
    rs = torch.full((N, V // 256, 4), float("nan"), device="cuda")
    rsT = None if temperature is None else torch.full((N, V // 256), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hlb.headloss_lmhead_logits_rowstats(x, eye, N, V, V, softcap, scale, logits, rs, err,
                                        temperature=temperature or 1.0, row_stats_t=rsT)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(logits.view(torch.int16), x.view(torch.int16))
    return logits, rs, rsT


def _run(wl, inp, inplace=False):
    N, V = wl.N, wl.V
    teach = inp.get("teacher") is not None
    T = float(np.float32(wl.temperature))
    logits, rs, rsT = _gemm(inp["logits"], wl.softcap, wl.logits_scale,
                            T if teach and T != 1.0 else None)
    teacher, trs = None, None
    if teach:
        teacher, trs, _ = _gemm(inp["teacher"], 0.0, 1.0 / T)
    h = pkg.headloss_for(wl)
    g = logits if inplace else torch.empty_like(logits)
    out = torch.full((16,), float("nan"), device="cuda")
    ref_x = logits.clone() if inplace else logits
    hlb.headloss_forward_backward_rowstats(h.h, logits, N, V, hlb.HEADLOSS_BF16, inp["labels"],
                                           inp["old_logprobs"], inp["advantages"], rs, g, out,
                                           teacher=teacher, row_stats_t=rsT,
                                           teacher_stats=trs)
    torch.cuda.synchronize()
    assert h.device_error() == hlb.HEADLOSS_OK
    h.close()
    return out.double().cpu().numpy(), g, dict(inp, logits=ref_x)


SETS = [("ce", "z"), ("grpo", "grpo_stats", "z", "entropy"), ("ce", "z", "grpo", "grpo_stats",
                                                                "entropy")]
W_ALL = dict(ce=0.9, z=0.3, dist_ce=0.0, fkl=0.0, rkl=0.0, grpo=1.1, entropy=0.5, grad_scale=1.3)


@pytest.mark.parametrize("softcap,scale", [(0.0, 1.0), (30.0, 0.5), (3.0, 0.7)])
@pytest.mark.parametrize("losses", SETS)
def test_rowstats_loss_against_oracle(losses, softcap, scale):
    wl = W.Workload("rowstats", 256, 4096, torch.bfloat16, losses, dict(W_ALL), softcap=softcap,
                    logits_scale=scale, mask_frac=0.15, seed=len(losses))
    inp = W.make_inputs(wl, "cuda")
    got, g, ref_inp = _run(wl, inp)
    cfg, rec, ref, gmag = H.oracle_rows(wl, ref_inp)
    H.check_scalars(wl, got, cfg, rec)
    H.check_grad(wl, g, ref, gmag, rec)


def test_rowstats_in_place_and_wider_rows():
    wl = W.Workload("rowstats", 128, 32000, torch.bfloat16, SETS[2], dict(W_ALL), softcap=30.0,
                    logits_scale=0.5, mask_frac=0.1, seed=7)
    inp = W.make_inputs(wl, "cuda")
    got, g, ref_inp = _run(wl, inp, inplace=True)
    cfg, rec, ref, gmag = H.oracle_rows(wl, ref_inp)
    H.check_scalars(wl, got, cfg, rec)
    H.check_grad(wl, g, ref, gmag, rec)


W_DIST = dict(W_ALL, dist_ce=0.4, fkl=0.6)
TEACH_SETS = [("ce", "z", "fkl", "grpo", "grpo_stats", "entropy"), ("dist_ce", "fkl"),
              ("ce", "dist_ce", "fkl", "entropy")]


@pytest.mark.parametrize("T", [1.0, 1.5, 2.0])
@pytest.mark.parametrize("softcap,scale", [(0.0, 1.0), (30.0, 0.5), (3.0, 0.7)])
@pytest.mark.parametrize("losses", TEACH_SETS)
def test_rowstats_with_teacher_against_oracle(losses, softcap, scale, T):
    wl = W.Workload("rowstats", 256, 4096, torch.bfloat16, losses, dict(W_DIST), softcap=softcap,
                    logits_scale=scale, temperature=T, teacher_noise=1.0, mask_frac=0.15,
                    seed=len(losses) + int(2 * T))
    inp = W.make_inputs(wl, "cuda")
    got, g, ref_inp = _run(wl, inp)
    cfg, rec, ref, gmag = H.oracle_rows(wl, ref_inp)
    H.check_scalars(wl, got, cfg, rec)
    H.check_grad(wl, g, ref, gmag, rec)


@pytest.mark.parametrize("losses", [("dist_ce", "fkl", "entropy"), ("z", "entropy")])
def test_rowstats_without_labels(losses):
    """No labels (every row valid): the losses that need none, with and without a
    teacher."""
    wl = W.Workload("rowstats", 256, 4096, torch.bfloat16, losses, dict(W_DIST), softcap=30.0,
                    logits_scale=0.5, temperature=1.5, teacher_noise=1.0, seed=3)
    inp = dict(W.make_inputs(wl, "cuda"), labels=None)
    got, g, ref_inp = _run(wl, inp)
    cfg, rec, ref, gmag = H.oracle_rows(wl, ref_inp)
    assert got[14] == 256
    H.check_scalars(wl, got, cfg, rec)
    H.check_grad(wl, g, ref, gmag, rec)


def _oracle_stats(inp, wl):
    """Per-tile records from the oracle's plain definition (for rows too wide
    for an identity-weight GEMM), as the kernel takes them."""
    import oracle as orc
    T = float(np.float32(wl.temperature))
    st = orc.tile_records(inp["logits"].float().cpu().numpy(), wl.softcap, wl.logits_scale,
                          temperature=T)
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    if inp["teacher"] is None:
        return f(st[..., :4]), f(st[..., 4]), None
    tt = orc.tile_records(inp["teacher"].float().cpu().numpy(), 0.0, 1.0 / T)
    return f(st[..., :4]), f(st[..., 4]), f(tt)


def test_rowstats_with_teacher_wide_rows_in_place_and_metrics_only():
    """The all-in label-and-teacher set at 152064 columns (38 chunks of 128
    words per unit: beyond the 32 whose softcap tiers are recorded), records
    from the oracle's definition, in place; then without a gradient, the
    scalars alone (the pass still runs for the distillation values)."""
    wl = W.Workload("rowstats", 48, 152064, torch.bfloat16, TEACH_SETS[0], dict(W_DIST),
                    softcap=30.0, logits_scale=0.5, temperature=1.5, teacher_noise=1.0,
                    mask_frac=0.1, seed=11)
    inp = W.make_inputs(wl, "cuda")
    rs, rsT, trs = _oracle_stats(inp, wl)
    ref_inp = dict(inp, logits=inp["logits"].clone())
    for grad in (True, False):
        h = pkg.headloss_for(wl)
        out = torch.full((16,), float("nan"), device="cuda")
        g = inp["logits"] if grad else None
        hlb.headloss_forward_backward_rowstats(h.h, inp["logits"], 48, 152064,
                                               hlb.HEADLOSS_BF16, inp["labels"],
                                               inp["old_logprobs"], inp["advantages"], rs, g,
                                               out, teacher=inp["teacher"], row_stats_t=rsT,
                                               teacher_stats=trs)
        torch.cuda.synchronize()
        assert h.device_error() == hlb.HEADLOSS_OK
        h.close()
        cfg, rec, ref, gmag = H.oracle_rows(wl, ref_inp, want_grad=grad, want_gmag=grad)
        H.check_scalars(wl, out.double().cpu().numpy(), cfg, rec)
        if grad:
            H.check_grad(wl, g, ref, gmag, rec)
            inp["logits"].copy_(ref_inp["logits"])  # the logits back for the second call


def test_rowstats_rejects_what_it_does_not_cover():
    wl = W.Workload("rowstats", 128, 256, torch.bfloat16, ("ce", "fkl"),
                    dict(W_ALL, fkl=0.5), teacher_noise=1.0, temperature=2.0)
    inp = W.make_inputs(wl, "cuda")
    rs = torch.zeros(128, 1, 4, device="cuda")
    rsT = torch.ones(128, 1, device="cuda")
    out = torch.empty(16, device="cuda")
    h = pkg.headloss_for(wl)
    fb = hlb.headloss_forward_backward_rowstats
    args = (h.h, inp["logits"], 128, 256, hlb.HEADLOSS_BF16, inp["labels"], None, None, rs, None,
            out)
    with pytest.raises(hlb.HeadlossError) as e:  # a teacher loss without the teacher
        fb(*args)
    assert e.value.status == hlb.HEADLOSS_ERR_MISSING_INPUT
    with pytest.raises(hlb.HeadlossError) as e:  # ... without the teacher's records
        fb(*args, teacher=inp["teacher"], row_stats_t=rsT)
    assert e.value.status == hlb.HEADLOSS_ERR_MISSING_INPUT
    with pytest.raises(hlb.HeadlossError) as e:  # ... at T = 2 without the sums at T
        fb(*args, teacher=inp["teacher"], teacher_stats=rs)
    assert e.value.status == hlb.HEADLOSS_ERR_MISSING_INPUT
    with pytest.raises(hlb.HeadlossError) as e:  # misaligned teacher records
        fb(*args, teacher=inp["teacher"], teacher_stats=rs.data_ptr() + 8, row_stats_t=rsT)
    assert e.value.status == hlb.HEADLOSS_ERR_ALIGN
    h.close()
    wr = wl.replace(losses=("ce", "rkl"))
    hr = pkg.headloss_for(wr)
    with pytest.raises(hlb.HeadlossError) as e:  # reverse KL: a cross sum before the pass
        fb(hr.h, inp["logits"], 128, 256, hlb.HEADLOSS_BF16, inp["labels"], None, None, rs,
           None, out, teacher=inp["teacher"], teacher_stats=rs, row_stats_t=rsT)
    assert e.value.status == hlb.HEADLOSS_ERR_ARG
    hr.close()
    wl2 = wl.replace(losses=("ce",), V=300, teacher_noise=None)
    h2 = pkg.headloss_for(wl2)
    x = torch.zeros(128, 300, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(hlb.HeadlossError) as e:  # V not a multiple of 256
        fb(h2.h, x, 128, 300, hlb.HEADLOSS_BF16, inp["labels"], None, None, rs, None, out)
    assert e.value.status == hlb.HEADLOSS_ERR_ARG
    with pytest.raises(hlb.HeadlossError) as e:  # fp16 logits
        fb(h2.h, x, 128, 256, hlb.HEADLOSS_FP16, inp["labels"], None, None, rs, None, out)
    assert e.value.status == hlb.HEADLOSS_ERR_DTYPE
    with pytest.raises(hlb.HeadlossError) as e:  # misaligned statistics
        fb(h2.h, x, 128, 256, hlb.HEADLOSS_BF16, inp["labels"], None, None, rs.data_ptr() + 8,
           None, out)
    assert e.value.status == hlb.HEADLOSS_ERR_ALIGN
    h2.close()


@pytest.mark.parametrize("softcap,scale", [(0.0, 1.0), (30.0, 0.5), (3.0, 0.7)])
def test_gemm_tile_records_against_oracle(softcap, scale):
    """The GEMM epilogue's per-tile records (m2, S, E, X) against the oracle's
    plain definition on the same (seeded, identity-reproduced) logits: X exactly
    (the largest |bf16 logit|), the rest within fp32 rounding of 256-term sums
    of exponentials (relative 2e-5; E against 2e-5 (S + |E|): all its terms
    share one sign)."""
    import oracle as orc
    N, V = 256, 4096
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    x = (torch.randn(N, V, generator=g, device="cuda") * 3.0).to(torch.bfloat16)
    x[5, 100:356] = 0.0  # a constant tile
    x[9, 1000] = 200.0   # a saturating logit
    eye = torch.eye(V, dtype=torch.bfloat16, device="cuda")
    logits = torch.empty_like(x)
    rs = torch.full((N, V // 256, 4), float("nan"), device="cuda")
    rsT = torch.full((N, V // 256), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hlb.headloss_lmhead_logits_rowstats(x, eye, N, V, V, softcap, scale, logits, rs, err,
                                        temperature=1.5, row_stats_t=rsT)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(logits.view(torch.int16), x.view(torch.int16))
    got = rs.double().cpu().numpy()
    ref = orc.tile_records(x.float().cpu().numpy(), softcap, scale, temperature=1.5)
    np.testing.assert_allclose(rsT.double().cpu().numpy(), ref[..., 4], rtol=2e-5, atol=0)
    np.testing.assert_array_equal(got[..., 3], ref[..., 3])
    np.testing.assert_allclose(got[..., 0], ref[..., 0], rtol=2e-5, atol=2e-5)
    np.testing.assert_allclose(got[..., 1], ref[..., 1], rtol=2e-5, atol=0)
    assert np.all(np.abs(got[..., 2] - ref[..., 2]) <= 2e-5 * (ref[..., 1] + np.abs(ref[..., 2])))


@pytest.mark.parametrize("N,V", [(1, 256), (3, 512), (130, 256), (5, 4352)])
@pytest.mark.parametrize("losses", [("ce", "z", "grpo", "grpo_stats", "entropy"), TEACH_SETS[0]])
def test_rowstats_small_and_ragged_batches(N, V, losses):
    """Batches below one CTA's eight warps, a ragged count of units, the
    smallest vocabulary (one tile, a partial chunk per unit), with and without
    a teacher; records from the oracle's definition (the GEMM takes 128-row
    multiples only)."""
    wl = W.Workload("rowstats", N, V, torch.bfloat16, losses, dict(W_DIST), softcap=30.0,
                    logits_scale=0.5, temperature=1.5, teacher_noise=1.0, mask_frac=0.2,
                    seed=N + V)
    inp = W.make_inputs(wl, "cuda")
    rs, rsT, trs = _oracle_stats(inp, wl)
    h = pkg.headloss_for(wl)
    g = torch.empty_like(inp["logits"])
    out = torch.full((16,), float("nan"), device="cuda")
    teach = "fkl" in losses
    hlb.headloss_forward_backward_rowstats(h.h, inp["logits"], N, V, hlb.HEADLOSS_BF16,
                                           inp["labels"], inp["old_logprobs"],
                                           inp["advantages"], rs, g, out,
                                           teacher=inp["teacher"] if teach else None,
                                           row_stats_t=rsT if teach else None,
                                           teacher_stats=trs if teach else None)
    torch.cuda.synchronize()
    assert h.device_error() == hlb.HEADLOSS_OK
    h.close()
    cfg, rec, ref, gmag = H.oracle_rows(wl, inp)
    H.check_scalars(wl, out.double().cpu().numpy(), cfg, rec)
    H.check_grad(wl, g, ref, gmag, rec)
