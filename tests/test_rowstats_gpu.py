"""GPU parity of the fused LM head's single-pass loss: the GEMM epilogue's
per-tile row statistics (headloss_lmhead_logits_rowstats) consumed by the
loss's gradient pass alone (headloss_forward_backward_rowstats), against the
fp64 row oracle on the same logits.

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


def _run(wl, inp, inplace=False):
    N, V = wl.N, wl.V
    x = inp["logits"]
    eye = torch.eye(V, dtype=torch.bfloat16, device="cuda")
    logits = torch.empty_like(x)
    rs = torch.full((N, V // 256, 4), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hlb.headloss_lmhead_logits_rowstats(x, eye, N, V, V, wl.softcap, wl.logits_scale, logits, rs,
                                        err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(logits.view(torch.int16), x.view(torch.int16))
    h = pkg.headloss_for(wl)
    g = logits if inplace else torch.empty_like(logits)
    out = torch.full((16,), float("nan"), device="cuda")
    ref_x = logits.clone() if inplace else logits
    hlb.headloss_forward_backward_rowstats(h.h, logits, N, V, hlb.HEADLOSS_BF16, inp["labels"],
                                           inp["old_logprobs"], inp["advantages"], rs, g, out)
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


def test_rowstats_rejects_what_it_does_not_cover():
    wl = W.Workload("rowstats", 128, 256, torch.bfloat16, ("ce", "fkl"),
                    dict(W_ALL, fkl=0.5), teacher_noise=1.0)
    inp = W.make_inputs(wl, "cuda")
    rs = torch.zeros(128, 1, 4, device="cuda")
    out = torch.empty(16, device="cuda")
    h = pkg.headloss_for(wl)
    fb = hlb.headloss_forward_backward_rowstats
    with pytest.raises(hlb.HeadlossError) as e:  # a teacher loss
        fb(h.h, inp["logits"], 128, 256, hlb.HEADLOSS_BF16, inp["labels"], None, None, rs, None,
           out)
    assert e.value.status == hlb.HEADLOSS_ERR_ARG
    h.close()
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
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hlb.headloss_lmhead_logits_rowstats(x, eye, N, V, V, softcap, scale, logits, rs, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(logits.view(torch.int16), x.view(torch.int16))
    got = rs.double().cpu().numpy()
    ref = orc.tile_records(x.float().cpu().numpy(), softcap, scale)
    np.testing.assert_array_equal(got[..., 3], ref[..., 3])
    np.testing.assert_allclose(got[..., 0], ref[..., 0], rtol=2e-5, atol=2e-5)
    np.testing.assert_allclose(got[..., 1], ref[..., 1], rtol=2e-5, atol=0)
    assert np.all(np.abs(got[..., 2] - ref[..., 2]) <= 2e-5 * (ref[..., 1] + np.abs(ref[..., 2])))
