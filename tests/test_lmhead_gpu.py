"""The LM-head GEMM with its row-statistics epilogue (include/headloss_lmhead.h)
on the GPU, against the fp64 oracle of the LM head in front of the loss
(oracle.lm_head_forward_backward: logits = hidden @ weight^T in fp64).

- logits: within one bf16 step of the fp64 product (fp32 accumulation in
  another order, one rounding), plus 2^-20 of sum_d |h_d w_d| where the sum
  over D cancels;
- per-tile statistics: exactly the max of the tile's bf16 logits, and the sum
  of exp(logit - max) to fp32 accuracy;
- the row log-sum-exp rebuilt from the tiles' (max, sum) pairs: against the
  oracle's log-sum-exp of the same bf16 logits (to fp32 accuracy) and of the
  fp64 logits (to the logits' own rounding).

Shapes: one tile and one K block; K loops that wrap the 4-stage ring several
times (D = 640, 2048); grids with several tiles per CTA, so both TMEM
accumulators and the grouped tile order (with a narrower last group) are
used; large shapes compare sampled rows."""
import numpy as np
import pytest
import torch

import oracle as orc
from gradient_row_online_gb300 import headloss as hlb

pytestmark = pytest.mark.gpu

# accumulation bound for cancelling sums (fp32 accumulation over D)
TAU = 2.0 ** -20


def _inputs(N, D, V, seed=0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    hid = (torch.randn(N, D, generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    wt = (torch.randn(V, D, generator=g, device="cuda") * (1.0 / D) ** 0.5).to(torch.bfloat16)
    return hid, wt


def _run(hid, wt, N, D, V):
    out = torch.full((N, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.full((N, V // 256, 2), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hlb.headloss_lmhead_logits(hid, wt, N, D, V, out, st, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out, st


def _check_rows(hid, wt, out, st, rows):
    """Oracle comparison on the given rows."""
    V = wt.shape[0]
    sel = torch.as_tensor(rows, device="cuda")
    h64 = hid.index_select(0, sel).double().cpu().numpy()
    w64 = wt.double().cpu().numpy()
    cfg = orc.make_cfg(orc.CE)
    labels = np.zeros(len(rows), np.int64)
    _, rec, _, _, x, _ = orc.lm_head_forward_backward(cfg, h64, w64, labels)
    got = out.index_select(0, sel).double().cpu().numpy()
    # within one bf16 step of the fp64 product, except where the sum over D
    # cancels: there the fp32 accumulation's own error, a small multiple of
    # 2^-24 of sum_d |h_d w_d|, may exceed a step of the small result
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126))) - 7)
    mag = np.abs(h64) @ np.abs(w64).T
    bad = np.abs(got - x) > ulp + TAU * mag
    if bad.any():
        ii, jj = np.nonzero(bad)
        raise AssertionError(("logits beyond one bf16 step", int(bad.sum()),
                              [(int(rows[i]), int(j), float(x[i, j]), float(got[i, j]))
                               for i, j in zip(ii[:6], jj[:6])]))
    # per-tile statistics of the kernel's own bf16 logits
    s = st.index_select(0, sel).double().cpu().numpy()
    t = got.reshape(len(rows), V // 256, 256)
    m = t.max(-1)
    assert np.array_equal(s[..., 0], m)
    ssum = np.exp(t - m[..., None]).sum(-1)
    assert float(np.abs(s[..., 1] / ssum - 1).max()) < 2e-6
    # the row log-sum-exp from the tile pairs
    mstar = s[..., 0].max(-1)
    lse = mstar + np.log((s[..., 1] * np.exp(s[..., 0] - mstar[:, None])).sum(-1))
    rec_b, _, _ = orc.rows(cfg, got, labels, want_grad=False)
    assert float(np.abs(lse - rec_b[:, orc.RF["lse"]]).max()) < 2e-5 * max(1.0, float(np.abs(lse).max()))
    tol = np.abs(x).max(-1) * 2.0 ** -8 + 1e-6
    assert bool((np.abs(lse - rec[:, orc.RF["lse"]]) <= tol).all())


@pytest.mark.parametrize("N,D,V", [(128, 64, 256), (256, 128, 512), (256, 640, 4096),
                                   (256, 2048, 4096), (384, 192, 4352)])
def test_lmhead_against_oracle(N, D, V):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hid, wt = _inputs(N, D, V)
    out, st = _run(hid, wt, N, D, V)
    _check_rows(hid, wt, out, st, np.arange(N))


# a full-width grid: 8 x 128 tiles, about seven per CTA
def test_lmhead_large_grid_sampled_rows():
    N, D, V = 1024, 1024, 32768
    hid, wt = _inputs(N, D, V, seed=1)
    out, st = _run(hid, wt, N, D, V)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.choice(N, 12, replace=False)]))
    _check_rows(hid, wt, out, st, rows)
    # every logit against torch's fp32 matmul, rounded once (a whole-grid check)
    ref = (hid.float() @ wt.float().T)
    d = (out.float() - ref).abs()
    assert bool((d <= ref.abs() * 2.0 ** -7 + 1e-3).all()), float(d.max())


def test_lmhead_back_to_back_calls_identical():
    N, D, V = 512, 512, 8192
    hid, wt = _inputs(N, D, V, seed=2)
    a, sa = _run(hid, wt, N, D, V)
    b, sb = _run(hid, wt, N, D, V)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(sa, sb)


def test_lmhead_host_checks():
    hid, wt = _inputs(128, 64, 256)
    out = torch.empty(128, 256, dtype=torch.bfloat16, device="cuda")
    st = torch.empty(128, 1, 2, device="cuda")
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    call = hlb.headloss_lmhead_logits
    for args, status in [((hid, wt, 100, 64, 256, out, st, err), hlb.HEADLOSS_ERR_ARG),
                         ((hid, wt, 128, 60, 256, out, st, err), hlb.HEADLOSS_ERR_ARG),
                         ((hid, wt, 128, 64, 200, out, st, err), hlb.HEADLOSS_ERR_ARG),
                         ((hid, wt, 128, 64, 256, out, st.data_ptr() + 4, err),
                          hlb.HEADLOSS_ERR_ALIGN)]:
        with pytest.raises(hlb.HeadlossError) as e:
            call(*args)
        assert e.value.status == status


def test_lmhead_rowstats_host_checks():
    """The statistics call's own checks: softcap, scale and (with sums at a
    temperature) the temperature and the sums' alignment."""
    hid, wt = _inputs(128, 64, 256)
    out = torch.empty(128, 256, dtype=torch.bfloat16, device="cuda")
    rs = torch.empty(128, 1, 4, device="cuda")
    rsT = torch.empty(128, 2, device="cuda")
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    call = hlb.headloss_lmhead_logits_rowstats
    base = (hid, wt, 128, 64, 256)
    for kw, status in [(dict(softcap=-1.0), hlb.HEADLOSS_ERR_ARG),
                       (dict(scale=0.0), hlb.HEADLOSS_ERR_ARG),
                       (dict(temperature=0.0, row_stats_t=rsT), hlb.HEADLOSS_ERR_ARG),
                       (dict(temperature=float("inf"), row_stats_t=rsT), hlb.HEADLOSS_ERR_ARG),
                       (dict(row_stats_t=rsT.data_ptr() + 2), hlb.HEADLOSS_ERR_ALIGN),
                       (dict(row_stats=rs.data_ptr() + 8), hlb.HEADLOSS_ERR_ALIGN)]:
        a = dict(softcap=0.0, scale=1.0, temperature=1.5, row_stats_t=None, row_stats=rs)
        a.update(kw)
        with pytest.raises(hlb.HeadlossError) as e:
            call(*base, a["softcap"], a["scale"], out, a["row_stats"], err,
                 temperature=a["temperature"], row_stats_t=a["row_stats_t"])
        assert e.value.status == status
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0  # nothing ran
