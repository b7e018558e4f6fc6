"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.  Small cases compare every output element; the full-size
workloads compare every scalar over all rows and the gradient on sampled
rows, in the launch configuration the benchmark times."""
import itertools

import numpy as np
import pytest
import torch

import oracle as orc
import gradient_row_online_gb300 as pkg
from gradient_row_online_gb300 import headloss as hlb
from gradient_row_online_gb300 import workloads as W
from tests import _harness as H

pytestmark = pytest.mark.gpu

ALL_LOSSES = ("ce", "z", "dist_ce", "fkl", "rkl", "grpo", "grpo_stats", "entropy")
FULL_W = dict(ce=0.9, z=0.3, dist_ce=0.4, fkl=0.6, rkl=0.7, grpo=1.1, entropy=0.5,
              grad_scale=1.3)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hlb.load_library()


def small(losses, N=33, V=257, dtype=torch.bfloat16, **kw):
    base = W.Workload("small", N, V, dtype, tuple(losses), dict(FULL_W), sigma=3.0,
                      mask_frac=0.2, teacher_noise=1.0, temperature=1.7, clip_eps=0.2)
    return base.replace(**kw) if kw else base


def full_check(wl, plan=None, inplace=False):
    inp = W.make_inputs(wl, "cuda")
    ref_inp = dict(inp, logits=inp["logits"].clone()) if inplace else inp
    got, g, _ = H.run_gpu(wl, inp, plan=plan, inplace=inplace)
    cfg, rec, ref, gmag = H.oracle_rows(wl, ref_inp)
    H.check_scalars(wl, got, cfg, rec)
    H.check_grad(wl, g, ref, gmag, rec)


# ------------------------------------------------------------ small, every output

def test_tiny_ce_z_fp32_workload():
    full_check(W.WORKLOADS["tiny_ce_z_fp32"])


SUBSETS = [c for r in range(1, 9) for c in itertools.combinations(ALL_LOSSES, r)]


# softcap 20: |x| / c stays in the polynomial tanh range; softcap 3: most rows
# fall back to the exp / reciprocal tanh
@pytest.mark.parametrize("softcap,scale", [(0.0, 1.0), (20.0, 0.6), (3.0, 0.7)])
def test_every_loss_subset_bf16(softcap, scale):
    for losses in SUBSETS:
        full_check(small(losses, softcap=softcap, logits_scale=scale, seed=len(losses)))


@pytest.mark.parametrize("dtype", [torch.float16, torch.float32])
@pytest.mark.parametrize("losses", [("ce",), ("ce", "z"), ("grpo", "grpo_stats", "entropy"),
                                    ("dist_ce", "fkl", "rkl"), ALL_LOSSES])
def test_loss_sets_fp16_fp32(dtype, losses):
    full_check(small(losses, dtype=dtype))
    full_check(small(losses, dtype=dtype, softcap=15.0, logits_scale=1.3, seed=3))


@pytest.mark.parametrize("V", [1, 2, 7, 8, 9, 1000, 1023, 1024, 32001])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_ragged_and_tiny_vocab(V, dtype):
    full_check(small(ALL_LOSSES, N=19, V=V, dtype=dtype))


RESIDENT, STREAM = hlb.HEADLOSS_KERNEL_RESIDENT, hlb.HEADLOSS_KERNEL_STREAM


@pytest.mark.parametrize("cluster,stages,threads", [
    (1, 2, 512), (2, 2, 512), (2, 3, 256), (3, 1, 256), (4, 2, 512), (5, 1, 256), (6, 1, 512),
    (7, 1, 256), (8, 2, 256), (8, 4, 512)])
def test_forced_resident_plans(cluster, stages, threads):
    plan = dict(kernel=RESIDENT, cluster=cluster, stages=stages, threads=threads)
    wl = small(ALL_LOSSES, N=40, V=20011, softcap=30.0, logits_scale=0.5)
    full_check(wl, plan=plan)
    full_check(small(("ce", "z", "entropy"), N=40, V=8000, dtype=torch.float32), plan=plan)


# the streaming kernel: aligned rows only (V a multiple of 8), several chunks
# per row plus a partial last chunk, every feature set, both tanh paths
@pytest.mark.parametrize("stages,threads,words", [(2, 256, 1), (3, 512, 1), (4, 256, 2),
                                                   (6, 256, 4), (6, 512, 2), (8, 256, 1),
                                                   (3, 512, 4)])
@pytest.mark.parametrize("V", [8, 1000, 20008])
def test_forced_stream_plans(stages, threads, words, V):
    plan = dict(kernel=STREAM, stages=stages, threads=threads, chunk_words=words)
    full_check(small(ALL_LOSSES, N=23, V=V, softcap=30.0, logits_scale=0.5), plan=plan)
    full_check(small(ALL_LOSSES, N=23, V=V, softcap=2.0, seed=5), plan=plan)
    full_check(small(("ce", "z", "grpo", "grpo_stats"), N=23, V=V, dtype=torch.float16),
               plan=plan)
    full_check(small(("dist_ce", "fkl", "rkl", "entropy"), N=23, V=V, sigma=6.0), plan=plan)


def structured_check(wl, plan=None):
    inp = W.make_structured_inputs(wl, "cuda")
    got, g, _ = H.run_gpu(wl, inp, plan=plan)
    cfg, rec, ref, gmag = H.oracle_rows(wl, inp)
    H.check_scalars(wl, got, cfg, rec)
    H.check_grad(wl, g, ref, gmag, rec)


# rows whose maximum comes last, first or as one spike, large offsets and
# wide ranges: the streaming kernel's lazily raised shifts and its per-chunk
# softcap tiers (35 chunks per row at V = 70000, beyond the 32 it records one
# by one), with and without the entropy gradient and the teacher-entropy sum
@pytest.mark.parametrize("softcap,scale", [(0.0, 0.7), (30.0, 0.5), (10.0, 1.0), (60.0, 1.0)])
@pytest.mark.parametrize("V", [4104, 70000])
def test_stream_structured_rows(softcap, scale, V):
    plan = dict(kernel=STREAM, stages=3, threads=256, chunk_words=1)
    for losses, ent in ((ALL_LOSSES, 0.5), (("ce", "z", "fkl", "grpo", "grpo_stats", "entropy"), 0.0),
                        (("dist_ce", "rkl", "entropy"), 0.0)):
        wl = small(losses, N=24, V=V, softcap=softcap, logits_scale=scale,
                   weights=dict(FULL_W, entropy=ent))
        structured_check(wl, plan=plan)


# fp16 rows through the streaming kernel: its own unpack and packed abs-max,
# every softcap tier, teacher and reverse KL
@pytest.mark.parametrize("softcap,scale", [(0.0, 0.7), (30.0, 0.5), (10.0, 1.0)])
def test_stream_structured_rows_fp16(softcap, scale):
    plan = dict(kernel=STREAM, stages=3, threads=256, chunk_words=1)
    wl = small(ALL_LOSSES, N=24, V=4104, dtype=torch.float16, softcap=softcap,
               logits_scale=scale, weights=dict(FULL_W, entropy=0.0))
    structured_check(wl, plan=plan)
    full_check(small(ALL_LOSSES, N=23, V=20008, dtype=torch.float16, softcap=softcap,
                     logits_scale=scale), plan=dict(kernel=STREAM, stages=3, threads=256,
                                                    chunk_words=4))


@pytest.mark.parametrize("softcap,scale", [(0.0, 1.0), (30.0, 0.5), (15.0, 1.3)])
def test_stream_structured_rows_default_plan(softcap, scale):
    wl = small(ALL_LOSSES, N=40, V=128256, softcap=softcap, logits_scale=scale,
               weights=dict(FULL_W, entropy=0.0))
    structured_check(wl)


@pytest.mark.parametrize("softcap,scale", [(0.0, 0.7), (10.0, 1.0), (30.0, 0.5)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_resident_structured_rows(softcap, scale, dtype):
    for plan in (dict(kernel=RESIDENT, cluster=2, stages=2, threads=256),
                 dict(kernel=RESIDENT, cluster=1, stages=1, threads=512)):
        wl = small(ALL_LOSSES, N=24, V=4100, dtype=dtype, softcap=softcap, logits_scale=scale)
        structured_check(wl, plan=plan)


def test_stream_every_loss_subset():
    plan = dict(kernel=STREAM, stages=4, threads=256, chunk_words=1)
    for losses in SUBSETS:
        full_check(small(losses, N=17, V=4104, seed=len(losses)), plan=plan)


# the gradient written over the logits with a pinned streaming plan, a
# teacher, softcap and a partial last chunk: an in-place call takes the
# resident kernel whatever plan is pinned (the streaming kernel would re-read
# the row from global memory as it stores the gradient over it)
@pytest.mark.parametrize("words", [1, 4])
def test_stream_plan_in_place_takes_resident(words):
    plan = dict(kernel=STREAM, stages=3, threads=256, chunk_words=words)
    full_check(small(ALL_LOSSES, N=23, V=20008, softcap=30.0, logits_scale=0.5), plan=plan,
               inplace=True)
    full_check(small(("ce", "z", "grpo", "grpo_stats", "entropy"), N=23, V=20008), plan=plan,
               inplace=True)


# fp32 logits without a teacher, softcap or entropy gradient take the
# double-float kernel (fp32 pairs instead of fp64): every loss subset, three
# scales, ragged rows, structured rows (ramps, +300 offsets, spikes, wide
# noise: many terms far below the maximum and subnormal gradients), forced
# cluster plans, and logits far apart (sigma 1e4); same tolerances as fp64
DF_LOSSES = ("ce", "z", "grpo", "grpo_stats", "entropy")
DF_SUBSETS = [c for r in range(1, 6) for c in itertools.combinations(DF_LOSSES, r)]
NO_ENT_GRAD = dict(FULL_W, entropy=0.0)


@pytest.mark.parametrize("scale", [1.0, 0.6, 1.7])
def test_fp32_double_float_every_subset(scale):
    for losses in DF_SUBSETS:
        full_check(small(losses, N=40, V=1031, dtype=torch.float32, logits_scale=scale,
                         sigma=5.0, seed=len(losses), weights=NO_ENT_GRAD))


@pytest.mark.parametrize("V", [1, 2, 7, 1023, 1024, 32001])
def test_fp32_double_float_ragged(V):
    full_check(small(DF_LOSSES, N=19, V=V, dtype=torch.float32, weights=NO_ENT_GRAD))


@pytest.mark.parametrize("plan", [None, dict(kernel=RESIDENT, cluster=2, stages=2, threads=256),
                                  dict(kernel=RESIDENT, cluster=4, stages=1, threads=512),
                                  dict(kernel=RESIDENT, cluster=1, stages=1, threads=512)])
@pytest.mark.parametrize("scale", [1.0, 0.7])
def test_fp32_double_float_structured_rows(plan, scale):
    wl = small(DF_LOSSES, N=24, V=4100, dtype=torch.float32, logits_scale=scale,
               weights=NO_ENT_GRAD)
    structured_check(wl, plan=plan)
    structured_check(wl.replace(losses=("ce", "z")), plan=plan)


@pytest.mark.parametrize("losses", [("ce", "z"), ("ce", "grpo", "grpo_stats", "entropy")])
def test_fp32_double_float_confident_rows(losses):
    """Rows whose label logit leads by 4 .. 36: p(label) up to 1 - 1e-8, so the
    label element pc p - bc cancels; it is held to the cancellation bound."""
    wl = small(losses, N=36, V=1000, dtype=torch.float32, sigma=1.0, weights=NO_ENT_GRAD)
    inp = W.make_inputs(wl, "cuda")
    lab = inp["labels"]
    rows = torch.nonzero(lab >= 0)[:, 0]
    margin = 4.0 + (rows % 10).to(torch.float32) * 3.5
    inp["logits"][rows, lab[rows]] += margin
    got, g, _ = H.run_gpu(wl, inp)
    cfg, rec, ref, gmag = H.oracle_rows(wl, inp)
    H.check_scalars(wl, got, cfg, rec)
    H.check_grad(wl, g, ref, gmag, rec)


def test_fp32_double_float_far_apart_logits():
    full_check(small(("ce", "z", "grpo", "grpo_stats", "entropy"), N=8, V=513,
                     dtype=torch.float32, sigma=1e4, weights=NO_ENT_GRAD))
    full_check(small(("ce",), N=30, V=2000, dtype=torch.float32, sigma=40.0))


# no labels (no mask, every row valid): the losses that need none, both kernels
@pytest.mark.parametrize("plan", [dict(kernel=RESIDENT, cluster=2, stages=1, threads=256),
                                  dict(kernel=STREAM, stages=3, threads=256, chunk_words=4)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_without_labels(plan, dtype):
    if dtype == torch.float32 and plan["kernel"] == STREAM:
        pytest.skip("the streaming kernel takes 16-bit rows")
    # fp32 rows without softcap and entropy gradient take the double-float kernel
    for losses, w in ((("dist_ce", "fkl", "rkl", "entropy"), FULL_W), (("z", "entropy"), NO_ENT_GRAD),
                      (("fkl",), FULL_W)):
        wl = small(losses, N=29, V=4104, dtype=dtype, logits_scale=0.7, weights=dict(w),
                   softcap=20.0 if dtype == torch.bfloat16 else 0.0)
        inp = dict(W.make_inputs(wl, "cuda"), labels=None)
        got, g, _ = H.run_gpu(wl, inp, plan=plan)
        cfg, rec, ref, gmag = H.oracle_rows(wl, inp)
        assert got[14] == wl.N
        H.check_scalars(wl, got, cfg, rec)
        H.check_grad(wl, g, ref, gmag, rec)


def test_large_logits_fp32():
    wl = small(("ce", "z", "entropy", "fkl", "rkl"), N=8, V=513, dtype=torch.float32,
               sigma=1e4)
    full_check(wl)


def test_in_place_gradient():
    full_check(small(("ce", "z", "grpo", "grpo_stats", "entropy"), N=50, V=3000), inplace=True)


def test_metrics_without_gradient_match_and_write_nothing():
    wl = small(ALL_LOSSES, N=30, V=999, weights=dict(FULL_W, ce=0.0, grpo=0.0))
    inp = W.make_inputs(wl, "cuda")
    a, g, h = H.run_gpu(wl, inp, grad=True)
    b, _, _ = H.run_gpu(wl, inp, grad=False, handle=h)
    assert np.array_equal(a, b)
    cfg, rec, ref, gmag = H.oracle_rows(wl, inp)
    H.check_scalars(wl, b, cfg, rec)


def test_deterministic_bitwise():
    wl = small(ALL_LOSSES, N=300, V=4099, softcap=10.0)
    inp = W.make_inputs(wl, "cuda")
    a, ga, h = H.run_gpu(wl, inp)
    b, gb, _ = H.run_gpu(wl, inp, handle=h)
    assert np.array_equal(a, b)
    assert torch.equal(ga.view(torch.int16), gb.view(torch.int16))


def test_all_rows_masked_and_empty_batch():
    wl = small(ALL_LOSSES, N=12, V=300, mask_frac=1.1)
    inp = W.make_inputs(wl, "cuda")
    got, g, h = H.run_gpu(wl, inp)
    assert np.all(got == 0.0)
    assert int(g.view(torch.int16).abs().max()) == 0
    empty = {k: (None if v is None else v[:0]) for k, v in inp.items()}
    out = torch.full((16,), 7.0, device="cuda")
    h(empty["logits"], empty["labels"], empty["teacher"], empty["old_logprobs"],
      empty["advantages"], empty["logits"], out)
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def test_label_out_of_range_is_reported_and_masked():
    wl = small(("ce", "z"), N=20, V=100, mask_frac=0.0)
    inp = W.make_inputs(wl, "cuda")
    inp["labels"][3] = 100
    h = __import__("gradient_row_online_gb300").headloss_for(wl)
    g = torch.empty_like(inp["logits"])
    out = torch.empty(16, device="cuda")
    h(inp["logits"], inp["labels"], None, None, None, g, out)
    assert h.device_error() == hlb.HEADLOSS_ERR_LABEL_RANGE
    assert h.device_error() == hlb.HEADLOSS_OK  # read clears it
    assert int(g[3].view(torch.int16).abs().max()) == 0
    assert out[14].item() == 19


def test_host_side_argument_errors():
    wl = small(ALL_LOSSES, N=4, V=64)
    inp = W.make_inputs(wl, "cuda")
    h = __import__("gradient_row_online_gb300").headloss_for(wl)
    x, lab, t = inp["logits"], inp["labels"], inp["teacher"]
    o, a = inp["old_logprobs"], inp["advantages"]
    out = torch.empty(16, device="cuda")
    fb = hlb.headloss_forward_backward
    cases = [
        (dict(teacher_logits=None), hlb.HEADLOSS_ERR_MISSING_INPUT),
        (dict(labels=None), hlb.HEADLOSS_ERR_MISSING_INPUT),
        (dict(old_logprobs=None), hlb.HEADLOSS_ERR_MISSING_INPUT),
        (dict(logits=x.data_ptr() + 2), hlb.HEADLOSS_ERR_ALIGN),
        (dict(grad_out=x.data_ptr() + 4), hlb.HEADLOSS_ERR_ALIGN),
        (dict(grad_out=t), hlb.HEADLOSS_ERR_ARG),
        (dict(dtype=7), hlb.HEADLOSS_ERR_DTYPE),
        (dict(N=-1), hlb.HEADLOSS_ERR_ARG),
        (dict(V=0), hlb.HEADLOSS_ERR_ARG),
        (dict(scalars_out=None), hlb.HEADLOSS_ERR_ARG),
    ]
    for over, status in cases:
        args = dict(h=h.h, logits=x, N=4, V=64, dtype=hlb.HEADLOSS_BF16, labels=lab,
                    teacher_logits=t, old_logprobs=o, advantages=a, grad_out=None,
                    scalars_out=out, stream=None)
        args.update(over)
        with pytest.raises(hlb.HeadlossError) as e:
            fb(**args)
        assert e.value.status == status, (over, e.value.status)


def test_create_rejects_bad_configuration():
    bad = [dict(flags=0), dict(flags=1 << 9), dict(temperature=0.0), dict(clip_eps=-1.0),
           dict(softcap=-1.0), dict(logits_scale=0.0)]
    for b in bad:
        args = dict(flags=hlb.HEADLOSS_CE, weights=None, temperature=1.0, clip_eps=0.2,
                    softcap=0.0, logits_scale=1.0)
        args.update(b)
        with pytest.raises(hlb.HeadlossError) as e:
            hlb.headloss_create(**args)
        assert e.value.status == hlb.HEADLOSS_ERR_ARG


# ----------------------------------------------- full-size workloads (bench plan)

FULL = ("ce_z_bf16", "ce_distill_bf16", "grpo_z_entropy_bf16", "all_in_bf16", "ce_z_fp32")


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    wl = W.WORKLOADS[name]
    inp = W.make_inputs(wl, "cuda")
    got, g, h = H.run_gpu(wl, inp)
    # every scalar over all rows (oracle without gradient)
    cfg, rec, _, _ = H.oracle_rows(wl, inp, want_grad=False, want_gmag=False)
    H.check_scalars(wl, got, cfg, rec)
    # the gradient on sampled rows: first, last, masked, and a seeded spread
    rng = np.random.default_rng(0)
    labels = inp["labels"].cpu().numpy()
    rows = set([0, 1, wl.N - 1]) | set(rng.choice(wl.N, 40, replace=False).tolist())
    rows |= set(np.nonzero(labels < 0)[0][:4].tolist())
    rows = np.array(sorted(rows))
    _, srec, ref, gmag = H.oracle_rows(wl, inp, rows=rows)
    sel = torch.as_tensor(rows, device="cuda")
    H.check_grad(wl, g.index_select(0, sel), ref, gmag, srec)
    del inp, g
    torch.cuda.empty_cache()


# distillation at T = 2 exactly: bf16 teacher rows without softcap or entropy
# take the one-exponential form (2^d = (2^(d/2))^2) on the streaming kernel;
# every teacher loss combination, several chunk shapes with a partial last
# chunk, structured rows (large offsets, spikes, ramps), and the same call at
# T = 2 where that form does not apply (fp16 logits, accumulation, entropy)
T2_SETS = [("ce", "fkl", "rkl"), ("dist_ce", "fkl"), ("rkl",),
           ("ce", "z", "dist_ce", "rkl", "grpo", "grpo_stats")]


@pytest.mark.parametrize("losses", T2_SETS)
@pytest.mark.parametrize("plan", [None, dict(kernel=STREAM, stages=3, threads=512, chunk_words=4),
                                  dict(kernel=STREAM, stages=3, threads=256, chunk_words=1)])
@pytest.mark.parametrize("V", [1000, 20008, 70000])
def test_temperature_two_streaming(losses, plan, V):
    wl = small(losses, N=23, V=V, temperature=2.0, sigma=4.0, logits_scale=0.8)
    full_check(wl, plan=plan)
    structured_check(wl.replace(N=24, seed=3), plan=plan or dict(kernel=STREAM, stages=3,
                                                                  threads=256, chunk_words=4))


@pytest.mark.parametrize("kw", [dict(dtype=torch.float16), dict(losses=("ce", "fkl", "entropy")),
                                dict(softcap=30.0)])
def test_temperature_two_general_path(kw):
    losses = kw.pop("losses", ("ce", "fkl", "rkl"))
    wl = small(losses, N=23, V=20008, temperature=2.0, **kw)
    full_check(wl, plan=dict(kernel=STREAM, stages=3, threads=256, chunk_words=4))


def test_temperature_two_accumulating():
    wl = small(("ce", "fkl", "rkl"), N=23, V=20008, temperature=2.0)
    inp = W.make_inputs(wl, "cuda")
    h = pkg.headloss_for(wl)
    h.force_plan(kernel=STREAM, stages=3, threads=256, chunk_words=4)
    g0 = (torch.randn(inp["logits"].shape, device="cuda") * 1e-4).to(wl.dtype)
    g = g0.clone()
    h(inp["logits"], inp["labels"], inp["teacher"], inp["old_logprobs"], inp["advantages"], g,
      accumulate=True)
    torch.cuda.synchronize()
    assert h.device_error() == hlb.HEADLOSS_OK
    cfg, rec, ref, gmag = H.oracle_rows(wl, inp)
    valid = rec[:, orc.RF["valid"]] > 0
    sel = torch.from_numpy(np.nonzero(valid)[0]).cuda()
    g0h = g0.double().cpu().numpy()
    H.check_grad(wl, g.index_select(0, sel), (g0h + ref)[valid], (gmag + np.abs(g0h))[valid],
                 rec[valid])


def test_temperature_two_without_labels():
    """The temperature-2 form with no labels (every row valid, no label term)."""
    plan = dict(kernel=STREAM, stages=3, threads=512, chunk_words=4)
    for losses in (("dist_ce", "fkl"), ("fkl", "rkl"), ("rkl",)):
        wl = small(losses, N=29, V=20008, temperature=2.0, logits_scale=0.7)
        inp = dict(W.make_inputs(wl, "cuda"), labels=None)
        got, g, _ = H.run_gpu(wl, inp, plan=plan)
        cfg, rec, ref, gmag = H.oracle_rows(wl, inp)
        assert got[14] == wl.N
        H.check_scalars(wl, got, cfg, rec)
        H.check_grad(wl, g, ref, gmag, rec)


def test_temperature_two_per_row_outputs_and_divisor():
    """The temperature-2 form with the call's per-row outputs and a batch split
    over two calls that share one divisor."""
    from tests import test_call_ext_gpu as CX
    wl = small(("ce", "fkl", "rkl"), N=40, V=20008, temperature=2.0)
    inp = W.make_inputs(wl, "cuda")
    cfg, rec, ref, gmag = H.oracle_rows(wl, inp)
    whole = orc.reduce(cfg, rec)
    valid = rec[:, orc.RF["valid"]] > 0
    lp_ref, rl_ref = CX.expected_rows(wl, rec)
    h = pkg.headloss_for(wl)
    h.force_plan(kernel=STREAM, stages=3, threads=512, chunk_words=4)
    g = torch.empty_like(inp["logits"])
    lp = torch.full((wl.N,), float("nan"), device="cuda")
    rl = torch.full((wl.N,), float("nan"), device="cuda")
    sums = np.zeros(16)
    for sl in (slice(0, 13), slice(13, 40)):
        pick = lambda t: None if t is None else t[sl].contiguous()
        gp = torch.empty_like(inp["logits"][sl])
        lpp = torch.empty(sl.stop - sl.start, device="cuda")
        rlp = torch.empty(sl.stop - sl.start, device="cuda")
        out = h(pick(inp["logits"]), pick(inp["labels"]), pick(inp["teacher"]), None, None, gp,
                new_logprobs=lpp, row_loss=rlp, divisor=float(whole[14]))
        torch.cuda.synchronize()
        assert h.device_error() == hlb.HEADLOSS_OK
        g[sl] = gp
        lp[sl] = lpp
        rl[sl] = rlp
        sums += out.double().cpu().numpy()
    tol = H.SCALAR_TOL[wl.dtype]
    CX.close_rows(lp.double().cpu().numpy(), lp_ref, valid, tol)
    CX.close_rows(rl.double().cpu().numpy(), rl_ref, valid, tol)
    for slot in (0, 1, 4, 5):  # total, CE, forward KL, reverse KL
        assert abs(sums[slot] - whole[slot]) <= tol * max(1.0, abs(whole[slot])), (slot, sums,
                                                                                   whole)
    H.check_grad(wl, g, ref, gmag, rec)


def test_planner_choices_on_the_benchmarked_sets():
    """The plans the measured figures come from: streamed teacher rows without
    softcap on one 512-thread CTA per SM (half the rows in flight), streamed
    teacher rows with softcap on two 256-thread CTAs per SM, student-only rows
    resident (GRPO rows in 6-CTA clusters), fp32 rows resident in 3-CTA clusters."""
    want = {"ce_distill_bf16": ("stream", 1, 512, 4), "all_in_bf16": ("stream", 1, 256, 4),
            "grpo_z_entropy_bf16": ("resident", 6, 256, 0), "ce_z_bf16": ("resident", 1, 256, 0),
            "ce_z_fp32": ("resident", 3, 256, 0)}
    for name, (kernel, cluster, threads, words) in want.items():
        wl = W.WORKLOADS[name]
        h = pkg.headloss_for(wl)
        p = h.plan(wl.V, hlb.dtype_code(wl.dtype))
        h.close()
        assert (p["kernel"], p["cluster"], p["threads"], p["chunk_words"]) == \
            (kernel, cluster, threads, words), (name, p)
