"""GPU test of headloss_forward_backward_noalloc, the entry point for callers
that cannot allocate device memory while computing the loss (for example
inside a CUDA-graph capture, or under a pool that forbids raw cudaMalloc).

It must give the handle-based call's results within the parity tolerances
(scalars: 1e-3 relative for bf16 logits; gradient: within 2 ulp of bf16) on
two calls in a row -- the second call reuses the library's fixed scratch
array the first one left behind.  The file runs last so that a failure here
cannot hide the rest of the suite, and it needs nothing from other tests.
"""
import numpy as np
import pytest
import torch

import gradient_row_online_gb300 as pkg
from gradient_row_online_gb300 import headloss as hlb
from gradient_row_online_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ALL = ("ce", "z", "dist_ce", "fkl", "rkl", "grpo", "grpo_stats", "entropy")
WEIGHTS = dict(ce=0.9, z=0.3, dist_ce=0.4, fkl=0.6, rkl=0.7, grpo=1.1, entropy=0.5,
               grad_scale=1.3)


def _ulp_bf16(a, b):
    ia = a.view(torch.int16).to(torch.int64).cpu().numpy()
    ib = b.view(torch.int16).to(torch.int64).cpu().numpy()
    oa = np.where(ia < 0, -(ia & 0x7FFF), ia)
    ob = np.where(ib < 0, -(ib & 0x7FFF), ib)
    return np.abs(oa - ob)


@pytest.mark.parametrize("V,softcap", [(4099, 30.0), (20008, 0.0)])
def test_noalloc_matches_the_handle_call_twice(V, softcap):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hlb.load_library()
    wl = W.Workload("noalloc", 300, V, torch.bfloat16, ALL, dict(WEIGHTS), teacher_noise=1.0,
                    temperature=1.7, softcap=softcap, logits_scale=0.5 if softcap else 1.0,
                    mask_frac=0.1)
    inp = W.make_inputs(wl, "cuda")
    args = (inp["logits"], wl.N, wl.V, hlb.HEADLOSS_BF16, inp["labels"], inp["teacher"],
            inp["old_logprobs"], inp["advantages"])

    # the handle-based call
    h = pkg.headloss_for(wl)
    g_ref = torch.empty_like(inp["logits"])
    s_ref = torch.empty(16, dtype=torch.float32, device="cuda")
    h(inp["logits"], inp["labels"], inp["teacher"], inp["old_logprobs"], inp["advantages"],
      g_ref, s_ref)
    torch.cuda.synchronize()
    assert h.device_error() == hlb.HEADLOSS_OK

    flags = pkg.flags_of(wl.losses)
    weights = hlb.make_weights(**wl.weights)
    g = torch.empty_like(inp["logits"])
    out = torch.empty(16, dtype=torch.float32, device="cuda")
    results = []
    free = []
    for call in range(2):
        g.fill_(float("nan"))
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        hlb.headloss_forward_backward_noalloc(flags, weights, wl.temperature, wl.clip_eps,
                                              wl.softcap, wl.logits_scale, *args, g, out)
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        results.append((out.clone(), g.clone()))
    # the second call allocated no device memory: free memory is the same on
    # both sides of it (only the library runs in between)
    assert free[3] == free[2]
    b = s_ref.double().cpu().numpy()
    for call, (o, gg) in enumerate(results):
        a = o.double().cpu().numpy()
        rel = np.abs(a - b) / np.maximum(np.abs(b), 1e-30)
        assert np.all((rel <= 1e-3) | (np.abs(a - b) <= 1e-6)), (call, a, b)
        assert a[14] == b[14] and a[15] == b[15]  # counts are exact
        assert int(_ulp_bf16(gg, g_ref).max()) <= 2, call
    h.close()


def test_noalloc_rejects_bad_arguments_before_any_work():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lib = hlb.load_library()
    out = torch.empty(16, device="cuda")
    x = torch.zeros(2, 8, dtype=torch.bfloat16, device="cuda")
    lab = torch.zeros(2, dtype=torch.int64, device="cuda")
    w = hlb.make_weights()
    cases = [
        (dict(flags=0), hlb.HEADLOSS_ERR_ARG),
        (dict(temperature=0.0), hlb.HEADLOSS_ERR_ARG),
        (dict(N=-1), hlb.HEADLOSS_ERR_ARG),
        (dict(labels=None), hlb.HEADLOSS_ERR_MISSING_INPUT),
        (dict(logits=x.data_ptr() + 2), hlb.HEADLOSS_ERR_ALIGN),
    ]
    for over, status in cases:
        a = dict(flags=hlb.HEADLOSS_CE, weights=w, temperature=1.0, clip_eps=0.2, softcap=0.0,
                 logits_scale=1.0, logits=x, N=2, V=8, dtype=hlb.HEADLOSS_BF16, labels=lab,
                 teacher_logits=None, old_logprobs=None, advantages=None, grad_out=None,
                 scalars_out=out)
        a.update(over)
        with pytest.raises(hlb.HeadlossError) as e:
            hlb.headloss_forward_backward_noalloc(**a)
        assert e.value.status == status, (over, e.value.status)
    del lib
