"""Shared helpers of the parity tests: run the library and the oracle on the
same seeded inputs and compare them under the stated tolerances.

Tolerances (the scalar and gradient bounds of the loss's stated accuracy --
1e-5 / 1e-3 relative scalars, 1e-3 rms-relative and 2-ulp gradients -- read
as follows):
  scalars   rel. error <= 1e-5 (fp32 logits) / 1e-3 (bf16, fp16), where the
            error is divided by max(|ref|, mean_i |row value_i|) so that means
            close to 0 (GRPO) stay well defined; counts exact (n_clipped up to
            the rows the oracle marks as boundary-ambiguous).
  gradient  rms-relative error <= 1e-3, counting only the error beyond the
            output dtype's own rounding (half an ulp), and per element within
            2 ulp of the
            output dtype of the correctly rounded fp64 value -- except where
            the element is a cancellation of larger loss terms, where the bound
            is the compute precision at the terms' scale (TAU * sum |term|);
            masked rows bit-exact +0.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as orc
from gradient_row_online_gb300 import headloss as hlb
from gradient_row_online_gb300 import headloss_for

ORACLE_BITS = {"ce": orc.CE, "z": orc.Z, "dist_ce": orc.DIST_CE, "fkl": orc.FKL, "rkl": orc.RKL,
               "grpo": orc.GRPO, "grpo_stats": orc.GRPO_STATS, "entropy": orc.ENTROPY}

SCALAR_TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-3, torch.float16: 1e-3}
# cancellation bound: fp32 arithmetic (bf16 / fp16 outputs) resolves a sum of
# terms to ~2^-19 of their magnitude; fp64 arithmetic (fp32 output) to ~2^-50.
TAU = {torch.float32: 2.0 ** -45, torch.bfloat16: 2.0 ** -17, torch.float16: 2.0 ** -17}
RMS_TOL = 1e-3
ULP_TOL = 2

# per-row record field behind each scalar slot (for the error denominator)
SLOT_FIELD = {1: "ce", 2: "z", 3: "dist_ce", 4: "fkl", 5: "rkl", 6: "grpo", 7: "logprob",
              8: "ratio", 10: "kl3", 11: "adv", 13: "entropy"}


def oracle_cfg(wl):
    """Oracle configuration of a workload.  The C ABI takes its weights and
    constants as fp32, so the oracle gets exactly those fp32 values."""
    flags = 0
    for name in wl.losses:
        flags |= ORACLE_BITS[name]
    f = lambda v: float(np.float32(v))
    w = {k: f(v) for k, v in wl.weights.items()}
    return orc.make_cfg(flags, dict(ce=w["ce"], z=w["z"], dist_ce=w["dist_ce"], fkl=w["fkl"],
                                    rkl=w["rkl"], grpo=w["grpo"], entropy=w["entropy"]),
                        temperature=f(wl.temperature), clip_eps=f(wl.clip_eps),
                        softcap=f(wl.softcap), logits_scale=f(wl.logits_scale),
                        grad_scale=w["grad_scale"])


def host64(t):
    return None if t is None else t.detach().to(torch.float64).cpu().numpy()


def host_i64(t):
    return None if t is None else t.detach().cpu().numpy().astype(np.int64)


def run_gpu(wl, inp, grad=True, inplace=False, plan=None, handle=None):
    """One library call; returns (scalars f64 numpy[16], grad tensor or None, handle).
    plan: keyword arguments of HeadLoss.force_plan, or None for the automatic plan."""
    h = handle or headloss_for(wl)
    if plan is not None:
        h.force_plan(**plan)
    x = inp["logits"]
    g = None
    if grad:
        g = x if inplace else torch.empty_like(x)
    out = torch.full((16,), float("nan"), dtype=torch.float32, device=x.device)
    h(x, inp["labels"], inp["teacher"], inp["old_logprobs"], inp["advantages"], g, out)
    torch.cuda.synchronize()
    err = h.device_error()
    assert err == hlb.HEADLOSS_OK, hlb.STATUS[err]
    return out.double().cpu().numpy(), g, h


def oracle_rows(wl, inp, rows=None, want_grad=True, want_gmag=True, chunk=1024):
    """Oracle records (and gradient / magnitude) of the selected rows (default all)."""
    cfg = oracle_cfg(wl)
    labels_all = host_i64(inp["labels"])  # None: no mask, every row valid
    n_valid = orc.count_valid(labels_all, inp["logits"].shape[0])
    idx = np.arange(inp["logits"].shape[0]) if rows is None else np.asarray(rows)
    recs, grads, gmags = [], [], []
    for c0 in range(0, len(idx), chunk):
        sel = torch.as_tensor(idx[c0:c0 + chunk], device=inp["logits"].device)
        pick = lambda t: None if t is None else t.index_select(0, sel)
        rec, g, gm = orc.rows(cfg, host64(pick(inp["logits"])), host_i64(pick(inp["labels"])),
                              host64(pick(inp["teacher"])), host64(pick(inp["old_logprobs"])),
                              host64(pick(inp["advantages"])), n_valid, want_grad, want_gmag)
        recs.append(rec)
        if want_grad:
            grads.append(g)
        if want_gmag:
            gmags.append(gm)
    rec = np.concatenate(recs)
    return (cfg, rec, np.concatenate(grads) if want_grad else None,
            np.concatenate(gmags) if want_gmag else None)


def check_scalars(wl, got, cfg, rec):
    ref = orc.reduce(cfg, rec)
    tol = SCALAR_TOL[wl.dtype]
    valid = rec[:, orc.RF["valid"]] > 0
    assert got[14] == ref[14], ("n_valid", got[14], ref[14])
    n_amb = int(rec[:, orc.RF["ambiguous"]].sum())
    assert abs(got[15] - ref[15]) <= n_amb, ("n_clipped", got[15], ref[15], n_amb)
    if ref[14] > 0:
        assert abs(got[9] - ref[9]) <= n_amb / ref[14] + 1e-7, ("clip_frac", got[9], ref[9])
    for slot in range(14):
        if slot == 9:
            continue
        r = ref[slot]
        scale = abs(r)
        if slot in SLOT_FIELD and valid.any():
            scale = max(scale, float(np.abs(rec[valid, orc.RF[SLOT_FIELD[slot]]]).mean()))
        if slot == 0:
            scale = max(scale, max(abs(ref[i]) for i in range(1, 14)))
        if slot == 12:
            scale = max(scale, abs(ref[11]))
        if scale == 0.0:
            assert got[slot] == 0.0, (slot, got[slot])
            continue
        rel = abs(got[slot] - r) / scale
        assert rel <= tol, (hlb.SLOTS[slot], float(got[slot]), float(r), rel)
    return ref


# (explicit mantissa bits, minimum normal exponent) of each output dtype
_FMT = {torch.float32: (23, -126), torch.bfloat16: (7, -126), torch.float16: (10, -14)}


def ulp_of(x, dtype):
    """Spacing of `dtype` values at |x| (subnormal spacing below the normal range)."""
    m, emin = _FMT[dtype]
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.where(ax > 0, np.maximum(e, emin), emin)
    return np.exp2(e - m)


def _ordered(bits_int, nbits):
    mag = bits_int & ((1 << (nbits - 1)) - 1)
    return np.where(bits_int < 0, -mag, mag)


def ulp_distance(got, ref64, dtype):
    """Distance in representable steps of `dtype` between got and RNE(ref64)."""
    ref_d = torch.from_numpy(ref64).to(dtype)
    if dtype == torch.float32:
        a = got.view(torch.int32).to(torch.int64).numpy()
        b = ref_d.view(torch.int32).to(torch.int64).numpy()
        return np.abs(_ordered(a, 32) - _ordered(b, 32))
    a = got.view(torch.int16).to(torch.int64).numpy()
    b = ref_d.view(torch.int16).to(torch.int64).numpy()
    return np.abs(_ordered(a, 16) - _ordered(b, 16))


def check_grad(wl, got_rows, ref, gmag, rec):
    """got_rows: gradient rows (dtype tensor, on host); ref, gmag: fp64 oracle rows."""
    got = got_rows.cpu()
    valid = rec[:, orc.RF["valid"]] > 0
    # masked rows: bit-exact +0
    if (~valid).any():
        bits = got[torch.from_numpy(~valid)]
        bits = bits.view(torch.int32 if wl.dtype == torch.float32 else torch.int16)
        assert int(bits.abs().max()) == 0, "masked row gradient is not +0"
    # rows whose GRPO branch is boundary-ambiguous may legitimately differ
    keep = valid & ~(rec[:, orc.RF["ambiguous"]] > 0)
    if not keep.any():
        return
    g64 = got.double().numpy()[keep]
    r = ref[keep]
    # rms of the error beyond the output dtype's own rounding (half an ulp per
    # element): bf16 rounding alone is ~2^-9 / sqrt(3) = 1.1e-3 rms
    excess = np.maximum(0.0, np.abs(g64 - r) - 0.5 * ulp_of(r, wl.dtype))
    num = np.sqrt(np.sum(excess ** 2))
    den = np.sqrt(np.sum(r ** 2))
    if den > 0:
        assert num / den <= RMS_TOL, ("rms-relative", num / den)
    d = ulp_distance(got[torch.from_numpy(keep)], r, wl.dtype)
    bad = d > ULP_TOL
    if bad.any():
        cancel_ok = np.abs(g64 - r) <= TAU[wl.dtype] * gmag[keep]
        still = bad & ~cancel_ok
        assert not still.any(), ("ulp", int(still.sum()), int(d[still].max()),
                                 g64[still][:4], r[still][:4], gmag[keep][still][:4])
