"""Writes two_class_rows.json: hand-written two-class (V = 2) rows with the
oracle's scalars, per-row records, gradient and term magnitudes.

The pages (ServiceNow Fast-LLM issue #507 and PRs #549 / #558 / #568) print
no worked example with values, so the stored values come from the oracle
alone (this script calls nothing else).  tests/test_golden.py pins them
against two-class closed forms (logistic sigmoid / softplus identities)
derived independently of the oracle's log-sum-exp code, and runs the CUDA
library on the same rows.

Inputs are multiples of 1/8 within [-8, 8], so every logit is exact in
bf16, fp16 and fp32; old log-probabilities and advantages are fp32 values.
Run this file to regenerate the fixture.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle as orc  # noqa: E402

BITS = {"ce": orc.CE, "z": orc.Z, "dist_ce": orc.DIST_CE, "fkl": orc.FKL, "rkl": orc.RKL,
        "grpo": orc.GRPO, "grpo_stats": orc.GRPO_STATS, "entropy": orc.ENTROPY}

# Each case: a loss set with its constants and a handful of rows.  Labels mix
# both classes and a masked row (-100); the GRPO rows put the ratio on both
# sides of both clip bounds and inside them, away from the bounds.
CASES = [
    dict(name="ce_z",
         cite="label CE and z-loss: issue #507 Problem; PR #549 Loss coverage",
         losses=["ce", "z"], weights=dict(ce=1.0, z=0.1), grad_scale=1.0,
         temperature=1.0, clip_eps=0.2, softcap=0.0, logits_scale=1.0,
         logits=[[1.5, -0.25], [0.0, 2.0], [3.0, 3.0], [-1.25, 0.5], [4.0, -3.5]],
         labels=[0, 1, -100, 1, 1]),
    dict(name="distillation_T2",
         cite="from-distribution CE, forward and reverse KL with temperature: "
              "PR #549 Loss coverage and Bundled fix",
         losses=["ce", "dist_ce", "fkl", "rkl"],
         weights=dict(ce=1.0, dist_ce=0.25, fkl=0.5, rkl=0.5), grad_scale=1.0,
         temperature=2.0, clip_eps=0.2, softcap=0.0, logits_scale=1.0,
         logits=[[1.5, -0.25], [0.0, 2.0], [-2.0, 1.0], [0.75, 0.75]],
         teacher=[[0.5, 1.0], [2.5, -1.0], [-2.5, 1.5], [0.0, 3.0]],
         labels=[0, 1, 1, -100]),
    dict(name="grpo_stats_entropy",
         cite="GRPO clipped objective, its ratio / clamp / KL / advantage statistics "
              "and entropy: issue #507 Problem; PR #549 Loss coverage",
         losses=["grpo", "grpo_stats", "entropy", "z"],
         weights=dict(grpo=1.0, z=1e-4, entropy=0.3), grad_scale=1.0,
         temperature=1.0, clip_eps=0.2, softcap=0.0, logits_scale=1.0,
         logits=[[1.0, 0.0], [0.0, 1.0], [2.0, -1.0], [-0.5, 0.5], [0.25, 0.0], [1.0, 1.0],
                 [-1.0, 0.5], [0.5, -0.5]],
         labels=[0, 1, 1, 0, 0, -100, 1, 1],
         # ratios about 1.55 (A > 0: clipped), 0.94, 0.95, 0.73 (A < 0: clipped),
         # 1.05, masked, 1.73 (A < 0: unclipped branch), 0.65 (A > 0: unclipped)
         old_logprobs=[-0.75, -0.25, -3.0, -1.0, -0.625, -0.5, -0.75, -0.875],
         advantages=[1.0, -0.5, 1.0, -1.5, 0.75, 2.0, -1.0, 0.5]),
    dict(name="all_in_softcap",
         cite="every loss from one softmax with softcap and logit scaling: issue #507 "
              "Proposed direction; PR #549 Approach and Correctness",
         losses=["ce", "z", "fkl", "grpo", "grpo_stats", "entropy"],
         weights=dict(ce=1.0, z=1e-4, fkl=0.5, grpo=1.0, entropy=0.0), grad_scale=1.0,
         temperature=1.5, clip_eps=0.2, softcap=4.0, logits_scale=0.5,
         logits=[[6.0, -2.0], [-7.5, 1.25], [0.5, 0.625], [3.0, -8.0]],
         teacher=[[2.0, 0.0], [-1.0, 1.0], [0.25, 0.5], [1.5, -1.5]],
         labels=[0, 1, 0, 1],
         old_logprobs=[-0.25, -0.5, -0.875, -5.0],
         advantages=[0.5, -1.0, 1.25, 2.0]),
]


def run_case(c):
    flags = 0
    for name in c["losses"]:
        flags |= BITS[name]
    f32 = lambda v: float(np.float32(v))
    cfg = orc.make_cfg(flags, {k: f32(v) for k, v in c["weights"].items()},
                       temperature=f32(c["temperature"]), clip_eps=f32(c["clip_eps"]),
                       softcap=f32(c["softcap"]), logits_scale=f32(c["logits_scale"]),
                       grad_scale=f32(c["grad_scale"]))
    x = np.array(c["logits"], np.float64)
    lab = np.array(c["labels"], np.int64)
    t = np.array(c["teacher"], np.float64) if "teacher" in c else None
    o = np.array(c["old_logprobs"], np.float32).astype(np.float64) if "old_logprobs" in c else None
    a = np.array(c["advantages"], np.float32).astype(np.float64) if "advantages" in c else None
    scalars, rec, grad, gmag = orc.forward_backward(cfg, x, lab, t, o, a, want_grad=True,
                                                    want_gmag=True, n_threads=1)
    out = dict(c)
    out["expected"] = dict(scalars=scalars.tolist(), records=rec.tolist(), grad=grad.tolist(),
                           gmag=gmag.tolist())
    return out


def main():
    doc = dict(
        what="two-class rows for the monolithic LM-head loss; inputs hand-written, expected "
             "values written by make_golden.py from the fp64 oracle",
        slots=list(orc.SLOTS),
        record_fields=orc.RF,
        cases=[run_case(c) for c in CASES],
    )
    with open(os.path.join(HERE, "two_class_rows.json"), "w") as fh:
        json.dump(doc, fh, indent=1)
        fh.write("\n")


if __name__ == "__main__":
    main()
