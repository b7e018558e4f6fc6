"""Fused language-model head loss for GB300 (sm_103a).

The computation lives in libheadloss.so (CUDA kernels behind the C ABI of
include/headloss.h); `headloss` is its thin ctypes binding and `workloads`
the seeded synthetic inputs it is measured on.
"""
from . import headloss, workloads  # noqa: F401
from .headloss import HeadLoss  # noqa: F401

LOSS_BITS = {
    "ce": headloss.HEADLOSS_CE, "z": headloss.HEADLOSS_Z, "dist_ce": headloss.HEADLOSS_DIST_CE,
    "fkl": headloss.HEADLOSS_FKL, "rkl": headloss.HEADLOSS_RKL, "grpo": headloss.HEADLOSS_GRPO,
    "grpo_stats": headloss.HEADLOSS_GRPO_STATS, "entropy": headloss.HEADLOSS_ENTROPY,
}


def flags_of(losses) -> int:
    f = 0
    for name in losses:
        f |= LOSS_BITS[name]
    return f


def headloss_for(wl) -> "HeadLoss":
    """A handle configured for a workload of `workloads.WORKLOADS`."""
    w = dict(wl.weights)
    return HeadLoss(flags_of(wl.losses), headloss.make_weights(**w), wl.temperature,
                    wl.clip_eps, wl.softcap, wl.logits_scale)
