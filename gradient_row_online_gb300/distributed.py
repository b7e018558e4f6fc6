"""Combining the sixteen scalars of a data-parallel step across ranks.

Token rows are independent, so each rank runs the fused head loss on its own
rows with no collective on the data path.  The one exchange data parallelism
needs is this: every scalar slot is a mean over the rank's valid rows (or a
count, or a function of means), so the global value follows from one
all-reduce of per-rank sums, second moments and counts.

Gradients: the library normalises each rank's gradient by its own valid-row
count.  For the gradient of the global mean instead, either give every rank
grad_scale * n_valid_local / n_valid_global (see `global_grad_scale`), or
pass the global count as the call's divisor (headloss_forward_backward_ext;
see `global_divisor`): then each rank's gradient is already its share of the
global mean and its loss slots are partial sums that `sum_loss_slots` adds.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

# slot indices (enum headloss_slot)
TOTAL, CE, Z, DIST_CE, FKL, RKL, GRPO, NEW_LOGPROB, RATIO, CLIP_FRAC, KL_K3, ADV_MEAN, \
    ADV_STD, ENTROPY, N_VALID, N_CLIPPED = range(16)
MEAN_SLOTS = (TOTAL, CE, Z, DIST_CE, FKL, RKL, GRPO, NEW_LOGPROB, RATIO, KL_K3, ADV_MEAN,
              ENTROPY)


def allreduce_scalars(scalars: torch.Tensor, group=None) -> torch.Tensor:
    """Global scalars (fp64, 16) from this rank's `scalars` (the 16 floats one
    headloss_forward_backward call wrote), by one all-reduce over `group`."""
    s = scalars.detach().to(torch.float64).reshape(16)
    n = s[N_VALID]
    v = torch.zeros(18, dtype=torch.float64, device=s.device)
    for i in MEAN_SLOTS:
        v[i] = s[i] * n
    v[ADV_STD] = (s[ADV_STD] ** 2 + s[ADV_MEAN] ** 2) * n  # sum of A^2
    v[N_VALID] = n
    v[N_CLIPPED] = s[N_CLIPPED]
    dist.all_reduce(v, op=dist.ReduceOp.SUM, group=group)
    out = torch.zeros(16, dtype=torch.float64, device=s.device)
    N = v[N_VALID]
    out[N_VALID] = N
    out[N_CLIPPED] = v[N_CLIPPED]
    if N > 0:
        for i in MEAN_SLOTS:
            out[i] = v[i] / N
        out[CLIP_FRAC] = v[N_CLIPPED] / N
        var = v[ADV_STD] / N - out[ADV_MEAN] ** 2
        out[ADV_STD] = torch.sqrt(torch.clamp(var, min=0.0))
    return out


def global_grad_scale(n_valid_local: int, grad_scale: float = 1.0, group=None) -> float:
    """The grad_scale that makes this rank's gradient the gradient of the mean
    over all ranks' valid rows (one all-reduce of the counts)."""
    t = torch.tensor([float(n_valid_local)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    total = float(t.item())
    return grad_scale * (n_valid_local / total) if total > 0 else 0.0


# loss slots: partial sums over the global divisor when every rank passes it
LOSS_SLOTS = (TOTAL, CE, Z, DIST_CE, FKL, RKL, GRPO, ENTROPY)


def global_divisor(labels: torch.Tensor, V: int, group=None) -> float:
    """The batch's valid-row count over all ranks (0 <= label < V), by one
    all-reduce: the divisor every rank passes to headloss_forward_backward_ext."""
    n = ((labels >= 0) & (labels < V)).sum().to(torch.float64).reshape(1).cpu()
    dist.all_reduce(n, op=dist.ReduceOp.SUM, group=group)
    return float(n.item())


def sum_loss_slots(scalars: torch.Tensor, group=None) -> torch.Tensor:
    """Global loss slots (fp64, 16; metric slots zero) from this rank's scalars
    of a call made with the global divisor: the loss slots add across ranks."""
    s = scalars.detach().to(torch.float64).reshape(16)
    v = torch.zeros(16, dtype=torch.float64, device=s.device)
    for i in LOSS_SLOTS:
        v[i] = s[i]
    dist.all_reduce(v, op=dist.ReduceOp.SUM, group=group)
    return v
