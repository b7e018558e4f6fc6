"""Seeded synthetic workloads (inputs only -- no loss arithmetic).

The five loss sets the library is measured and checked on.  Each workload
names its losses as strings; the library binding and the oracle map the names
to their own flag bits.  Inputs are drawn with torch generators, one seeded
generator per stream (logits, labels, mask, teacher noise, old-log-prob
noise, advantages), in row chunks so that no fp32 copy of a whole tensor is
ever materialised.

The one input that depends on the logits is the GRPO old-policy log-prob:
"the new policy's label log-prob plus N(0, 0.05^2) noise".  It is produced
here with torch's own log_softmax of the capped / scaled logits, so the
ratios sit near 1 as in a real policy step; it is an input, and both the
library and the oracle receive the same bytes.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int
    V: int
    dtype: torch.dtype
    losses: tuple            # subset of ce, z, dist_ce, fkl, rkl, grpo, grpo_stats, entropy
    weights: dict            # ce, z, dist_ce, fkl, rkl, grpo, entropy, grad_scale
    sigma: float = 3.0       # logits ~ N(0, sigma^2)
    mask_frac: float = 0.05  # rows with label = -100
    teacher_noise: Optional[float] = None  # teacher = student + N(0, noise^2)
    temperature: float = 1.0
    clip_eps: float = 0.2
    softcap: float = 0.0
    logits_scale: float = 1.0
    adv_block: int = 1024    # one advantage per block of tokens (a sequence)
    old_noise: float = 0.05
    seed: int = 0

    @property
    def has_teacher(self) -> bool:
        return any(l in self.losses for l in ("dist_ce", "fkl", "rkl"))

    @property
    def has_grpo(self) -> bool:
        return any(l in self.losses for l in ("grpo", "grpo_stats"))

    @property
    def elem_bytes(self) -> int:
        return torch.tensor([], dtype=self.dtype).element_size()

    def min_bytes_per_row(self) -> int:
        """Algorithmic HBM bytes per token: logits (+ teacher) read once, the
        gradient written once, the int64 label, and the two fp32 GRPO inputs."""
        b = self.V * self.elem_bytes * (3 if self.has_teacher else 2) + 8
        if self.has_grpo:
            b += 8
        return b

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


_W = dict(ce=0.0, z=0.0, dist_ce=0.0, fkl=0.0, rkl=0.0, grpo=0.0, entropy=0.0, grad_scale=1.0)


def _w(**kw):
    d = dict(_W)
    d.update(kw)
    return d


WORKLOADS = {
    # small fp32 case the oracle finishes in seconds
    "tiny_ce_z_fp32": Workload(
        "tiny_ce_z_fp32", 64, 1024, torch.float32, ("ce", "z"), _w(ce=1.0, z=0.1), sigma=2.0,
        mask_frac=0.10),
    "ce_z_bf16": Workload(
        "ce_z_bf16", 8192, 32000, torch.bfloat16, ("ce", "z"), _w(ce=1.0, z=1e-4)),
    "ce_distill_bf16": Workload(
        "ce_distill_bf16", 16384, 128256, torch.bfloat16, ("ce", "fkl", "rkl"),
        _w(ce=1.0, fkl=0.5, rkl=0.5), teacher_noise=1.0, temperature=2.0),
    "grpo_z_entropy_bf16": Workload(
        "grpo_z_entropy_bf16", 32768, 151936, torch.bfloat16,
        ("grpo", "grpo_stats", "z", "entropy"), _w(grpo=1.0, z=1e-4), clip_eps=0.2),
    "all_in_bf16": Workload(
        "all_in_bf16", 65536, 128256, torch.bfloat16,
        ("ce", "z", "fkl", "grpo", "grpo_stats", "entropy"),
        _w(ce=1.0, z=1e-4, fkl=0.5, grpo=1.0), teacher_noise=1.0, temperature=1.5,
        clip_eps=0.2, softcap=30.0, logits_scale=0.5, mask_frac=0.10),
    # the CE + z loss set on fp32 logits at a full-size shape (fp32 is one of
    # the logits dtypes the head loss is validated on)
    "ce_z_fp32": Workload(
        "ce_z_fp32", 8192, 32000, torch.float32, ("ce", "z"), _w(ce=1.0, z=1e-4)),
}

ORDER = ("tiny_ce_z_fp32", "ce_z_bf16", "ce_distill_bf16", "grpo_z_entropy_bf16", "all_in_bf16")
# measured beside the five sets above
EXTRA = ("ce_z_fp32",)


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + stream)
    return g


def make_inputs(wl: Workload, device="cuda", rows: Optional[int] = None,
                chunk_rows: int = 2048) -> dict:
    """Inputs of `wl` (its first `rows` rows if given) on `device`.

    Returns dict(logits, labels, teacher, old_logprobs, advantages); absent
    inputs are None.  Deterministic for a given (workload, device type)."""
    device = torch.device(device)
    N = wl.N if rows is None else min(rows, wl.N)
    V = wl.V
    g_x, g_lab, g_mask = _gen(device, wl.seed, 0), _gen(device, wl.seed, 1), _gen(device, wl.seed, 2)
    g_t, g_old, g_adv = _gen(device, wl.seed, 3), _gen(device, wl.seed, 4), _gen(device, wl.seed, 5)

    logits = torch.empty((N, V), dtype=wl.dtype, device=device)
    teacher = torch.empty((N, V), dtype=wl.dtype, device=device) if wl.has_teacher else None
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        xf = torch.randn((r1 - r0, V), generator=g_x, device=device, dtype=torch.float32)
        xf.mul_(wl.sigma)
        logits[r0:r1].copy_(xf)
        if teacher is not None:
            tf = torch.randn((r1 - r0, V), generator=g_t, device=device, dtype=torch.float32)
            tf.mul_(wl.teacher_noise).add_(logits[r0:r1].float())
            teacher[r0:r1].copy_(tf)
        del xf

    labels = torch.randint(0, V, (N,), generator=g_lab, device=device, dtype=torch.int64)
    mask = torch.rand((N,), generator=g_mask, device=device) < wl.mask_frac
    labels[mask] = -100

    old = adv = None
    if wl.has_grpo:
        old, adv = _grpo_side(wl, logits, labels, g_old, g_adv, chunk_rows)
    return dict(logits=logits, labels=labels, teacher=teacher, old_logprobs=old, advantages=adv)


def _grpo_side(wl, logits, labels, g_old, g_adv, chunk_rows=2048):
    """Per-sequence advantages and old log-probs near the current label
    log-probs (torch's log_softmax of the transformed logits, plus noise)."""
    N = logits.shape[0]
    device = logits.device
    nblk = (N + wl.adv_block - 1) // wl.adv_block
    adv = torch.randn((nblk,), generator=g_adv, device=device, dtype=torch.float32)
    adv = adv.repeat_interleave(wl.adv_block)[:N].contiguous()
    old = torch.empty((N,), dtype=torch.float32, device=device)
    noise = torch.randn((N,), generator=g_old, device=device, dtype=torch.float32)
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        z = logits[r0:r1].float()
        if wl.softcap > 0:
            z = torch.tanh(z / wl.softcap) * wl.softcap
        z = z * wl.logits_scale
        lp = torch.log_softmax(z, dim=-1)
        lab = labels[r0:r1]
        picked = lp.gather(1, lab.clamp(min=0)[:, None])[:, 0]
        old[r0:r1] = torch.where(lab >= 0, picked + wl.old_noise * noise[r0:r1],
                                 torch.zeros_like(picked))
        del z, lp
    return old, adv


def make_structured_inputs(wl: Workload, device="cuda") -> dict:
    """Rows whose shape stresses the online statistics (small cases only).

    Row r takes pattern r % 6 on top of N(0, sigma^2) noise, for the student
    and (with its own pattern) the teacher: 0 an ascending ramp -20 -> +40
    along the row (the maximum comes last), 1 the descending ramp, 2 a +300
    offset, 3 one spike of +60 at a random column, 4 the noise alone, 5 the
    noise scaled by 8.  Labels, mask and GRPO side inputs as in make_inputs."""
    device = torch.device(device)
    N, V = wl.N, wl.V
    g_x, g_lab, g_mask = _gen(device, wl.seed, 0), _gen(device, wl.seed, 1), _gen(device, wl.seed, 2)
    g_t, g_old, g_adv = _gen(device, wl.seed, 3), _gen(device, wl.seed, 4), _gen(device, wl.seed, 5)
    g_pos = _gen(device, wl.seed, 6)
    j = torch.arange(V, device=device, dtype=torch.float32) / max(V - 1, 1)
    kind = torch.arange(N, device=device) % 6
    spike = torch.randint(0, V, (N,), generator=g_pos, device=device)

    def shaped(base, flip):
        out = base.clone()
        ramp = -20.0 + 60.0 * (1.0 - j if flip else j)
        out[kind == 0] += ramp
        out[kind == 1] += -20.0 + 60.0 * (j if flip else 1.0 - j)
        out[kind == 2] += 300.0
        rows = torch.nonzero(kind == 3)[:, 0]
        out[rows, spike[rows]] += 60.0
        out[kind == 5] *= 8.0
        return out

    xf = torch.randn((N, V), generator=g_x, device=device, dtype=torch.float32) * wl.sigma
    logits = shaped(xf, False).to(wl.dtype)
    teacher = None
    if wl.has_teacher:
        tf = torch.randn((N, V), generator=g_t, device=device, dtype=torch.float32)
        teacher = shaped(tf * wl.teacher_noise + xf, True).to(wl.dtype)
    labels = torch.randint(0, V, (N,), generator=g_lab, device=device, dtype=torch.int64)
    mask = torch.rand((N,), generator=g_mask, device=device) < wl.mask_frac
    labels[mask] = -100
    old = adv = None
    if wl.has_grpo:
        old, adv = _grpo_side(wl, logits, labels, g_old, g_adv)
    return dict(logits=logits, labels=labels, teacher=teacher, old_logprobs=old, advantages=adv)
