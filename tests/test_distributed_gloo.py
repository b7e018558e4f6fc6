"""The multi-rank reduction step on CPU: two gloo ranks each hold half of a
batch; their per-rank scalars, combined by one all-reduce, must equal the
scalars of the whole batch, and `global_grad_scale` must turn each rank's
gradient into its share of the whole batch's gradient.  Per-rank scalars
come from the oracle (no GPU here), in fp64."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as orc

ALL = (orc.CE | orc.Z | orc.DIST_CE | orc.FKL | orc.RKL | orc.GRPO | orc.GRPO_STATS |
       orc.ENTROPY)
W = dict(ce=0.9, z=0.3, dist_ce=0.4, fkl=0.6, rkl=0.7, grpo=1.1, entropy=0.5)


def _problem():
    rng = np.random.default_rng(7)
    n, V = 40, 33
    x = rng.normal(0, 3, (n, V))
    t = x + rng.normal(0, 1, (n, V))
    labels = rng.integers(0, V, n).astype(np.int64)
    labels[rng.random(n) < 0.2] = -100
    # old log-probs near the current ones (torch's log_softmax, a library routine)
    lp = torch.log_softmax(torch.from_numpy(x), -1).numpy()
    old = np.where(labels >= 0, lp[np.arange(n), np.maximum(labels, 0)], 0.0)
    old = old + rng.normal(0, 0.3, n)
    adv = rng.normal(0, 1, n)
    return x, labels, t, old, adv


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from gradient_row_online_gb300.distributed import allreduce_scalars, global_grad_scale
        x, labels, t, old, adv = _problem()
        half = slice(rank * 20, (rank + 1) * 20)
        cfg = orc.make_cfg(ALL, W, temperature=1.5, clip_eps=0.2, grad_scale=1.0)
        s, rec, g, _ = orc.forward_backward(cfg, x[half], labels[half], t[half], old[half],
                                            adv[half])
        comb = allreduce_scalars(torch.from_numpy(s).float())
        n_local = int((labels[half] >= 0).sum())
        gs = global_grad_scale(n_local)
        q.put((rank, comb.numpy(), g * gs))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_combine_to_the_whole_batch():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort(key=lambda r: r[0])
    x, labels, t, old, adv = _problem()
    cfg = orc.make_cfg(ALL, W, temperature=1.5, clip_eps=0.2, grad_scale=1.0)
    ref, _, g_ref, _ = orc.forward_backward(cfg, x, labels, t, old, adv)
    for rank, comb, _ in results:
        # scalars travelled as fp32 (the library's output type)
        assert np.allclose(comb, ref, rtol=1e-6, atol=1e-6), (rank, comb, ref)
    # each rank's rescaled gradient is its half of the whole batch's gradient
    g = np.concatenate([results[0][2], results[1][2]])
    assert np.allclose(g, g_ref, rtol=1e-12, atol=1e-15)


def _rank_divisor(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from gradient_row_online_gb300.distributed import global_divisor, sum_loss_slots
        x, labels, t, old, adv = _problem()
        half = slice(rank * 20, (rank + 1) * 20)
        D = global_divisor(torch.from_numpy(labels[half]), x.shape[1])
        cfg = orc.make_cfg(ALL, W, temperature=1.5, clip_eps=0.2, grad_scale=1.0)
        # what a call with divisor D writes: the oracle's per-row records of this
        # rank's rows, with the gradient normalised by D
        rec, g, _ = orc.rows(cfg, x[half], labels[half], t[half], old[half], adv[half], int(D),
                             True, False)
        valid = rec[:, orc.RF["valid"]] > 0
        loss = {1: "ce", 2: "z", 3: "dist_ce", 4: "fkl", 5: "rkl", 6: "grpo", 13: "entropy"}
        s = np.zeros(16)
        for slot, field in loss.items():
            s[slot] = rec[valid, orc.RF[field]].sum() / D
        s[0] = sum(W[f] * s[slot] for slot, f in loss.items())
        q.put((rank, D, sum_loss_slots(torch.from_numpy(s)).numpy(), g))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_with_the_global_divisor():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_divisor, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort(key=lambda r: r[0])
    x, labels, t, old, adv = _problem()
    cfg = orc.make_cfg(ALL, W, temperature=1.5, clip_eps=0.2, grad_scale=1.0)
    ref, _, g_ref, _ = orc.forward_backward(cfg, x, labels, t, old, adv)
    n_total = float(((labels >= 0) & (labels < x.shape[1])).sum())
    for rank, D, sums, _ in results:
        assert D == n_total
        for slot in (0, 1, 2, 3, 4, 5, 6, 13):
            assert np.isclose(sums[slot], ref[slot], rtol=1e-12, atol=1e-12), (slot, sums, ref)
    # each rank's gradient rows are the whole batch's gradient rows, unscaled
    g = np.concatenate([results[0][3], results[1][3]])
    assert np.allclose(g, g_ref, rtol=1e-12, atol=1e-15)

