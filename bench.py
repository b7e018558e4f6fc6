"""Benchmark of the fused LM-head loss (one JSON line on stdout).

A step is one headloss_forward_backward call over the whole batch of the
workload (default: the all-in combined loss set, 65536 tokens x 128256 vocab,
bf16): every loss scalar plus the one combined logits gradient.  Inputs are
seeded synthetic tensors larger than L2, resident in HBM before timing.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Under torchrun each rank runs its own batch on its own GPU (rows are
independent: weak scaling, no data-path collective); the time is the max over
ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import glob
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused head-loss tokens/s and HBM GB/s (% of GB300 peak) per loss set, 1 GPU"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all_in_bf16")
    ap.add_argument("--rows", type=int, default=0,
                    help="use only the first ROWS tokens of the workload (profiling cases)")
    ap.add_argument("--plan", default="",
                    help="pin the launch plan, e.g. kernel=2,stages=2,threads=512,chunk_words=4 "
                         "(profiling; default: the library's planner)")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-loss-sets", action="store_true")
    ap.add_argument("--no-per-loss", action="store_true",
                    help="skip the per-loss-loop comparison")
    ap.add_argument("--no-lmhead", action="store_true",
                    help="skip the LM-head GEMM leg (tensor cores, beside torch.matmul)")
    ap.add_argument("--lmhead-shape", default="8192,4096,128256",
                    help="N,D,V of the LM-head GEMM leg")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="wall time the CPU-baseline sample is sized for")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0


def tensor_peak():
    """Dense bf16 tensor throughput (TFLOP/s) for a kernel timed alone: the
    measured burst figure, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_hash():
    """Hash of the loss kernels' sources (hl_* and headloss_* files, comments
    and blank lines stripped, so an edit to a comment does not mark recorded
    counters stale; the LM-head GEMM's source is not part of the loss path)."""
    h = hashlib.sha256()
    for fn in sorted(glob.glob(os.path.join(ROOT, "gradient_row_online_gb300", "csrc", "*"))):
        if not fn.endswith((".cu", ".cuh", ".h")):
            continue
        if not os.path.basename(fn).startswith(("hl_", "headloss_")):
            continue
        with open(fn) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        code = "\n".join(l.rstrip() for l in src.splitlines() if l.strip())
        h.update(os.path.basename(fn).encode())
        h.update(code.encode())
    return h.hexdigest()[:16]


def kernel_label(plan, wl):
    """The dominant kernel of one call, as the roofline entry names it."""
    if plan["kernel"] == "stream":
        k = "hl::stream_kernel16"
    else:
        k = "hl::rows_kernel" if wl.dtype == torch.float32 else "hl::rows_kernel16"
    return (f"{k} (timed as the whole call: valid-row count + row kernel + finalize; the "
            f"row kernel is >99.5% of the call's device time in the ncu launch list)")


def recorded_traffic(workload):
    """DRAM bytes per launch of the row kernel from a committed ncu summary,
    if it was taken on the current kernel sources (else None)."""
    fn = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(fn) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(workload)
    if not ent or ent.get("kernel_source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, interval_ms=100):
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.path = None
        self.start_at = 0  # file offset where the timed region's samples begin

    def __enter__(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=self.out, stderr=subprocess.DEVNULL)
            # wait (at most 3 s) for the first sample, so that the samples
            # counted are the ones taken while the timed region runs
            deadline = time.time() + 3.0
            while time.time() < deadline and self.proc.poll() is None:
                if os.path.getsize(self.path) > 0:
                    break
                time.sleep(0.005)
            self.start_at = os.path.getsize(self.path)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

        def parse(lines):
            out = []
            for line in lines:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm, mx = float(parts[1]), float(parts[2])
                except ValueError:
                    continue
                out.append((sm, mx, {n for n, v in zip(names, parts[5:9])
                                     if v.lower() == "active"}))
            return out

        with open(self.path) as f:
            text = f.read()
        os.unlink(self.path)
        inside = parse(text[self.start_at:].splitlines())
        # a region shorter than the sampling interval may hold no sample: then
        # the last one taken before it stands in, and "samples" says 0
        use = inside or parse(text[:self.start_at].splitlines())[-1:]
        if not use:
            return None
        return {"sm_mhz": statistics.median(u[0] for u in use),
                "sm_max_mhz": max(u[1] for u in use),
                "reasons": sorted(set().union(*(u[2] for u in use))),
                "samples": len(inside), "interval_ms": self.interval_ms}


# ------------------------------------------------------------- our arm

def time_calls(fn, stream, steps):
    """Per-call durations (ms) by CUDA events on `stream`, synchronised around."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def run_ours(args, rank, world, local):
    import gradient_row_online_gb300 as pkg
    from gradient_row_online_gb300 import headloss as hlb
    from gradient_row_online_gb300 import workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    wl = W.WORKLOADS[args.workload].replace(seed=rank)  # each rank its own batch
    if args.rows:
        wl = wl.replace(N=min(args.rows, wl.N))
    hlb.load_library()
    h = pkg.headloss_for(wl)
    if args.plan:
        h.force_plan(**{k: int(v) for k, v in (kv.split("=") for kv in args.plan.split(","))})
    inp = W.make_inputs(wl, dev)
    grad = torch.empty_like(inp["logits"])
    out = torch.empty(16, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    dcode = hlb.dtype_code(wl.dtype)

    def step():
        hlb.headloss_forward_backward(h.h, inp["logits"], wl.N, wl.V, dcode, inp["labels"],
                                      inp["teacher"], inp["old_logprobs"], inp["advantages"],
                                      grad, out, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        per_call = []
        # per-call events inside the timed region (same stream)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in evs:
            a.record(stream)
            step()
            b.record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        total_ms = t0.elapsed_time(t1)
        per_call = [a.elapsed_time(b) for a, b in evs]
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([total_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
        dist.barrier()
    scal = out.double().cpu().numpy()
    err = h.device_error()
    if err != hlb.HEADLOSS_OK:
        raise RuntimeError(hlb.STATUS[err])

    ms_per_step = total_ms / args.steps
    tokens_per_s = wl.N * world * args.steps / (total_ms / 1e3)
    bytes_per_launch = wl.min_bytes_per_row() * wl.N
    call_ms = statistics.mean(per_call)
    achieved = bytes_per_launch / (call_ms / 1e3) / 1e9
    peak, peak_kind = peaks()
    plan = h.plan(wl.V, dcode)
    clocks = clk.summary()

    line = {
        "metric": METRIC,
        "value": tokens_per_s,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded N(0,3^2) logits; see workloads.py)",
        "config": {
            "workload": wl.name, "N_tokens": wl.N, "V": wl.V, "io_dtype": str(wl.dtype)[6:],
            "losses": list(wl.losses), "temperature": wl.temperature, "softcap": wl.softcap,
            "logits_scale": wl.logits_scale, "clip_eps": wl.clip_eps,
            "parallelism": f"rows sharded over {world} GPU(s), no collective",
            "l2": f"inputs larger than L2 ({bytes_per_launch / 1e9:.1f} GB per step)",
            "plan": plan,
        },
        "roofline": {
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_kind": peak_kind,
            "frac_of_nominal_8000": achieved / 8000.0,
            # the recorded counters describe the full workload in its automatic plan
            "traffic": (recorded_traffic(wl.name)
                        if wl.N == W.WORKLOADS[args.workload].N and not args.plan else None),
            "algorithmic_bytes_per_launch": bytes_per_launch,
            "kernel": kernel_label(plan, wl),
        },
        "gpu_launches": args.steps * hlb.headloss_launches_per_call(),
        "clocks": clocks,
        "scalars": {n: float(v) for n, v in zip(hlb.SLOTS, scal)},
    }
    if not args.no_per_loss and world == 1:
        line["per_loss_loop"] = per_loss_loop(wl, inp, grad, dev)
    # the end-to-end steps next, on the main workload's tensors, before the
    # other legs' allocations (the host link's speed varies from run to run;
    # this keeps the other legs out of it)
    if not args.no_e2e:
        del grad
        line["e2e"] = e2e(wl, h, inp, args, dev, world)
    if not args.no_loss_sets and world == 1:
        line["loss_sets"] = loss_sets(args, dev, exclude=wl.name, peak=peak)
    if not args.no_lmhead and world == 1:
        line["lm_head_gemm"] = lm_head_gemm(args, dev)
        line["lm_head_loss"] = lm_head_loss(args, dev, peak)
        line["lm_head_loss_distill"] = lm_head_loss_distill(args, dev, peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, inp, args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return line


def loss_sets(args, dev, exclude, peak):
    """Short measurement of the other full-size loss sets (same call, same clock)."""
    import gradient_row_online_gb300 as pkg
    from gradient_row_online_gb300 import headloss as hlb
    from gradient_row_online_gb300 import workloads as W

    res = {}
    for name in W.ORDER[1:] + W.EXTRA:
        if name == exclude:
            continue
        wl = W.WORKLOADS[name]
        inp = W.make_inputs(wl, dev)
        g = torch.empty_like(inp["logits"])
        out = torch.empty(16, dtype=torch.float32, device=dev)
        h = pkg.headloss_for(wl)
        s = torch.cuda.current_stream(dev)
        fn = lambda: h(inp["logits"], inp["labels"], inp["teacher"], inp["old_logprobs"],
                       inp["advantages"], g, out, s)
        for _ in range(3):
            fn()
        ms = statistics.mean(time_calls(fn, s, 10))
        gbs = wl.min_bytes_per_row() * wl.N / (ms / 1e3) / 1e9
        res[name] = {"tokens_per_s": wl.N / (ms / 1e3), "ms_per_call": ms, "gbs": gbs,
                     "frac_of_measured_peak": gbs / peak, "plan": h.plan(wl.V, hlb.dtype_code(wl.dtype))}
        del inp, g
        h.close()
        torch.cuda.empty_cache()
    return res


def per_loss_loop(wl, inp, grad, dev, steps=5):
    """The status quo the pages replace: one call per loss (each re-reads the
    row and recomputes its softmax), gradients accumulated into one buffer,
    against the one fused call.  Same kernels; only the flag sets differ."""
    import gradient_row_online_gb300 as pkg
    from gradient_row_online_gb300 import headloss as hlb

    s = torch.cuda.current_stream(dev)
    fused = pkg.headloss_for(wl)
    out = torch.empty(16, dtype=torch.float32, device=dev)
    args = (inp["logits"], inp["labels"], inp["teacher"], inp["old_logprobs"], inp["advantages"])
    wkey = {"ce": "ce", "z": "z", "dist_ce": "dist_ce", "fkl": "fkl", "rkl": "rkl",
            "grpo": "grpo", "entropy": "entropy"}
    calls = []  # (handle, writes a gradient)
    for name in wl.losses:
        w = {k: 0.0 for k in ("ce", "z", "dist_ce", "fkl", "rkl", "grpo", "entropy")}
        w["grad_scale"] = wl.weights["grad_scale"]
        bearing = name in wkey and wl.weights.get(wkey[name], 0.0) != 0.0
        if name in wkey:
            w[wkey[name]] = wl.weights.get(wkey[name], 0.0)
        hd = pkg.HeadLoss(pkg.flags_of((name,)), hlb.make_weights(**w), wl.temperature,
                          wl.clip_eps, wl.softcap, wl.logits_scale)
        calls.append((hd, bearing))
    n_bearing = sum(1 for _, b in calls if b)
    extra = [torch.empty_like(grad) for _ in range(max(0, n_bearing - 1))]

    def loop():
        first = True
        k = 0
        for hd, bearing in calls:
            if not bearing:
                hd(*args, None, out, s)
            elif first:
                hd(*args, grad, out, s)
                first = False
            else:
                hd(*args, extra[k], out, s)
                grad.add_(extra[k])
                k += 1

    f = lambda: fused(*args, grad, out, s)
    for fn in (f, loop):
        fn()
    ms_fused = statistics.mean(time_calls(f, s, steps))
    ms_loop = statistics.mean(time_calls(loop, s, steps))
    for hd, _ in calls:
        hd.close()
    fused.close()
    del extra
    torch.cuda.empty_cache()
    return {"workload": wl.name, "losses": list(wl.losses), "fused_ms": ms_fused,
            "per_loss_ms": ms_loop, "speedup": ms_loop / ms_fused, "calls_in_loop": len(calls),
            "gradient_writes_in_loop": n_bearing}


def lm_head_gemm(args, dev, steps=10):
    """The LM-head GEMM in front of the loss (tcgen05, TMEM, TMA) with its
    per-tile row statistics, timed beside torch.matmul (cuBLAS) on the same
    bf16 operands; tensor-pipe roofline against the measured bf16 peak."""
    from gradient_row_online_gb300 import headloss as hlb

    N, D, V = (int(v) for v in args.lmhead_shape.split(","))
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    hid = (torch.randn(N, D, generator=g, device=dev) * 0.5).to(torch.bfloat16)
    wt = (torch.randn(V, D, generator=g, device=dev) * (1.0 / D) ** 0.5).to(torch.bfloat16)
    out = torch.empty(N, V, dtype=torch.bfloat16, device=dev)
    st = torch.empty(N, V // 256, 2, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.current_stream(dev)
    ours = lambda: hlb.headloss_lmhead_logits(hid, wt, N, D, V, out, st, err, s)
    ref = lambda: torch.matmul(hid, wt.T)
    for fn in (ours, ref, ours, ref, ours, ref):
        fn()
    ms = statistics.mean(time_calls(ours, s, steps))
    ms_ref = statistics.mean(time_calls(ref, s, steps))
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError("LM-head GEMM: a bounded wait gave up")
    flops = 2.0 * N * D * V
    peak, kind = tensor_peak()
    tf = flops / (ms / 1e3) / 1e12
    res = {"shape": {"N": N, "D": D, "V": V}, "ms": ms, "tflops": tf,
           "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                        "frac": tf / peak, "peak_kind": kind + " (bf16 burst)"},
           "torch_matmul_ms": ms_ref, "torch_matmul_tflops": flops / (ms_ref / 1e3) / 1e12,
           "vs_torch": ms_ref / ms,
           "outputs": "bf16 logits + per-(row, 256-column tile) fp32 (max, sum exp)"}
    del hid, wt, out, st
    torch.cuda.empty_cache()
    return res


def host_link_bandwidth(dev, gib=2, reps=3):
    """Pinned host <-> device copy bandwidth of this machine (GB/s), one direction
    at a time and both at once, best of `reps` copies of `gib` GiB."""
    n = gib << 30
    hb = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    hb2 = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    db = torch.empty(n, dtype=torch.uint8, device=dev)
    db2 = torch.empty(n, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            best = min(best, time.perf_counter() - t0)
        return best

    def both():
        with torch.cuda.stream(s1):
            db.copy_(hb, non_blocking=True)
        with torch.cuda.stream(s2):
            hb2.copy_(db2, non_blocking=True)

    t_h2d = timed(lambda: db.copy_(hb, non_blocking=True))
    t_d2h = timed(lambda: hb2.copy_(db2, non_blocking=True))
    t_both = timed(both)
    del hb, hb2, db, db2
    torch.cuda.empty_cache()
    return {"h2d_gbs": n / t_h2d / 1e9, "d2h_gbs": n / t_d2h / 1e9,
            "both_directions_gbs": 2 * n / t_both / 1e9,
            "how": f"pinned {gib} GiB copies, best of {reps}, wall clock around a synchronize"}


def lm_head_loss_distill(args, dev, peak, steps=6):
    """The fused LM head with a teacher: the student's GEMM emits its per-tile
    records and sums at the temperature, the teacher's GEMM its records, and
    the loss makes one read of both logits and one write of the gradient per
    row (headloss_forward_backward_rowstats), against the two GEMMs plus the
    two-pass call on their logits.  Loss set: the all-in set (CE, z, forward KL
    at T 1.5, GRPO with statistics, entropy; softcap 30, scale 0.5); the
    single-pass kernel's HBM roofline beside."""
    import gradient_row_online_gb300 as pkg
    from gradient_row_online_gb300 import headloss as hlb
    import torch.nn.functional as F

    N, D, V = (int(v) for v in args.lmhead_shape.split(","))
    T, softcap, scale = 1.5, 30.0, 0.5
    g = torch.Generator(device=dev)
    g.manual_seed(2)
    hid = torch.randn(N, D, generator=g, device=dev).to(torch.bfloat16)
    wt = (torch.randn(V, D, generator=g, device=dev) * (9.0 / D) ** 0.5).to(torch.bfloat16)
    # the teacher: the student's weights plus a perturbation (logit noise ~1)
    wt_t = (wt.float() + torch.randn(V, D, generator=g, device=dev) * (1.0 / D) ** 0.5).to(
        torch.bfloat16)
    labels = torch.randint(0, V, (N,), generator=g, device=dev)
    labels[torch.rand(N, generator=g, device=dev) < 0.1] = -100
    adv = torch.randn(N // 1024 + 1, generator=g, device=dev).repeat_interleave(1024)[:N].contiguous()
    logits = torch.empty(N, V, dtype=torch.bfloat16, device=dev)
    tlog = torch.empty_like(logits)
    grad = torch.empty_like(logits)
    NT = V // 256
    rs = torch.empty(N, NT, 4, device=dev)
    rsT = torch.empty(N, NT, device=dev)
    trs = torch.empty(N, NT, 4, device=dev)
    st2 = torch.empty(N, NT, 2, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty(16, device=dev)
    losses = ("ce", "z", "fkl", "grpo", "grpo_stats", "entropy")
    h = pkg.HeadLoss(pkg.flags_of(losses), hlb.make_weights(ce=1.0, z=1e-4, fkl=0.5, grpo=1.0),
                     T, 0.2, softcap, scale)
    s = torch.cuda.current_stream(dev)
    hlb.headloss_lmhead_logits(hid, wt, N, D, V, logits, st2, err, s)
    with torch.no_grad():
        z = scale * softcap * torch.tanh(logits.float() / softcap)
        lp = F.log_softmax(z, -1).gather(1, labels.clamp(min=0)[:, None])[:, 0]
        old = (lp + 0.05 * torch.randn(N, generator=g, device=dev)).contiguous()
        del z, lp
    dcode = hlb.HEADLOSS_BF16

    def gemms_rs():
        hlb.headloss_lmhead_logits_rowstats(hid, wt, N, D, V, softcap, scale, logits, rs, err, s,
                                            temperature=T, row_stats_t=rsT)
        hlb.headloss_lmhead_logits_rowstats(hid, wt_t, N, D, V, 0.0, 1.0 / T, tlog, trs, err, s)

    def loss_rs():
        hlb.headloss_forward_backward_rowstats(h.h, logits, N, V, dcode, labels, old, adv, rs,
                                               grad, out, s, teacher=tlog, row_stats_t=rsT,
                                               teacher_stats=trs)

    def gemms_plain():
        hlb.headloss_lmhead_logits(hid, wt, N, D, V, logits, st2, err, s)
        hlb.headloss_lmhead_logits(hid, wt_t, N, D, V, tlog, st2, err, s)

    def loss_2pass():
        hlb.headloss_forward_backward(h.h, logits, N, V, dcode, labels, tlog, old, adv, grad,
                                      out, s)

    fused = lambda: (gemms_rs(), loss_rs())
    separate = lambda: (gemms_plain(), loss_2pass())
    for fn in (fused, separate, fused, separate):
        fn()
    t_fused = statistics.mean(time_calls(fused, s, steps))
    t_sep = statistics.mean(time_calls(separate, s, steps))
    gemms_rs()
    t_loss1 = statistics.mean(time_calls(loss_rs, s, steps))
    gemms_plain()
    t_loss2 = statistics.mean(time_calls(loss_2pass, s, steps))
    torch.cuda.synchronize()
    if int(err.item()) != 0 or h.device_error() != hlb.HEADLOSS_OK:
        raise RuntimeError("LM-head distillation leg: device error")
    bytes_min = N * V * 2 * 3 + N * 16
    gbs = bytes_min / (t_loss1 / 1e3) / 1e9
    res = {"shape": {"N": N, "D": D, "V": V}, "losses": list(losses), "temperature": T,
           "softcap": softcap, "logits_scale": scale,
           "fused_ms": t_fused, "separate_ms": t_sep, "speedup": t_sep / t_fused,
           "loss_one_pass_ms": t_loss1, "loss_two_pass_ms": t_loss2,
           "loss_one_pass_roofline": {"bound": "hbm", "achieved": gbs, "peak": peak,
                                      "unit": "GB/s", "frac": gbs / peak,
                                      "algorithmic_bytes": bytes_min,
                                      "bytes_with_row_stats": bytes_min + N * NT * 36},
           "loss_two_pass_plan": h.plan(V, dcode)}
    h.close()
    del hid, wt, wt_t, logits, tlog, grad, rs, rsT, trs, st2
    torch.cuda.empty_cache()
    return res


def lm_head_loss(args, dev, peak, steps=10):
    """The fused LM head: the GEMM emits each tile's first-pass record of the
    loss (headloss_lmhead_logits_rowstats) and the loss makes one read and one
    write per row (headloss_forward_backward_rowstats), against the GEMM plus
    the two-pass call on its logits.  Loss set: the all-in set's label-based
    losses (CE, z, GRPO with statistics, entropy metric; softcap 30, scale
    0.5); the one-pass loss kernel's HBM roofline beside."""
    import gradient_row_online_gb300 as pkg
    from gradient_row_online_gb300 import headloss as hlb
    import torch.nn.functional as F

    N, D, V = (int(v) for v in args.lmhead_shape.split(","))
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    hid = torch.randn(N, D, generator=g, device=dev).to(torch.bfloat16)
    wt = (torch.randn(V, D, generator=g, device=dev) * (9.0 / D) ** 0.5).to(torch.bfloat16)
    labels = torch.randint(0, V, (N,), generator=g, device=dev)
    labels[torch.rand(N, generator=g, device=dev) < 0.1] = -100
    adv = torch.randn(N // 1024 + 1, generator=g, device=dev).repeat_interleave(1024)[:N].contiguous()
    logits = torch.empty(N, V, dtype=torch.bfloat16, device=dev)
    grad = torch.empty_like(logits)
    rs = torch.empty(N, V // 256, 4, device=dev)
    st2 = torch.empty(N, V // 256, 2, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty(16, device=dev)
    softcap, scale = 30.0, 0.5
    losses = ("ce", "z", "grpo", "grpo_stats", "entropy")
    h = pkg.HeadLoss(pkg.flags_of(losses), hlb.make_weights(ce=1.0, z=1e-4, grpo=1.0), 1.0, 0.2,
                     softcap, scale)
    s = torch.cuda.current_stream(dev)
    hlb.headloss_lmhead_logits(hid, wt, N, D, V, logits, st2, err, s)
    with torch.no_grad():
        z = scale * softcap * torch.tanh(logits.float() / softcap)
        lp = F.log_softmax(z, -1).gather(1, labels.clamp(min=0)[:, None])[:, 0]
        old = (lp + 0.05 * torch.randn(N, generator=g, device=dev)).contiguous()
        del z, lp
    dcode = hlb.HEADLOSS_BF16

    def gemm_rs():
        hlb.headloss_lmhead_logits_rowstats(hid, wt, N, D, V, softcap, scale, logits, rs, err, s)

    def loss_rs():
        hlb.headloss_forward_backward_rowstats(h.h, logits, N, V, dcode, labels, old, adv, rs,
                                               grad, out, s)

    def gemm_plain():
        hlb.headloss_lmhead_logits(hid, wt, N, D, V, logits, st2, err, s)

    def loss_2pass():
        hlb.headloss_forward_backward(h.h, logits, N, V, dcode, labels, None, old, adv, grad,
                                      out, s)

    fused = lambda: (gemm_rs(), loss_rs())
    separate = lambda: (gemm_plain(), loss_2pass())
    for fn in (fused, separate, fused, separate, fused, separate):
        fn()
    t_fused = statistics.mean(time_calls(fused, s, steps))
    t_sep = statistics.mean(time_calls(separate, s, steps))
    gemm_rs()
    t_loss1 = statistics.mean(time_calls(loss_rs, s, steps))
    gemm_plain()
    t_loss2 = statistics.mean(time_calls(loss_2pass, s, steps))
    torch.cuda.synchronize()
    if int(err.item()) != 0 or h.device_error() != hlb.HEADLOSS_OK:
        raise RuntimeError("LM-head loss leg: device error")
    bytes_1 = N * V * 2 * 2 + N * (V // 256) * 16 + N * 16
    bytes_min = N * V * 2 * 2 + N * 16
    gbs = bytes_min / (t_loss1 / 1e3) / 1e9
    res = {"shape": {"N": N, "D": D, "V": V}, "losses": list(losses), "softcap": softcap,
           "logits_scale": scale,
           "fused_ms": t_fused, "separate_ms": t_sep, "speedup": t_sep / t_fused,
           "loss_one_pass_ms": t_loss1, "loss_two_pass_ms": t_loss2,
           "loss_one_pass_roofline": {"bound": "hbm", "achieved": gbs, "peak": peak,
                                      "unit": "GB/s", "frac": gbs / peak,
                                      "algorithmic_bytes": bytes_min,
                                      "bytes_with_row_stats": bytes_1},
           "loss_two_pass_plan": h.plan(V, dcode)}
    h.close()
    del hid, wt, logits, grad, rs, st2
    torch.cuda.empty_cache()
    return res


def e2e(wl, h, inp, args, dev, world):
    """The same metric through the public call with pinned HOST buffers: every
    step copies its inputs host->device and reads its gradient and scalars
    back.  Steps are pipelined over two device buffer sets on three streams
    (copy in, compute, copy out), so one step's copies overlap another's
    compute; the timed region spans the first copy in to the last copy out."""
    from gradient_row_online_gb300 import headloss as hlb

    names = ["logits", "labels", "teacher", "old_logprobs", "advantages"]
    # pinned host memory: the inputs and two gradient buffers, per rank (71 GB
    # for the all-in batch); the rows are cut, if need be, until every local
    # rank's buffers fit in 70% of the host's available memory (several ranks
    # on one host), and the line reports the rows used
    per_row = sum(inp[k][0].numel() * inp[k].element_size() for k in names
                  if inp[k] is not None) + 2 * inp["logits"][0].numel() * inp["logits"].element_size()
    rows = wl.N
    try:
        with open("/proc/meminfo") as f:
            avail = next(int(l.split()[1]) * 1024 for l in f if l.startswith("MemAvailable:"))
        local = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
        fit = int(0.7 * avail / max(1, local) / per_row)
        if fit < rows:
            rows = max(1024, fit // 1024 * 1024)
    except (OSError, StopIteration, ValueError):
        pass
    if rows < wl.N:
        inp = {k: (None if inp[k] is None else inp[k][:rows]) for k in inp}
        wl = wl.replace(N=rows)
    host = {k: (None if inp[k] is None else torch.empty(inp[k].shape, dtype=inp[k].dtype,
                                                        pin_memory=True)) for k in names}
    for k in names:
        if host[k] is not None:
            host[k].copy_(inp[k])
    # two device sets: the bench's own input tensors and one more
    dsets = [inp, {k: (None if inp[k] is None else torch.empty_like(inp[k])) for k in names}]
    d_grad = [torch.empty_like(inp["logits"]) for _ in range(2)]
    d_out = [torch.empty(16, dtype=torch.float32, device=dev) for _ in range(2)]
    h_grad = [torch.empty(inp["logits"].shape, dtype=inp["logits"].dtype, pin_memory=True)
              for _ in range(2)]
    h_out = [torch.empty(16, dtype=torch.float32, pin_memory=True) for _ in range(2)]
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()
    in_done, cmp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    h2d = sum(host[k].numel() * host[k].element_size() for k in names if host[k] is not None)
    d2h = h_grad[0].numel() * h_grad[0].element_size() + 64
    dcode = hlb.dtype_code(wl.dtype)
    used = [False, False]

    def step(k):
        b = k % 2
        d = dsets[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(cmp_done[b])  # the inputs of buffer set b are free
            for name in names:
                if host[name] is not None:
                    d[name].copy_(host[name], non_blocking=True)
            in_done[b].record(s_in)
        s_cmp.wait_event(in_done[b])
        if used[b]:
            s_cmp.wait_event(out_done[b])  # the gradient of set b has been read back
        hlb.headloss_forward_backward(h.h, d["logits"], wl.N, wl.V, dcode, d["labels"],
                                      d["teacher"], d["old_logprobs"], d["advantages"],
                                      d_grad[b], d_out[b], s_cmp)
        cmp_done[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(cmp_done[b])
            h_grad[b].copy_(d_grad[b], non_blocking=True)
            h_out[b].copy_(d_out[b], non_blocking=True)
            out_done[b].record(s_out)
        used[b] = True

    link = host_link_bandwidth(dev)
    step(0)
    step(1)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    n = max(2, args.e2e_steps)
    t0.record(s_in)
    for k in range(n):
        step(k)
    s_in.wait_stream(s_out)
    t1.record(s_in)
    torch.cuda.synchronize()
    total = t0.elapsed_time(t1)
    del dsets[1], d_grad, h_grad
    # the host link bounds a step at its copies: host-to-device and
    # device-to-host run on separate copy engines and overlap
    bound_ms = 1e3 * max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9))
    return {"value": wl.N * world * n / (total / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "rows_per_rank": wl.N,
            "ms_per_step": total / n, "pipelined": "2 buffer sets, copy-in / compute / copy-out streams",
            "link": link, "link_bound_ms_per_step": bound_ms,
            "frac_of_link_bound": bound_ms / (total / n)}


def cpu_seconds(wl, x, lab, t, old, adv, n_valid, threads):
    import oracle as orc
    from tests import _harness as H
    cfg = H.oracle_cfg(wl)
    t0 = time.perf_counter()
    orc.rows(cfg, x, lab, t, old, adv, n_valid, True, False, threads)
    return time.perf_counter() - t0


def cpu_baseline(wl, inp, seconds, reps=1):
    """The fp64 oracle, as it stands, on this host's cores, on a bounded row
    sample of the same workload (rows sized for about `seconds` of wall time)."""
    import numpy as np

    import oracle as orc
    from tests import _harness as H

    cores = len(os.sched_getaffinity(0))
    n_valid = orc.count_valid(H.host_i64(inp["labels"]), inp["labels"].shape[0])

    def sample(r):
        pick = lambda k: None if inp[k] is None else inp[k][:r]
        return (H.host64(pick("logits")), H.host_i64(pick("labels")), H.host64(pick("teacher")),
                H.host64(pick("old_logprobs")), H.host64(pick("advantages")))

    probe = min(wl.N, max(8 * cores, 64))
    s = sample(probe)
    dt = cpu_seconds(wl, *s, n_valid, cores)
    rows = int(min(wl.N, max(probe, probe * seconds / max(dt, 1e-6))))
    s = sample(rows)
    dt = cpu_seconds(wl, *s, n_valid, cores)
    # the same oracle on one core, over a smaller sample (about a tenth of the time)
    rows1 = int(min(rows, max(8, rows / cores / 10)))
    dt1 = cpu_seconds(wl, *sample(rows1), n_valid, 1)
    return {"value": rows / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {rows} of {wl.N} rows of {wl.name} (gradient + all scalars, fp64, "
                      f"{cores} OpenMP threads), {dt:.1f} s",
            "one_core": {"value": rows1 / dt1, "unit": "tokens/s",
                         "sample": f"first {rows1} rows, 1 thread, {dt1:.1f} s"}}


# ---------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    """The oracle as the reference arm: fp64 CPU, bounded row sample per step."""
    import oracle as orc
    from gradient_row_online_gb300 import workloads as W
    from tests import _harness as H

    wl = W.WORKLOADS[args.workload]
    cores = len(os.sched_getaffinity(0))
    # size one step: probe, then rows for ~(150 s / (steps + warmup)) per step
    budget = max(1.0, 150.0 / (args.steps + max(3, args.warmup)))
    probe = 16
    inp = W.make_inputs(wl, "cpu", rows=probe)
    cfg = H.oracle_cfg(wl)
    nv = orc.count_valid(H.host_i64(inp["labels"]), probe)
    args_h = lambda d: (H.host64(d["logits"]), H.host_i64(d["labels"]), H.host64(d["teacher"]),
                        H.host64(d["old_logprobs"]), H.host64(d["advantages"]))
    t0 = time.perf_counter()
    orc.rows(cfg, *args_h(inp), nv, True, False, cores)
    dt = time.perf_counter() - t0
    rows = int(max(probe, min(wl.N, probe * budget / max(dt, 1e-6))))
    inp = W.make_inputs(wl, "cpu", rows=rows)
    a = args_h(inp)
    nv = orc.count_valid(a[1], rows)
    for _ in range(max(3, args.warmup)):
        orc.rows(cfg, *a, nv, True, False, cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        rec, _, _ = orc.rows(cfg, *a, nv, True, False, cores)
        orc.reduce(cfg, rec)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = rows * len(times) / total
    sample = (f"first {rows} of {wl.N} rows of {wl.name} per step (gradient + all scalars, "
              f"fp64, {cores} OpenMP threads)")
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; see workloads.py)", "impl": "reference",
        "config": {"workload": wl.name, "N_tokens": wl.N, "V": wl.V, "losses": list(wl.losses),
                   "rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0
    line = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
