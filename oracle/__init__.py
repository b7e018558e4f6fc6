"""fp64 CPU oracle for the monolithic LM-head loss -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library path never does, and this
package imports nothing from the library.

The arithmetic lives in ``headloss_oracle.c`` (plain C, fp64, one row at a
time); this module builds it with gcc on first use and marshals numpy arrays
through ctypes.  Inputs are passed as fp64 arrays that are exact upcasts of
the logits the library sees.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "headloss_oracle.c")
_LIB = os.path.join(_HERE, "libheadloss_oracle.so")
_lock = threading.Lock()
_lib = None

# Loss / metric bits, defined here independently of the library.
CE, Z, DIST_CE, FKL, RKL, GRPO, GRPO_STATS, ENTROPY = (1 << i for i in range(8))
DIST_ANY = DIST_CE | FKL | RKL

# Per-row record fields (headloss_oracle.c, enum RF_*).
RF = dict(valid=0, ce=1, z=2, dist_ce=3, fkl=4, rkl=5, grpo=6, logprob=7, ratio=8,
          clipped=9, kl3=10, adv=11, adv2=12, entropy=13, ambiguous=14, act=15, lse=16)
N_RF = 17

# Scalar slots of a call.
SLOTS = ("total", "ce", "z", "dist_ce", "fkl", "rkl", "grpo_loss", "new_logprob_mean",
         "ratio_mean", "clip_frac", "kl_k3", "adv_mean", "adv_std", "entropy_mean",
         "n_valid", "n_clipped")


class _Cfg(ctypes.Structure):
    _fields_ = [("flags", ctypes.c_uint32)] + [
        (n, ctypes.c_double)
        for n in ("w_ce", "w_z", "w_dist_ce", "w_fkl", "w_rkl", "w_grpo", "w_entropy",
                  "grad_scale", "temperature", "clip_eps", "softcap", "logits_scale")
    ]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, -O2, no fast-math)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                                   "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_rows.argtypes = [ctypes.POINTER(_Cfg), ctypes.c_int64, ctypes.c_int64, dp, ip,
                                    dp, dp, dp, ctypes.c_int64, dp, dp, dp, ctypes.c_int]
        lib.oracle_rows.restype = ctypes.c_int
        lib.oracle_reduce.argtypes = [ctypes.POINTER(_Cfg), dp, ctypes.c_int64, dp]
        lib.oracle_reduce.restype = None
        lib.oracle_count_valid.argtypes = [ip, ctypes.c_int64]
        lib.oracle_count_valid.restype = ctypes.c_int64
        lib.oracle_row_fields.restype = ctypes.c_int
        assert lib.oracle_row_fields() == N_RF
        _lib = lib
    return _lib


def make_cfg(flags: int, weights: dict | None = None, temperature: float = 1.0,
             clip_eps: float = 0.2, softcap: float = 0.0, logits_scale: float = 1.0,
             grad_scale: float = 1.0) -> _Cfg:
    w = dict(ce=1.0, z=0.0, dist_ce=0.0, fkl=0.0, rkl=0.0, grpo=1.0, entropy=0.0)
    if weights:
        w.update(weights)
    return _Cfg(flags, w["ce"], w["z"], w["dist_ce"], w["fkl"], w["rkl"], w["grpo"],
                w["entropy"], grad_scale, temperature, clip_eps, softcap, logits_scale)


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def count_valid(labels, n_rows: int) -> int:
    if labels is None:
        return int(n_rows)
    lab = np.ascontiguousarray(labels, dtype=np.int64)
    return int(_load().oracle_count_valid(_ptr(lab, ctypes.c_int64), lab.shape[0]))


def rows(cfg: _Cfg, x, labels=None, teacher=None, old_logprobs=None, advantages=None,
         n_valid_total: int | None = None, want_grad: bool = True, want_gmag: bool = False,
         n_threads: int = 0):
    """Per-row records (n x 17) and, optionally, gradient / term magnitude (n x V)."""
    lib = _load()
    x = _f64(x)
    n, V = x.shape
    lab = None if labels is None else np.ascontiguousarray(labels, dtype=np.int64)
    t = _f64(teacher)
    o = _f64(old_logprobs)
    a = _f64(advantages)
    if n_valid_total is None:
        n_valid_total = count_valid(lab, n)
    rec = np.zeros((n, N_RF), np.float64)
    grad = np.empty((n, V), np.float64) if want_grad else None
    gmag = np.empty((n, V), np.float64) if want_gmag else None
    rc = lib.oracle_rows(ctypes.byref(cfg), n, V, _ptr(x, ctypes.c_double),
                         _ptr(lab, ctypes.c_int64), _ptr(t, ctypes.c_double),
                         _ptr(o, ctypes.c_double), _ptr(a, ctypes.c_double), int(n_valid_total),
                         _ptr(rec, ctypes.c_double), _ptr(grad, ctypes.c_double),
                         _ptr(gmag, ctypes.c_double), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_rows rejected its arguments")
    return rec, grad, gmag


def reduce(cfg: _Cfg, rec) -> np.ndarray:
    """The sixteen scalars of a call from its per-row records."""
    rec = _f64(rec)
    out = np.zeros(16, np.float64)
    _load().oracle_reduce(ctypes.byref(cfg), _ptr(rec, ctypes.c_double), rec.shape[0],
                          _ptr(out, ctypes.c_double))
    return out


def forward_backward(cfg: _Cfg, x, labels=None, teacher=None, old_logprobs=None,
                     advantages=None, want_grad: bool = True, want_gmag: bool = False,
                     n_threads: int = 0):
    """A whole call: (scalars[16], per-row records, grad or None, gmag or None)."""
    rec, grad, gmag = rows(cfg, x, labels, teacher, old_logprobs, advantages, None, want_grad,
                           want_gmag, n_threads)
    return reduce(cfg, rec), rec, grad, gmag


def lm_head_forward_backward(cfg: _Cfg, hidden, weight, labels=None, teacher=None,
                             old_logprobs=None, advantages=None, n_threads: int = 0):
    """The LM head in front of the loss, written out plainly: logits = hidden @ weight^T
    (fp64), the loss of ``forward_backward`` on those logits, and the gradients of
    grad_scale * total with respect to hidden (N x D) and weight (V x D) by the chain
    rule through the linear map (dH = G @ weight, dW = G^T @ hidden, G the logits
    gradient).  The teacher enters as logits, as in ``forward_backward``.

    Returns (scalars[16], per-row records, dH, dW, logits, G)."""
    h = _f64(hidden)
    w = _f64(weight)
    if h.ndim != 2 or w.ndim != 2 or h.shape[1] != w.shape[1]:
        raise ValueError("hidden is N x D and weight is V x D")
    x = h @ w.T
    scalars, rec, g, _ = forward_backward(cfg, x, labels, teacher, old_logprobs, advantages,
                                          want_grad=True, n_threads=n_threads)
    return scalars, rec, g @ w, g.T @ h, x, g


def gspo_forward_backward(x, labels, old_logprobs, advantages, seg_offsets, clip_eps,
                          weight: float = 1.0, grad_scale: float = 1.0, softcap: float = 0.0,
                          logits_scale: float = 1.0, n_threads: int = 0):
    """GSPO, the sequence-level clipped policy objective, written out plainly.

    Reading (the pages name the objective and its per-segment form, not its
    formula; this is the objective of the GSPO method itself):
      - tokens [off_i, off_{i+1}) form segment i (seg_offsets: n_seq + 1
        increasing offsets, 0 .. N); a token is valid when 0 <= label < V;
      - lp_t = log p(label_t) of the student softmax at T = 1 (softcap and
        scale applied as for every loss), from the row oracle;
      - over the valid tokens T_i of a segment (L_i of them):
        s_i = exp((1 / L_i) sum_t (lp_t - old_t)) -- the geometric mean of the
        token ratios; A_i = mean of the tokens' advantages;
        obj_i = min(s_i A_i, clip(s_i, 1 - eps, 1 + eps) A_i);
      - G = segments with at least one valid token; loss = -(1/G) sum_i obj_i;
      - the unclipped branch carries the gradient unless it is the larger
        objective (ties count as unclipped);
      - d(weight * grad_scale * loss)/d lp_t = -weight * grad_scale * A_i s_i
        act_i / (G L_i), and the logits gradient of token t is that times
        d lp_t / d x_t (the chain rule through the row's log-softmax).

    Returns (scalars, coeff, grad): scalars = (loss, ratio_mean, clip_frac,
    n_segments); coeff = d(weight * grad_scale * loss)/d lp per token (0 on
    masked tokens); grad = N x V logits gradient."""
    x = _f64(x)
    n, V = x.shape
    lab = np.ascontiguousarray(labels, dtype=np.int64)
    old = _f64(old_logprobs)
    adv = _f64(advantages)
    off = np.asarray(seg_offsets, dtype=np.int64)
    if off.ndim != 1 or off[0] != 0 or off[-1] != n or np.any(np.diff(off) < 0):
        raise ValueError("seg_offsets: increasing offsets from 0 to N")
    # per-token log p(label) (the GRPO statistics' new log-prob) and d(-lp)/dx
    # (the gradient of a cross-entropy of weight 1 normalised by 1) from the
    # row oracle; the statistics' own ratio inputs are unused here
    cfg = make_cfg(CE | GRPO_STATS, dict(ce=1.0, grpo=0.0), softcap=softcap,
                   logits_scale=logits_scale, grad_scale=1.0)
    zeros = np.zeros(n)
    rec, neg_dlp, _ = rows(cfg, x, lab, None, zeros, zeros, n_valid_total=1, want_grad=True,
                           n_threads=n_threads)
    lp = rec[:, RF["logprob"]]
    valid = rec[:, RF["valid"]] > 0
    segs = []
    for i in range(len(off) - 1):
        t = np.arange(off[i], off[i + 1])
        t = t[valid[t]]
        if t.size == 0:
            continue
        L = t.size
        s = math.exp(float(np.sum(lp[t] - old[t])) / L)
        A = float(np.mean(adv[t]))
        sc = min(max(s, 1.0 - clip_eps), 1.0 + clip_eps)
        unc, clp = s * A, sc * A
        act = unc <= clp or (1.0 - clip_eps <= s <= 1.0 + clip_eps)
        segs.append((t, L, s, A, min(unc, clp), act, abs(s - 1.0) > clip_eps))
    G = len(segs)
    coeff = np.zeros(n)
    if G == 0:
        return np.zeros(4), coeff, np.zeros((n, V))
    loss = -sum(sg[4] for sg in segs) / G
    for t, L, s, A, _, act, _ in segs:
        if act:
            coeff[t] = -weight * grad_scale * A * s / (G * L)
    grad = -coeff[:, None] * neg_dlp
    scalars = np.array([loss, sum(sg[2] for sg in segs) / G, sum(sg[6] for sg in segs) / G,
                        float(G)])
    return scalars, coeff, grad


def tile_records(x, softcap: float = 0.0, logits_scale: float = 1.0, tile: int = 256,
                 temperature: float | None = None):
    """The first-pass statistics of each (row, tile of ``tile`` columns), written out
    plainly in fp64: the record the fused LM head's GEMM epilogue emits for the loss
    (ServiceNow Fast-LLM PR #549, "Approach": the row's softmax statistics built up
    block by block and merged by their running maximum; "Correctness": the LM head
    computed in front of the loss).

    With z = s c tanh(x / c) (c = 0: z = s x) and zs = z log2(e) (base 2):
      m2 = max zs, S = sum 2^(zs - m2), E = sum 2^(zs - m2) (zs - m2), X = max |x|,
    per tile, and with a temperature T also S_T = sum 2^((zs - m2) / T) (the
    student's sums at T, which the distillation losses' normaliser needs).
    Returns an N x (V / tile) x 4 array (m2, S, E, X), or x 5 with S_T last.
    A teacher's records are those of its logits with softcap 0 and
    logits_scale 1 / T (the teacher enters the losses as t / T)."""
    x = _f64(x)
    n, V = x.shape
    if V % tile:
        raise ValueError("V must be a multiple of the tile width")
    z = logits_scale * (softcap * np.tanh(x / softcap) if softcap > 0 else x)
    zs = z / math.log(2.0)
    out = np.zeros((n, V // tile, 4 if temperature is None else 5))
    for t in range(V // tile):
        blk = zs[:, t * tile:(t + 1) * tile]
        m2 = blk.max(axis=1)
        d = blk - m2[:, None]
        e = np.exp2(d)
        out[:, t, 0] = m2
        out[:, t, 1] = e.sum(axis=1)
        out[:, t, 2] = (e * d).sum(axis=1)
        out[:, t, 3] = np.abs(x[:, t * tile:(t + 1) * tile]).max(axis=1)
        if temperature is not None:
            out[:, t, 4] = np.exp2(d / temperature).sum(axis=1)
    return out
