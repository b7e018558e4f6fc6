"""Thin Python binding of the C ABI in include/headloss.h (ctypes).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libheadloss.so.  Tensors are passed as raw device pointers; torch
is used for device memory and streams.  There is no fallback: if the library
is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libheadloss.so")

# enum headloss_flag
HEADLOSS_CE = 1 << 0
HEADLOSS_Z = 1 << 1
HEADLOSS_DIST_CE = 1 << 2
HEADLOSS_FKL = 1 << 3
HEADLOSS_RKL = 1 << 4
HEADLOSS_GRPO = 1 << 5
HEADLOSS_GRPO_STATS = 1 << 6
HEADLOSS_ENTROPY = 1 << 7

# enum headloss_dtype
HEADLOSS_FP32, HEADLOSS_BF16, HEADLOSS_FP16 = 0, 1, 2

# enum headloss_status
STATUS = {0: "HEADLOSS_OK", 1: "HEADLOSS_ERR_ARG", 2: "HEADLOSS_ERR_DTYPE",
          3: "HEADLOSS_ERR_ALIGN", 4: "HEADLOSS_ERR_MISSING_INPUT", 5: "HEADLOSS_ERR_CUDA",
          6: "HEADLOSS_ERR_TIMEOUT", 7: "HEADLOSS_ERR_LABEL_RANGE", 8: "HEADLOSS_ERR_SIZE"}
HEADLOSS_OK = 0
HEADLOSS_ERR_ARG = 1
HEADLOSS_ERR_DTYPE = 2
HEADLOSS_ERR_ALIGN = 3
HEADLOSS_ERR_MISSING_INPUT = 4
HEADLOSS_ERR_CUDA = 5
HEADLOSS_ERR_TIMEOUT = 6
HEADLOSS_ERR_LABEL_RANGE = 7
HEADLOSS_ERR_SIZE = 8

# enum headloss_slot
SLOTS = ("total", "ce", "z", "dist_ce", "fkl", "rkl", "grpo_loss", "new_logprob_mean",
         "ratio_mean", "clip_frac", "kl_k3", "adv_mean", "adv_std", "entropy_mean", "n_valid",
         "n_clipped")

# Every function declared in include/headloss.h and include/headloss_lmhead.h.
EXPORTS = ("headloss_create", "headloss_forward_backward", "headloss_get_device_error",
           "headloss_plan", "headloss_force_plan", "headloss_launches_per_call",
           "headloss_destroy", "headloss_strerror", "headloss_version",
           "headloss_forward_backward_noalloc", "headloss_forward_backward_ext",
           "headloss_gspo_seam", "headloss_forward_backward_rowstats",
           "headloss_lmhead_logits", "headloss_lmhead_logits_rowstats")


# enum headloss_kernel
HEADLOSS_KERNEL_AUTO, HEADLOSS_KERNEL_RESIDENT, HEADLOSS_KERNEL_STREAM = 0, 1, 2
KERNELS = {0: "auto", 1: "resident", 2: "stream"}


class headloss_call_ext(ctypes.Structure):
    """struct headloss_call_ext: per-call extras (per-token outputs, gradient
    accumulation, the divisor of a split batch)."""
    _fields_ = [("new_logprobs", ctypes.c_void_p), ("row_loss", ctypes.c_void_p),
                ("accumulate", ctypes.c_int), ("divisor", ctypes.c_double),
                ("token_coeff", ctypes.c_void_p)]


class headloss_plan_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("kernel", "cluster", "stages", "threads",
                                             "chunk_words")]


class headloss_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in
                ("ce", "z", "dist_ce", "fkl", "rkl", "grpo", "entropy", "grad_scale")]


class HeadlossError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({_strerror(status)})")


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libheadloss.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with gradient_row_online_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    ip = ctypes.POINTER(ctypes.c_int)
    lib.headloss_create.argtypes = [ctypes.c_uint32, ctypes.POINTER(headloss_weights),
                                    ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                    ctypes.c_float, ctypes.POINTER(vp)]
    lib.headloss_create.restype = i32
    lib.headloss_forward_backward.argtypes = [vp, vp, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp]
    lib.headloss_forward_backward.restype = i32
    lib.headloss_get_device_error.argtypes = [vp, vp, ip]
    lib.headloss_get_device_error.restype = i32
    pp = ctypes.POINTER(headloss_plan_desc)
    lib.headloss_plan.argtypes = [vp, i64, i32, pp, ip, ip]
    lib.headloss_plan.restype = i32
    lib.headloss_force_plan.argtypes = [vp, pp]
    lib.headloss_force_plan.restype = i32
    lib.headloss_launches_per_call.argtypes = []
    lib.headloss_launches_per_call.restype = i32
    lib.headloss_destroy.argtypes = [vp]
    lib.headloss_destroy.restype = None
    lib.headloss_strerror.argtypes = [i32]
    lib.headloss_strerror.restype = ctypes.c_char_p
    lib.headloss_version.argtypes = []
    lib.headloss_version.restype = i32
    lib.headloss_forward_backward_noalloc.argtypes = [
        ctypes.c_uint32, ctypes.POINTER(headloss_weights), ctypes.c_float, ctypes.c_float,
        ctypes.c_float, ctypes.c_float, vp, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp]
    lib.headloss_forward_backward_noalloc.restype = i32
    lib.headloss_forward_backward_ext.argtypes = [vp, vp, i64, i64, i32, vp, vp, vp, vp, vp, vp,
                                                  ctypes.POINTER(headloss_call_ext), vp]
    lib.headloss_forward_backward_ext.restype = i32
    lib.headloss_lmhead_logits.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp]
    lib.headloss_lmhead_logits.restype = i32
    lib.headloss_gspo_seam.argtypes = [vp, vp, vp, vp, i64, i64, vp, i32, f32, f32, f32, vp, vp,
                                       vp]
    lib.headloss_gspo_seam.restype = i32
    lib.headloss_lmhead_logits_rowstats.argtypes = [vp, vp, i32, i32, i32, f32, f32, f32, vp, vp,
                                                    vp, vp, vp]
    lib.headloss_lmhead_logits_rowstats.restype = i32
    lib.headloss_forward_backward_rowstats.argtypes = [vp, vp, i64, i64, i32, vp, vp, vp, vp, vp,
                                                       vp, vp, vp, vp, vp, vp]
    lib.headloss_forward_backward_rowstats.restype = i32
    _lib = lib
    return lib


def _strerror(status: int) -> str:
    try:
        return load_library().headloss_strerror(status).decode()
    except Exception:
        return "?"


def _check(status: int, where: str):
    if status != HEADLOSS_OK:
        raise HeadlossError(status, where)


def _ptr(a):
    """Device address of a tensor (or an int address, or None)."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(stream):
    if stream is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream
        except Exception:
            return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dtype_code(torch_dtype) -> int:
    import torch
    return {torch.float32: HEADLOSS_FP32, torch.bfloat16: HEADLOSS_BF16,
            torch.float16: HEADLOSS_FP16}[torch_dtype]


def make_weights(ce=1.0, z=0.0, dist_ce=0.0, fkl=0.0, rkl=0.0, grpo=1.0, entropy=0.0,
                 grad_scale=1.0) -> headloss_weights:
    return headloss_weights(ce, z, dist_ce, fkl, rkl, grpo, entropy, grad_scale)


def headloss_create(flags: int, weights=None, temperature: float = 1.0, clip_eps: float = 0.2,
                    softcap: float = 0.0, logits_scale: float = 1.0) -> int:
    lib = load_library()
    if isinstance(weights, dict):
        weights = make_weights(**weights)
    h = ctypes.c_void_p()
    w = ctypes.byref(weights) if weights is not None else None
    _check(lib.headloss_create(flags, w, temperature, clip_eps, softcap, logits_scale,
                               ctypes.byref(h)), "headloss_create")
    return h.value


def headloss_forward_backward(h, logits, N, V, dtype, labels, teacher_logits, old_logprobs,
                              advantages, grad_out, scalars_out, stream=None) -> None:
    lib = load_library()
    _check(lib.headloss_forward_backward(h, _ptr(logits), int(N), int(V), int(dtype),
                                         _ptr(labels), _ptr(teacher_logits), _ptr(old_logprobs),
                                         _ptr(advantages), _ptr(grad_out), _ptr(scalars_out),
                                         _stream(stream)), "headloss_forward_backward")


def headloss_forward_backward_ext(h, logits, N, V, dtype, labels, teacher_logits, old_logprobs,
                                  advantages, grad_out, scalars_out, new_logprobs=None,
                                  row_loss=None, accumulate=False, divisor=0.0,
                                  token_coeff=None, stream=None) -> None:
    """The call with its extras: per-row log p(label) and total loss outputs,
    gradient accumulation into grad_out, the divisor of a split batch, and a
    per-token coefficient on the label column (GSPO's, from headloss_gspo_seam)."""
    lib = load_library()
    ext = headloss_call_ext(_ptr(new_logprobs), _ptr(row_loss), int(bool(accumulate)),
                            float(divisor), _ptr(token_coeff))
    _check(lib.headloss_forward_backward_ext(h, _ptr(logits), int(N), int(V), int(dtype),
                                             _ptr(labels), _ptr(teacher_logits),
                                             _ptr(old_logprobs), _ptr(advantages),
                                             _ptr(grad_out), _ptr(scalars_out),
                                             ctypes.byref(ext), _stream(stream)),
           "headloss_forward_backward_ext")


def headloss_forward_backward_noalloc(flags, weights, temperature, clip_eps, softcap,
                                      logits_scale, logits, N, V, dtype, labels, teacher_logits,
                                      old_logprobs, advantages, grad_out, scalars_out,
                                      stream=None) -> None:
    """The allocation-free call (no handle): for callers that must not allocate
    device memory while computing the loss, e.g. inside a CUDA-graph capture."""
    lib = load_library()
    if isinstance(weights, dict):
        weights = make_weights(**weights)
    w = ctypes.byref(weights) if weights is not None else None
    _check(lib.headloss_forward_backward_noalloc(
        flags, w, temperature, clip_eps, softcap, logits_scale, _ptr(logits), int(N), int(V),
        int(dtype), _ptr(labels), _ptr(teacher_logits), _ptr(old_logprobs), _ptr(advantages),
        _ptr(grad_out), _ptr(scalars_out), _stream(stream)), "headloss_forward_backward_noalloc")


def headloss_lmhead_logits(hidden, weight, N, D, V, logits, stats, err, stream=None) -> None:
    """logits = hidden . weight^T and per-(row, 256-column tile) (max, sum exp)
    statistics (include/headloss_lmhead.h); raises HeadlossError on a bad status."""
    _check(load_library().headloss_lmhead_logits(_ptr(hidden), _ptr(weight), int(N), int(D),
                                                 int(V), _ptr(logits), _ptr(stats), _ptr(err),
                                                 _stream(stream)),
           "headloss_lmhead_logits")


def headloss_lmhead_logits_rowstats(hidden, weight, N, D, V, softcap, logits_scale, logits,
                                    row_stats, err, stream=None, temperature=1.0,
                                    row_stats_t=None) -> None:
    """The LM-head GEMM with the loss's per-tile first-pass records, and with
    row_stats_t the tiles' sums at `temperature` (include/headloss_lmhead.h);
    raises HeadlossError on a bad status."""
    _check(load_library().headloss_lmhead_logits_rowstats(
        _ptr(hidden), _ptr(weight), int(N), int(D), int(V), float(softcap), float(logits_scale),
        float(temperature), _ptr(logits), _ptr(row_stats), _ptr(row_stats_t), _ptr(err),
        _stream(stream)), "headloss_lmhead_logits_rowstats")


def headloss_forward_backward_rowstats(h, logits, N, V, dtype, labels, old_logprobs, advantages,
                                       row_stats, grad_out, scalars_out, stream=None,
                                       teacher=None, row_stats_t=None, teacher_stats=None,
                                       new_logprobs=None, row_loss=None, accumulate=False,
                                       divisor=0.0, token_coeff=None) -> None:
    """The loss's gradient pass alone from the GEMMs' row statistics (the
    student's, its sums at the temperature, the teacher's; include/headloss.h),
    with the extras of headloss_forward_backward_ext; raises HeadlossError on a
    bad status."""
    ext = headloss_call_ext(_ptr(new_logprobs), _ptr(row_loss), int(bool(accumulate)),
                            float(divisor), _ptr(token_coeff))
    _check(load_library().headloss_forward_backward_rowstats(
        h, _ptr(logits), int(N), int(V), int(dtype), _ptr(labels), _ptr(teacher),
        _ptr(old_logprobs), _ptr(advantages), _ptr(row_stats), _ptr(row_stats_t),
        _ptr(teacher_stats), _ptr(grad_out), _ptr(scalars_out), ctypes.byref(ext),
        _stream(stream)), "headloss_forward_backward_rowstats")


def headloss_gspo_seam(new_logprobs, old_logprobs, advantages, labels, N, V, seg_offsets, n_seg,
                       clip_eps, weight, grad_scale, token_coeff, scalars_out,
                       stream=None) -> None:
    """GSPO's per-segment seam (include/headloss.h): the sequence ratios and
    the per-token coefficient for the backward call; raises on a bad status."""
    _check(load_library().headloss_gspo_seam(
        _ptr(new_logprobs), _ptr(old_logprobs), _ptr(advantages), _ptr(labels), int(N), int(V),
        _ptr(seg_offsets), int(n_seg), float(clip_eps), float(weight), float(grad_scale),
        _ptr(token_coeff), _ptr(scalars_out), _stream(stream)), "headloss_gspo_seam")


def headloss_get_device_error(h, stream=None) -> int:
    lib = load_library()
    e = ctypes.c_int()
    _check(lib.headloss_get_device_error(h, _stream(stream), ctypes.byref(e)),
           "headloss_get_device_error")
    return e.value


def headloss_plan(h, V: int, dtype: int) -> dict:
    lib = load_library()
    d = headloss_plan_desc()
    ctas, smem = ctypes.c_int(), ctypes.c_int()
    _check(lib.headloss_plan(h, int(V), int(dtype), ctypes.byref(d), ctypes.byref(ctas),
                             ctypes.byref(smem)), "headloss_plan")
    return dict(kernel=KERNELS[d.kernel], cluster=d.cluster, stages=d.stages,
                threads=d.threads, chunk_words=d.chunk_words, ctas=ctas.value,
                smem_bytes=smem.value)


def headloss_force_plan(h, kernel: int = 0, cluster: int = 0, stages: int = 0, threads: int = 0,
                        chunk_words: int = 0) -> None:
    """Pin plan choices (0 = the planner decides); all zero restores the automatic plan."""
    d = headloss_plan_desc(int(kernel), int(cluster), int(stages), int(threads), int(chunk_words))
    _check(load_library().headloss_force_plan(h, ctypes.byref(d)), "headloss_force_plan")


def headloss_launches_per_call() -> int:
    return load_library().headloss_launches_per_call()


def headloss_destroy(h) -> None:
    if h:
        load_library().headloss_destroy(h)


def headloss_strerror(status: int) -> str:
    return load_library().headloss_strerror(int(status)).decode()


def headloss_version() -> int:
    return load_library().headloss_version()


class HeadLoss:
    """A handle plus the call on torch tensors (same semantics as the C ABI)."""

    def __init__(self, flags: int, weights=None, temperature: float = 1.0,
                 clip_eps: float = 0.2, softcap: float = 0.0, logits_scale: float = 1.0):
        self.flags = flags
        self.h = headloss_create(flags, weights, temperature, clip_eps, softcap, logits_scale)

    def __call__(self, logits, labels=None, teacher_logits=None, old_logprobs=None,
                 advantages=None, grad_out=None, scalars_out=None, stream=None,
                 new_logprobs=None, row_loss=None, accumulate=False, divisor=0.0):
        import torch
        N, V = logits.shape
        if scalars_out is None:
            scalars_out = torch.empty(16, dtype=torch.float32, device=logits.device)
        if new_logprobs is None and row_loss is None and not accumulate and not divisor:
            headloss_forward_backward(self.h, logits, N, V, dtype_code(logits.dtype), labels,
                                      teacher_logits, old_logprobs, advantages, grad_out,
                                      scalars_out, stream)
        else:
            headloss_forward_backward_ext(self.h, logits, N, V, dtype_code(logits.dtype), labels,
                                          teacher_logits, old_logprobs, advantages, grad_out,
                                          scalars_out, new_logprobs, row_loss, accumulate,
                                          divisor, stream)
        return scalars_out

    def plan(self, V: int, dtype: int) -> dict:
        return headloss_plan(self.h, V, dtype)

    def force_plan(self, kernel: int = 0, cluster: int = 0, stages: int = 0, threads: int = 0,
                   chunk_words: int = 0) -> None:
        headloss_force_plan(self.h, kernel, cluster, stages, threads, chunk_words)

    def device_error(self, stream=None) -> int:
        return headloss_get_device_error(self.h, stream)

    def close(self):
        if self.h:
            headloss_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
