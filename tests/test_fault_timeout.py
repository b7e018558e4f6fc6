"""Failure detection without a GPU fault.

A test-only build of the library (-DHL_FAULT_INJECT, never the shipped
libheadloss.so) can skip the bulk copy of one row and shorten every in-kernel
wait.  The wait for the missing copy must give up, the call must report
HEADLOSS_ERR_TIMEOUT through headloss_get_device_error, and the next call on
the same context must run normally and match the shipped library.

The cases are sized so that no mbarrier whose copy was skipped is ever armed
again: one row per CTA (N small) and, for the streaming kernel, rows of one
chunk.  Every wait on it is bounded.
"""
import ctypes

import numpy as np
import pytest
import torch

import gradient_row_online_gb300 as pkg
from gradient_row_online_gb300 import build as B
from gradient_row_online_gb300 import headloss as hlb
from gradient_row_online_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _fault_lib():
    lib = ctypes.CDLL(B.build(fault_inject=True))
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.headloss_create.argtypes = [ctypes.c_uint32, ctypes.POINTER(hlb.headloss_weights),
                                    ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                    ctypes.c_float, ctypes.POINTER(vp)]
    lib.headloss_forward_backward.argtypes = [vp, vp, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp]
    lib.headloss_get_device_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
    lib.headloss_force_plan.argtypes = [vp, ctypes.POINTER(hlb.headloss_plan_desc)]
    lib.headloss_destroy.argtypes = [vp]
    lib.headloss_test_inject.argtypes = [vp, i64, ctypes.c_ulonglong]
    return lib


@pytest.mark.parametrize("kernel,dtype", [(hlb.HEADLOSS_KERNEL_RESIDENT, torch.bfloat16),
                                          (hlb.HEADLOSS_KERNEL_STREAM, torch.bfloat16),
                                          (hlb.HEADLOSS_KERNEL_RESIDENT, torch.float32)])
def test_skipped_copy_times_out_and_the_next_call_is_clean(kernel, dtype):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lib = _fault_lib()
    wl = W.Workload("fault", 2, 1024, dtype, ("ce", "z", "entropy"),
                    dict(ce=1.0, z=0.1, dist_ce=0.0, fkl=0.0, rkl=0.0, grpo=0.0, entropy=0.2,
                         grad_scale=1.0), mask_frac=0.0)
    inp = W.make_inputs(wl, "cuda")
    flags = pkg.flags_of(wl.losses)
    w = hlb.make_weights(**wl.weights)
    h = ctypes.c_void_p()
    assert lib.headloss_create(flags, ctypes.byref(w), 1.0, 0.2, 0.0, 1.0, ctypes.byref(h)) == 0
    plan = hlb.headloss_plan_desc(kernel, 0, 2, 256,
                                  1 if kernel == hlb.HEADLOSS_KERNEL_STREAM else 0)
    assert lib.headloss_force_plan(h, ctypes.byref(plan)) == 0
    dcode = hlb.dtype_code(dtype)
    stream = torch.cuda.current_stream().cuda_stream

    def call(g, out):
        return lib.headloss_forward_backward(h, inp["logits"].data_ptr(), wl.N, wl.V, dcode,
                                             inp["labels"].data_ptr(), None, None, None,
                                             g.data_ptr(), out.data_ptr(), stream)

    def device_error():
        e = ctypes.c_int()
        assert lib.headloss_get_device_error(h, stream, ctypes.byref(e)) == 0
        return e.value

    g = torch.empty_like(inp["logits"])
    out = torch.empty(16, dtype=torch.float32, device="cuda")
    # the copy of row 0 never comes; every wait gives up after 50 ms
    assert lib.headloss_test_inject(h, 0, 50_000_000) == 0
    assert call(g, out) == 0
    assert device_error() == hlb.HEADLOSS_ERR_TIMEOUT
    assert device_error() == hlb.HEADLOSS_OK  # reading clears it
    # the context is still usable: a normal call matches the shipped library
    assert lib.headloss_test_inject(h, -1, 0) == 0
    assert call(g, out) == 0
    assert device_error() == hlb.HEADLOSS_OK
    ref = pkg.headloss_for(wl)
    g_ref = torch.empty_like(inp["logits"])
    out_ref = ref(inp["logits"], inp["labels"], None, None, None, g_ref)
    torch.cuda.synchronize()
    assert np.allclose(out.cpu().numpy(), out_ref.cpu().numpy(), rtol=1e-5, atol=1e-6)
    assert torch.equal(g, g_ref) or torch.allclose(g.float(), g_ref.float(), rtol=1e-2,
                                                   atol=1e-6)
    lib.headloss_destroy(h)
    ref.close()
