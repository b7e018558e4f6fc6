"""CPU-only checks of the C ABI library: it builds for sm_103a, loads, exports
every function include/headloss.h declares, and answers host-only calls
without a GPU.  No compute call is made here."""
import ctypes
import os
import re

import pytest

from gradient_row_online_gb300 import build as B
from gradient_row_online_gb300 import headloss as hlb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(headloss_\w+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return hlb.load_library()


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(hlb.EXPORTS)


def test_host_only_calls(lib):
    assert hlb.headloss_version() == 1
    assert hlb.headloss_launches_per_call() == 3
    assert hlb.headloss_strerror(0) == "ok"
    assert "aligned" in hlb.headloss_strerror(hlb.HEADLOSS_ERR_ALIGN)
    assert lib.headloss_force_plan(None, None) == hlb.HEADLOSS_ERR_ARG
    assert lib.headloss_forward_backward(None, None, 1, 1, 1, None, None, None, None, None,
                                         None, None) == hlb.HEADLOSS_ERR_ARG
    assert lib.headloss_forward_backward_ext(None, None, 1, 1, 1, None, None, None, None, None,
                                             None, None, None) == hlb.HEADLOSS_ERR_ARG
    e = ctypes.c_int()
    assert lib.headloss_get_device_error(None, None, ctypes.byref(e)) == hlb.HEADLOSS_ERR_ARG
    # invalid configurations are rejected before any device is touched
    h = ctypes.c_void_p()
    assert lib.headloss_create(0, None, 1.0, 0.2, 0.0, 1.0, ctypes.byref(h)) == hlb.HEADLOSS_ERR_ARG
    assert lib.headloss_create(1, None, -1.0, 0.2, 0.0, 1.0, ctypes.byref(h)) == hlb.HEADLOSS_ERR_ARG
    assert lib.headloss_create(1, None, 1.0, 0.2, 0.0, 0.0, ctypes.byref(h)) == hlb.HEADLOSS_ERR_ARG


def test_missing_library_fails_loudly(tmp_path):
    saved = hlb._lib
    try:
        hlb._lib = None
        with pytest.raises(RuntimeError):
            hlb.load_library(str(tmp_path / "libheadloss.so"))
    finally:
        hlb._lib = saved


def test_build_targets_sm_103a_only():
    assert B.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_lmhead_rejects_bad_arguments_before_any_work(lib):
    """Sizes off the tile grid, null pointers and unaligned bases are refused
    on the host (no GPU needed)."""
    ok = 1 << 12  # a 16-byte aligned fake address; never dereferenced here
    f = lib.headloss_lmhead_logits
    assert f(ok, ok, 100, 64, 256, ok, ok, ok, None) == hlb.HEADLOSS_ERR_ARG   # N % 128
    assert f(ok, ok, 128, 60, 256, ok, ok, ok, None) == hlb.HEADLOSS_ERR_ARG   # D % 64
    assert f(ok, ok, 128, 64, 300, ok, ok, ok, None) == hlb.HEADLOSS_ERR_ARG   # V % 256
    assert f(None, ok, 128, 64, 256, ok, ok, ok, None) == hlb.HEADLOSS_ERR_ARG
    assert f(ok, ok, 128, 64, 256, ok, ok, None, None) == hlb.HEADLOSS_ERR_ARG
    assert f(ok + 2, ok, 128, 64, 256, ok, ok, ok, None) == hlb.HEADLOSS_ERR_ALIGN
    assert f(ok, ok, 128, 64, 256, ok + 8, ok, ok, None) == hlb.HEADLOSS_ERR_ALIGN

