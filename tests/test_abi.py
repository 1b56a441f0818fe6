"""The C-ABI library without a GPU: it loads, exports every symbol the
header declares, and refuses bad arguments on the host before any CUDA call.
"""

import ctypes
import os
import re

import pytest

import gated_deltanet_linear_gb300 as gdn
from gated_deltanet_linear_gb300 import _build

HEADER = os.path.join(_build.INCLUDE, "gdn.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return gdn.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(gdn.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    raw = ctypes.CDLL(_build.LIB)
    for name in declared_functions():
        assert ctypes.cast(getattr(raw, name), ctypes.c_void_p).value


def test_version_and_strerror(lib):
    assert gdn.gdn_version() == 100
    for code in range(-7, 1):
        assert gdn.gdn_strerror(code) != "unknown status"
    assert gdn.gdn_strerror(-99) == "unknown status"


def _call_step(lib, shape):
    null = None
    return lib.gdn_step(shape, *([null] * 7), None)


def test_host_side_refusals(lib):
    """Refusals decided from the shape and counts alone (no CUDA call)."""
    assert _call_step(lib, None) == gdn.GDN_EINVAL
    for bad in [gdn.Shape(1, 16, 48, 64, 128), gdn.Shape(1, 16, 48, 128, 64),
                gdn.Shape(1, 16, 40, 128, 128), gdn.Shape(-1, 16, 48, 128, 128),
                gdn.Shape(1, 0, 48, 128, 128)]:
        assert _call_step(lib, ctypes.byref(bad)) == gdn.GDN_ESHAPE
    ok = gdn.Shape(1, 16, 48, 128, 128)
    # NULL buffers with a valid shape
    assert _call_step(lib, ctypes.byref(ok)) == gdn.GDN_EINVAL
    # M out of range
    for M in (0, -3, gdn.GDN_MAX_TOKENS + 1):
        assert lib.gdn_step_m(ctypes.byref(ok), M, *([None] * 9),
                              None) == gdn.GDN_ERANGE
    # rollback m out of range
    assert lib.gdn_rollback(ctypes.byref(ok), 4, 5, None, None, None,
                            None) == gdn.GDN_ERANGE
    assert lib.gdn_rollback(ctypes.byref(ok), 4, -1, None, None, None,
                            None) == gdn.GDN_ERANGE
    # B == 0 is a no-op
    zero = gdn.Shape(0, 16, 48, 128, 128)
    assert _call_step(lib, ctypes.byref(zero)) == gdn.GDN_OK
    # misaligned pointers are refused before any device query
    fake = ctypes.c_void_p(0x1004)
    args = [fake] * 7
    assert lib.gdn_step(ctypes.byref(ok), *args, None) == gdn.GDN_EALIGN
    # prefill: T range and unknown precision
    assert lib.gdn_prefill(ctypes.byref(ok), 0, *([None] * 7), 64, 0, None,
                           0, None) == gdn.GDN_ERANGE
    assert lib.gdn_prefill(ctypes.byref(ok), 8, *([None] * 7), 64, 7, None,
                           0, None) == gdn.GDN_ERANGE
    # chunked modes: T * vh must stay below 2^31 (the tensor copies address
    # a sequence's rows with strides below 2^40 bytes); the fp32 mode has no
    # such limit and goes on to the buffer checks
    wide = gdn.Shape(1, 16, 4096, 128, 128)
    T = gdn.GDN_MAX_TOKENS                       # 2^20 * 4096 = 2^32
    for prec in (gdn.GDN_PREC_BF16X3, gdn.GDN_PREC_BF16):
        assert lib.gdn_prefill(ctypes.byref(wide), T, *([None] * 7), 64, prec,
                               None, 0, None) == gdn.GDN_ERANGE
    assert lib.gdn_prefill(ctypes.byref(wide), T, *([None] * 7), 64,
                           gdn.GDN_PREC_FP32, None, 0, None) == gdn.GDN_EINVAL


def test_binding_refuses_cpu_tensors(lib):
    import torch
    S = torch.zeros(1, 3, 128, 128)
    q = torch.zeros(1, 1, 1, 128)
    with pytest.raises(ValueError):
        gdn.gdn_step(S, q, q, torch.zeros(1, 1, 3, 128), torch.zeros(1, 1, 3),
                     torch.zeros(1, 1, 3), torch.zeros(1, 1, 3, 128))


def test_layer_and_norm_host_refusals(lib):
    """The layer-core and gated-RMSNorm entry points refuse bad shapes,
    counts and values on the host, before any CUDA call."""
    ok = gdn.Shape(2, 16, 48, 128, 128)
    bad = gdn.Shape(2, 16, 40, 128, 128)         # vh % kh != 0
    zero = gdn.Shape(0, 16, 48, 128, 128)
    n = None
    # gated RMSNorm: shape, count, eps, B == 0, NULL buffers
    norm = lambda sh, M, eps: lib.gdn_gated_rmsnorm_m(
        ctypes.byref(sh) if sh is not None else None, M, eps, n, n, n, n, n)
    assert norm(None, 1, 1e-6) == gdn.GDN_EINVAL
    assert norm(bad, 1, 1e-6) == gdn.GDN_ESHAPE
    assert norm(ok, 0, 1e-6) == gdn.GDN_ERANGE
    assert norm(ok, gdn.GDN_MAX_TOKENS + 1, 1e-6) == gdn.GDN_ERANGE
    assert norm(ok, 1, -1.0) == gdn.GDN_EINVAL
    assert norm(ok, 1, float("nan")) == gdn.GDN_EINVAL
    assert norm(zero, 1, 1e-6) == gdn.GDN_OK
    assert norm(ok, 1, 1e-6) == gdn.GDN_EINVAL     # NULL buffers
    # layer step: width-4 convolution only, count, eps, workspace size query
    step = lambda sh, M, ck, eps: lib.gdn_layer_step_m(
        ctypes.byref(sh), M, ck, eps, *([n] * 13), 0, n)
    assert step(ok, 1, 3, 1e-6) == gdn.GDN_ESHAPE
    assert step(ok, 0, 4, 1e-6) == gdn.GDN_ERANGE
    assert step(ok, 1, 4, -1.0) == gdn.GDN_EINVAL
    assert step(zero, 1, 4, 1e-6) == gdn.GDN_OK
    assert step(bad, 1, 4, 1e-6) == gdn.GDN_ESHAPE
    assert lib.gdn_layer_workspace(ctypes.byref(ok), 0) == 0
    per_token = 2 * 16 * 128 * 4 + 48 * 128 * 4 + 2 * 48 * 4
    assert lib.gdn_layer_workspace(ctypes.byref(ok), 3) == 2 * 3 * per_token
    # history rollback
    assert lib.gdn_layer_hist_rollback(ctypes.byref(ok), 4, 3, *([n] * 5),
                                       n) == gdn.GDN_ESHAPE
    assert lib.gdn_layer_hist_rollback(ctypes.byref(ok), 0, 4, *([n] * 5),
                                       n) == gdn.GDN_ERANGE
    assert gdn.gdn_strerror(gdn.GDN_ESCRATCH) != "unknown status"


def test_timeout_counters_refuse_a_null_destination(lib):
    """The wait time-out counters report through an out-parameter; a NULL
    one is refused on the host (no CUDA call)."""
    assert lib.gdn_prefill_timeouts(None) == gdn.GDN_EINVAL
    assert lib.gdn_wait_timeouts(None) == gdn.GDN_EINVAL
