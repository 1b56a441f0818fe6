"""gdn_layer_step_m_noalloc, the layer step that keeps its intermediates in
the library's static scratch instead of a caller workspace, against
gdn_layer_step_m on the same inputs, through the C ABI.

Two calls in a row: the second is smaller than the first and chains from its
state and history, so anything the first call left in the shared scratch that
the second read would show up as a mismatch.  Both entry points run the same
kernels on the same inputs, only the address of the intermediates differs,
so S, o, the checkpoints and the history must match bit for bit.  The
normwise error is also printed, with the layer tests' tolerances as a
sanity bar (1e-4 for several tokens, 1e-5 for one).
"""

import ctypes

import numpy as np
import pytest
import torch

import gated_deltanet_linear_gb300 as gdn
import gdn_inputs
from gated_deltanet_linear_gb300 import _build
from oracle.ref64 import max_rel

TOL_STEP = 1e-5
TOL_MULTI = 1e-4


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def _host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy().astype(np.float64)


def test_noalloc_checks_arguments_before_the_scratch_size():
    """Argument errors keep gdn_layer_step_m's status even for a request too
    large for the scratch (no GPU needed: every case is refused on the host
    before any buffer is looked at on a device)."""
    _build.build()
    lib = gdn.load()
    null = [None] * 12
    per_token = gdn.gdn_layer_workspace(1, 16, 48, 1)
    assert per_token == 41344
    fits = gdn.GDN_NOALLOC_SCRATCH_BYTES // per_token        # B * M = 405
    big = gdn.Shape(fits + 1, 16, 48, 128, 128)
    # oversized and NULL buffers: the NULL is reported, as gdn_layer_step_m
    assert lib.gdn_layer_step_m_noalloc(ctypes.byref(big), 1, 4, 1e-6, *null,
                                        None) == gdn.GDN_EINVAL
    # oversized and a bad conv width / eps / token count
    assert lib.gdn_layer_step_m_noalloc(ctypes.byref(big), 1, 3, 1e-6, *null,
                                        None) == gdn.GDN_ESHAPE
    assert lib.gdn_layer_step_m_noalloc(ctypes.byref(big), 1, 4, -1.0, *null,
                                        None) == gdn.GDN_EINVAL
    assert lib.gdn_layer_step_m_noalloc(ctypes.byref(big), 0, 4, 1e-6, *null,
                                        None) == gdn.GDN_ERANGE
    bad = gdn.Shape(1, 16, 48, 64, 128)
    assert lib.gdn_layer_step_m_noalloc(ctypes.byref(bad), 1, 4, 1e-6, *null,
                                        None) == gdn.GDN_ESHAPE
    assert lib.gdn_layer_step_m_noalloc(None, 1, 4, 1e-6, *null,
                                        None) == gdn.GDN_EINVAL
    # B == 0 is a no-op, whatever the token count
    empty = gdn.Shape(0, 16, 48, 128, 128)
    assert lib.gdn_layer_step_m_noalloc(ctypes.byref(empty), fits + 1, 4, 1e-6,
                                        *null, None) == gdn.GDN_OK
    assert "static scratch" in gdn.gdn_strerror(gdn.GDN_ESCRATCH)


def _run(L, S_in, hist_in, x, a, b, noalloc, ckpt=False):
    """One layer step over x's tokens: the no-alloc entry point called
    directly through the C ABI, or gdn_layer_step_m with a workspace."""
    B, vh, kd, vd = S_in.shape
    M = x.shape[1]
    S_out = torch.empty_like(S_in)
    hist_out = torch.empty_like(hist_in)
    o = torch.empty(B, M, vh, vd, device="cuda")
    ck = torch.empty(M, B, vh, kd, vd, device="cuda") if ckpt else None
    conv_w, A_log, dt_bias = _dev(L.conv_w), _dev(L.A_log), _dev(L.dt_bias)
    if noalloc:
        sh = gdn.Shape(B, L.kh, vh, kd, vd)
        P = lambda t: None if t is None else t.data_ptr()
        rc = gdn.load().gdn_layer_step_m_noalloc(
            ctypes.byref(sh), M, 4, 1e-6, P(S_in), P(S_out), P(ck),
            P(hist_in), P(hist_out), P(x), P(conv_w), P(a), P(b), P(A_log),
            P(dt_bias), P(o), torch.cuda.current_stream().cuda_stream)
        assert rc == gdn.GDN_OK, gdn.gdn_strerror(rc)
    else:
        ws = torch.empty(gdn.gdn_layer_workspace(B, L.kh, vh, M),
                         dtype=torch.uint8, device="cuda")
        gdn.gdn_layer_step_m(S_in, S_out, ck, hist_in, hist_out, x, conv_w,
                             a, b, A_log, dt_bias, o, L.kh, ws)
    return S_out, hist_out, o, ck


def _bitwise(got, ref, what):
    assert torch.equal(got, ref), f"{what}: no-alloc result differs from " \
        "gdn_layer_step_m"


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    B = 6
    L1 = gdn_inputs.make_layer_inputs(961, B=B, T=5)
    L2 = gdn_inputs.make_layer_inputs(962, B=B, T=1)
    S0, h0 = _dev(L1.S), _dev(L1.hist)

    # call 1: five tokens with checkpoints (the larger use of the scratch)
    x1, a1, b1 = _dev(L1.x), _dev(L1.a), _dev(L1.b)
    got1 = _run(L1, S0, h0, x1, a1, b1, noalloc=True, ckpt=True)
    ref1 = _run(L1, S0, h0, x1, a1, b1, noalloc=False, ckpt=True)
    es = max_rel(_host(got1[0]), _host(ref1[0]), axes=(-2, -1))
    eo = max_rel(_host(got1[2]), _host(ref1[2]), axes=(-2, -1))
    ec = max_rel(_host(got1[3]), _host(ref1[3]), axes=(-2, -1))
    print(f"no-alloc call 1 (M=5): state {es:.3e} o {eo:.3e} ckpt {ec:.3e}")
    assert es < TOL_MULTI and eo < TOL_MULTI and ec < TOL_MULTI
    for got, ref, what in zip(got1, ref1, ("state", "history", "o", "ckpt")):
        _bitwise(got, ref, f"call 1 {what}")

    # call 2: one more token of the same layer, chained from each side's own
    # state and history
    x2, a2, b2 = _dev(L2.x), _dev(L2.a), _dev(L2.b)
    got2 = _run(L1, got1[0], got1[1], x2, a2, b2, noalloc=True)
    ref2 = _run(L1, ref1[0], ref1[1], x2, a2, b2, noalloc=False)
    es = max_rel(_host(got2[0]), _host(ref2[0]), axes=(-2, -1))
    eo = max_rel(_host(got2[2]), _host(ref2[2]), axes=(-2, -1))
    print(f"no-alloc call 2 (M=1): state {es:.3e} o {eo:.3e}")
    assert es < TOL_STEP and eo < TOL_STEP
    for got, ref, what in zip(got2[:3], ref2[:3], ("state", "history", "o")):
        _bitwise(got, ref, f"call 2 {what}")


@pytest.mark.gpu
def test_noalloc_refuses_a_valid_request_larger_than_the_scratch():
    """With every buffer valid, B * M beyond the scratch gives GDN_ESCRATCH
    and launches nothing (the outputs keep their contents)."""
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    per_token = gdn.gdn_layer_workspace(1, 16, 48, 1)
    M = gdn.GDN_NOALLOC_SCRATCH_BYTES // per_token + 1          # 406 tokens
    conv_dim = 2 * 16 * 128 + 48 * 128
    S_in = torch.zeros(1, 48, 128, 128, device="cuda")
    S_out = torch.full_like(S_in, 7.0)
    hist_in = torch.zeros(1, 3, conv_dim, device="cuda")
    hist_out = torch.full_like(hist_in, 7.0)
    x = torch.zeros(1, M, conv_dim, device="cuda")
    conv_w = torch.zeros(conv_dim, 4, device="cuda")
    a = torch.zeros(1, M, 48, device="cuda")
    b = torch.zeros(1, M, 48, device="cuda")
    A_log = torch.zeros(48, device="cuda")
    dt_bias = torch.zeros(48, device="cuda")
    o = torch.full((1, M, 48, 128), 7.0, device="cuda")
    sh = gdn.Shape(1, 16, 48, 128, 128)
    P = lambda t: t.data_ptr()
    rc = gdn.load().gdn_layer_step_m_noalloc(
        ctypes.byref(sh), M, 4, 1e-6, P(S_in), P(S_out), None, P(hist_in),
        P(hist_out), P(x), P(conv_w), P(a), P(b), P(A_log), P(dt_bias), P(o),
        torch.cuda.current_stream().cuda_stream)
    assert rc == gdn.GDN_ESCRATCH
    torch.cuda.synchronize()
    assert bool((S_out == 7.0).all() and (hist_out == 7.0).all()
                and (o == 7.0).all())
    # one token fewer fits
    rc = gdn.load().gdn_layer_step_m_noalloc(
        ctypes.byref(sh), M - 1, 4, 1e-6, P(S_in), P(S_out), None, P(hist_in),
        P(hist_out), P(x), P(conv_w), P(a), P(b), P(A_log), P(dt_bias), P(o),
        torch.cuda.current_stream().cuda_stream)
    assert rc == gdn.GDN_OK, gdn.gdn_strerror(rc)
    torch.cuda.synchronize()
