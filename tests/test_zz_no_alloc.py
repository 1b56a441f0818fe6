"""gdn_layer_step_m_noalloc, the layer step that keeps its intermediates in
the library's static scratch instead of a caller workspace, against
gdn_layer_step_m on the same inputs, through the C ABI.

Two calls in a row: the second is smaller than the first and chains from its
state and history, so anything the first call left in the shared scratch that
the second read would show up as a mismatch.  Tolerances as in
test_gpu_layer.py (normwise; 1e-4 for several tokens, 1e-5 for one); the
history is a copy of inputs and must match bit for bit.
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


def test_noalloc_refuses_oversized_requests_on_the_host():
    """A request beyond the static scratch is refused before any CUDA call
    (no GPU needed); shape errors keep gdn_layer_step_m's status."""
    _build.build()
    lib = gdn.load()
    null = [None] * 12
    per_token = gdn.gdn_layer_workspace(1, 16, 48, 1)
    assert per_token == 41344
    fits = gdn.GDN_NOALLOC_SCRATCH_BYTES // per_token        # B * M = 405
    big = gdn.Shape(fits + 1, 16, 48, 128, 128)
    assert lib.gdn_layer_step_m_noalloc(ctypes.byref(big), 1, 4, 1e-6, *null,
                                        None) == gdn.GDN_ESCRATCH
    big = gdn.Shape(1, 16, 48, 128, 128)
    assert lib.gdn_layer_step_m_noalloc(ctypes.byref(big), fits + 1, 4, 1e-6,
                                        *null, None) == gdn.GDN_ESCRATCH
    bad = gdn.Shape(1, 16, 48, 64, 128)
    assert lib.gdn_layer_step_m_noalloc(ctypes.byref(bad), 1, 4, 1e-6, *null,
                                        None) == gdn.GDN_ESHAPE
    assert lib.gdn_layer_step_m_noalloc(None, 1, 4, 1e-6, *null,
                                        None) == gdn.GDN_EINVAL
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
    assert torch.equal(got1[1], ref1[1])

    # call 2: one more token of the same layer, chained from each side's own
    # state and history
    x2, a2, b2 = _dev(L2.x), _dev(L2.a), _dev(L2.b)
    got2 = _run(L1, got1[0], got1[1], x2, a2, b2, noalloc=True)
    ref2 = _run(L1, ref1[0], ref1[1], x2, a2, b2, noalloc=False)
    es = max_rel(_host(got2[0]), _host(ref2[0]), axes=(-2, -1))
    eo = max_rel(_host(got2[2]), _host(ref2[2]), axes=(-2, -1))
    print(f"no-alloc call 2 (M=1): state {es:.3e} o {eo:.3e}")
    assert es < TOL_STEP and eo < TOL_STEP
    assert torch.equal(got2[1], ref2[1])
