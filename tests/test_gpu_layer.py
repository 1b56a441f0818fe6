"""The layer core (conv1d + SiLU with rolling history, q/k normalisation,
gates) in front of the recurrence, against the layer oracle and against
fp64 closed forms of each step, its exactness across launch splits, and the
history rollback.

Tolerances as in test_gpu_parity.py: normwise per (sequence, token) over
all value heads for o, per (sequence, value head) for the state; 1e-5 for
one token, 1e-4 for several.  The history is a copy of inputs: bit-exact.
"""

import ctypes

import numpy as np
import pytest
import torch

import gated_deltanet_linear_gb300 as gdn
import gdn_inputs
from oracle.ref64 import max_rel
from gpu_util import dev, empty, host

pytestmark = pytest.mark.gpu

TOL_STEP = 1e-5
TOL_MULTI = 1e-4


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def run_layer(L, S=None, hist=None, x=None, a=None, b=None, ckpt=False):
    """One gdn_layer_step_m launch over L's tokens (or the given slices)."""
    S_in = dev(L.S) if S is None else S
    hist_in = dev(L.hist) if hist is None else hist
    x = dev(L.x) if x is None else x
    a = dev(L.a) if a is None else a
    b = dev(L.b) if b is None else b
    B, vh, kd, vd = S_in.shape
    M = x.shape[1]
    S_out = torch.empty_like(S_in)
    hist_out = torch.empty_like(hist_in)
    ck = empty(M, B, vh, kd, vd) if ckpt else None
    o = empty(B, M, vh, vd)
    ws = torch.empty(gdn.gdn_layer_workspace(B, L.kh, vh, M), dtype=torch.uint8,
                     device="cuda")
    gdn.gdn_layer_step_m(S_in, S_out, ck, hist_in, hist_out, x, dev(L.conv_w),
                         a, b, dev(L.A_log), dev(L.dt_bias), o, L.kh, ws)
    return S_out, hist_out, o, ck


@pytest.mark.parametrize("B,M,kh,vh", [(3, 1, 16, 48), (3, 5, 16, 48),
                                       (2, 7, 2, 6), (1, 2, 1, 1)])
def test_layer_vs_oracle(oracle_mod, B, M, kh, vh):
    L = gdn_inputs.make_layer_inputs(900 + M + vh, B=B, T=M, kh=kh, vh=vh)
    S, hist, o, _ = run_layer(L)
    S_ref, hist_ref, o_ref = oracle_mod.run_layer(
        L.S, L.hist, L.x, L.conv_w, L.a, L.b, L.A_log, L.dt_bias, L.kh)
    es = max_rel(host(S), S_ref, axes=(-2, -1))
    eo = max_rel(host(o), o_ref, axes=(-2, -1))
    print(f"layer B={B} M={M} kh={kh} vh={vh}: state {es:.3e} o {eo:.3e}")
    tol = TOL_STEP if M == 1 else TOL_MULTI
    assert es < tol and eo < tol
    assert np.array_equal(host(hist), hist_ref)


def test_prologue_outputs_closed_forms():
    """The prologue's q, k, v, g, beta against fp64 closed forms of each
    step (causal convolution over [history, inputs], SiLU, per-head unit
    norm, softplus and sigmoid gates)."""
    import oracle_pins
    L = gdn_inputs.make_layer_inputs(905, B=3, T=4)
    B, vh = 3, 48
    M = L.T
    q = empty(B, M, L.kh, 128)
    k = torch.empty_like(q)
    v = empty(B, M, vh, 128)
    g = empty(B, M, vh)
    beta = torch.empty_like(g)
    hist_out = torch.empty_like(dev(L.hist))
    gdn.gdn_layer_prologue_m(dev(L.hist), hist_out, dev(L.x), dev(L.conv_w),
                             dev(L.a), dev(L.b), dev(L.A_log),
                             dev(L.dt_bias), q, k, v, g, beta, L.kh)
    q64, k64, v64, g64, b64, h64 = oracle_pins._layer_inputs64(
        L.hist, L.x, L.conv_w, L.a, L.b, L.A_log, L.dt_bias, L.kh, 128, vh,
        128)
    for got, ref in ((q, q64), (k, k64), (v, v64)):
        assert max_rel(host(got), ref, axes=(-2, -1)) < 2e-6
    assert max_rel(host(g), g64) < 2e-6 and max_rel(host(beta), b64) < 2e-6
    assert np.array_equal(host(hist_out), h64.astype(np.float32))


def test_layer_decode_full_size(oracle_mod):
    """64 sequences x 48 heads, one token, every head against the oracle."""
    L = gdn_inputs.make_layer_inputs(911, B=64, T=1)
    S, hist, o, _ = run_layer(L)
    S_ref, hist_ref, o_ref = oracle_mod.run_layer(
        L.S, L.hist, L.x, L.conv_w, L.a, L.b, L.A_log, L.dt_bias, L.kh)
    es = max_rel(host(S), S_ref, axes=(-2, -1))
    eo = max_rel(host(o), o_ref, axes=(-2, -1))
    print(f"layer decode B=64: state {es:.3e} o {eo:.3e}")
    assert es < TOL_STEP and eo < TOL_STEP
    assert np.array_equal(host(hist), hist_ref)


def test_layer_m_tokens_bit_exact_vs_single_launches():
    """M tokens in one launch equal M one-token launches that pass the
    history forward (two history buffers in turn), bit for bit: o, every
    checkpoint, the final state and the final history."""
    M = 6
    L = gdn_inputs.make_layer_inputs(921, B=4, T=M)
    S_m, hist_m, o_m, ck_m = run_layer(L, ckpt=True)
    S = dev(L.S)
    hist = dev(L.hist)
    x, a, b = dev(L.x), dev(L.a), dev(L.b)
    for m in range(M):
        S, hist, o1, _ = run_layer(L, S=S, hist=hist,
                                   x=x[:, m:m + 1].contiguous(),
                                   a=a[:, m:m + 1].contiguous(),
                                   b=b[:, m:m + 1].contiguous())
        assert torch.equal(o1[:, 0], o_m[:, m]), m
        assert torch.equal(S, ck_m[m]), m
    assert torch.equal(S, S_m) and torch.equal(hist, hist_m)


def test_layer_history_rollback():
    """History after m of the M tokens, restored per sequence from the
    launch's input history and raw inputs, equals the history m one-token
    launches produce; an out-of-range count is refused on the device."""
    M = 5
    L = gdn_inputs.make_layer_inputs(931, B=6, T=M)
    hist0 = dev(L.hist)
    x, a, b = dev(L.x), dev(L.a), dev(L.b)
    hists = [hist0]
    S = dev(L.S)
    for m in range(M):
        S, h, _, _ = run_layer(L, S=S, hist=hists[-1],
                               x=x[:, m:m + 1].contiguous(),
                               a=a[:, m:m + 1].contiguous(),
                               b=b[:, m:m + 1].contiguous())
        hists.append(h)
    counts = [0, 1, 2, 3, 5, 7]
    m_dev = torch.tensor(counts, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sentinel = torch.full_like(hist0, 123.0)
    out = sentinel.clone()
    gdn.gdn_layer_hist_rollback(out, M, m_dev, hist0, x, L.kh, err_dev=err)
    torch.cuda.synchronize()
    for bi, m in enumerate(counts):
        want = sentinel[bi] if m > M else hists[m][bi]
        assert torch.equal(out[bi], want), bi
    assert int(err.item()) == 1


def test_layer_refusals():
    lib = gdn.load()
    L = gdn_inputs.make_layer_inputs(941, B=1, T=2)
    B, vh = 1, 48
    sh = gdn.Shape(B, L.kh, vh, 128, 128)
    S = dev(L.S)
    hist = dev(L.hist)
    hist2 = torch.empty_like(hist)
    x, w, a, b = dev(L.x), dev(L.conv_w), dev(L.a), dev(L.b)
    Al, dt = dev(L.A_log), dev(L.dt_bias)
    o = empty(B, 2, vh, 128)
    st = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()

    need = gdn.gdn_layer_workspace(B, L.kh, vh, 2)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def call(ck=4, eps=1e-6, h_out=None, ws_bytes=need, ws_ptr=None):
        return lib.gdn_layer_step_m(
            ctypes.byref(sh), 2, ck, eps, P(S), P(S), None, P(hist),
            P(hist2 if h_out is None else h_out), P(x), P(w), P(a), P(b),
            P(Al), P(dt), P(o), P(ws) if ws_ptr is None else ws_ptr,
            ws_bytes, st)

    assert call() == gdn.GDN_OK
    assert call(ck=3) == gdn.GDN_ESHAPE
    assert call(eps=-1.0) == gdn.GDN_EINVAL
    assert call(h_out=hist) == gdn.GDN_EALIAS   # in-place history refused
    assert call(ws_bytes=need - 16) == gdn.GDN_ERANGE
    assert call(ws_ptr=P(S)) == gdn.GDN_EALIAS  # workspace over the state
    torch.cuda.synchronize()
