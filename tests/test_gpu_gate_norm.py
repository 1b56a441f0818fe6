"""The gated RMSNorm epilogue against the oracle, alone and behind the layer
step (conv1d + SiLU, q/k norm, gates, update, then the norm: the layer core
from raw projections to the normalised output).

Tolerance: normwise per (sequence, token, value head) row, 1e-5 for a single
token (the sum of squares is a tree on the GPU and a left fold in the
oracle), 1e-4 where several tokens of the update come first.
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


@pytest.mark.parametrize("B,M,vh", [(3, 1, 48), (2, 5, 6), (1, 1, 3),
                                    (64, 1, 48), (32, 8, 48)])
def test_gate_norm_vs_oracle(oracle_mod, B, M, vh):
    o, z, w = gdn_inputs.make_gate_norm_inputs(970 + B + M, B, M, vh)
    y = empty(B, M, vh, 128)
    gdn.gdn_gated_rmsnorm_m(dev(o), dev(z), dev(w), y)
    ref = oracle_mod.run_gate_norm(o, z, w)
    e = max_rel(host(y), ref, axes=(-1,))
    print(f"gate norm B={B} M={M} vh={vh}: {e:.3e}")
    assert e < TOL_STEP


def test_gate_norm_in_place_equals_out_of_place():
    o, z, w = gdn_inputs.make_gate_norm_inputs(981, 4, 3, 48)
    od, zd, wd = dev(o), dev(z), dev(w)
    y = torch.empty_like(od)
    gdn.gdn_gated_rmsnorm_m(od, zd, wd, y)
    gdn.gdn_gated_rmsnorm_m(od, zd, wd, od)
    assert torch.equal(od, y)


def test_layer_core_to_normalised_output(oracle_mod):
    """gdn_layer_step_m writing o, then the norm in place on it, against
    the layer oracle followed by the norm oracle."""
    for B, M in ((4, 1), (3, 4)):
        L = gdn_inputs.make_layer_inputs(991 + M, B=B, T=M)
        _, z, w = gdn_inputs.make_gate_norm_inputs(995 + M, B, M, 48)
        S_out = torch.empty_like(dev(L.S))
        hist_out = torch.empty_like(dev(L.hist))
        y = empty(B, M, 48, 128)
        ws = torch.empty(gdn.gdn_layer_workspace(B, L.kh, 48, M),
                         dtype=torch.uint8, device="cuda")
        gdn.gdn_layer_step_m(dev(L.S), S_out, None, dev(L.hist), hist_out,
                             dev(L.x), dev(L.conv_w), dev(L.a), dev(L.b),
                             dev(L.A_log), dev(L.dt_bias), y, L.kh, ws)
        gdn.gdn_gated_rmsnorm_m(y, dev(z), dev(w), y)
        _, _, o_ref = oracle_mod.run_layer(L.S, L.hist, L.x, L.conv_w, L.a,
                                           L.b, L.A_log, L.dt_bias, L.kh)
        y_ref = oracle_mod.run_gate_norm(o_ref, z, w)
        e = max_rel(host(y), y_ref, axes=(-1,))
        print(f"layer core + norm B={B} M={M}: {e:.3e}")
        assert e < (TOL_STEP if M == 1 else TOL_MULTI)


def test_gate_norm_refusals():
    lib = gdn.load()
    o, z, w = gdn_inputs.make_gate_norm_inputs(999, 2, 1, 48)
    od, zd, wd = dev(o), dev(z), dev(w)
    big = torch.empty(2 * od.numel(), device="cuda")
    sh = gdn.Shape(2, 16, 48, 128, 128)
    st = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()

    def call(y, eps=1e-6, zp=None):
        return lib.gdn_gated_rmsnorm_m(ctypes.byref(sh), 1, eps, P(od),
                                       zp or P(zd), P(wd), y, st)

    assert call(P(big)) == gdn.GDN_OK
    assert call(P(od)) == gdn.GDN_OK                    # in place
    assert call(P(big), eps=-1.0) == gdn.GDN_EINVAL
    assert call(P(od) + 16) == gdn.GDN_EALIAS           # shifted over o
    assert call(P(zd)) == gdn.GDN_EALIAS                # over the gate
    assert call(P(big) + 4) == gdn.GDN_EALIGN
    torch.cuda.synchronize()
