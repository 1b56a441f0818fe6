"""Degenerate gates on the GPU paths: the identity step (alpha = 1, beta = 0)
and the hard reset (alpha = 0), in the token-serial kernel and in the
chunked tensor-core prefill, against the oracle and against what the gates
fix exactly.

The identity step leaves the state untouched: bit for bit in the
token-serial kernel (S * 1 + k * 0), and also in the chunked kernel, whose
state passes through fp32 tensor memory with a zero correction.  A reset
gate (g = -200, exp(g) = 0 in fp32) makes the state after that token
beta k v^T whatever came before.
"""

import numpy as np
import pytest
import torch

import gated_deltanet_linear_gb300 as gdn
import gdn_inputs
from oracle.ref64 import max_rel
from gpu_util import dev, empty, host, run_step_m

pytestmark = pytest.mark.gpu

TOL_STEP = 1e-5
TOL_MULTI = 1e-4
TOL_CHUNK = {gdn.GDN_PREC_BF16X3: 1e-4, gdn.GDN_PREC_BF16: 8 * 2.0 ** -9}


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _prefill(inp, precision):
    S = dev(inp.S)
    o = empty(inp.B, inp.T, inp.vh, inp.vd)
    gdn.gdn_prefill(S, dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.g),
                    dev(inp.beta), o, precision=precision)
    torch.cuda.synchronize()
    return host(S), host(o)


def _identity(inp):
    inp.g[:] = 0.0
    inp.beta[:] = 0.0
    return inp


def test_identity_step_token_serial(oracle_mod):
    inp = _identity(gdn_inputs.make_inputs(1201, B=3, T=4))
    _, S, _, o = run_step_m(inp, ckpt=False)
    assert np.array_equal(host(S), inp.S.astype(np.float64))
    _, o_ref = oracle_mod.run_inputs(inp)
    assert max_rel(host(o), o_ref, axes=(-2, -1)) < TOL_MULTI


@pytest.mark.parametrize("precision", [gdn.GDN_PREC_BF16X3, gdn.GDN_PREC_BF16])
def test_identity_chunked(oracle_mod, precision):
    inp = _identity(gdn_inputs.make_inputs(1202, B=2, T=130))
    S, o = _prefill(inp, precision)
    assert np.array_equal(S, inp.S.astype(np.float64))
    _, o_ref = oracle_mod.run_inputs(inp)
    assert max_rel(o, o_ref, axes=(-2, -1)) < TOL_CHUNK[precision]
    assert gdn.gdn_prefill_timeouts() == 0


def test_reset_token_serial(oracle_mod):
    """A reset at token 2 of 4: the state after it is beta k v^T of that
    token, whatever the earlier tokens did."""
    inp = gdn_inputs.make_inputs(1203, B=2, T=4)
    inp.g[:, 2] = -200.0
    _, S, ck, o = run_step_m(inp, ckpt=True)
    S_ref, o_ref = oracle_mod.run_inputs(inp)
    assert max_rel(host(S), S_ref, axes=(-2, -1)) < TOL_MULTI
    assert max_rel(host(o), o_ref, axes=(-2, -1)) < TOL_MULTI
    rep = inp.vh // inp.kh
    k2 = np.repeat(inp.k[:, 2].astype(np.float64), rep, axis=1)   # [B][vh][kd]
    want = inp.beta[:, 2, :, None, None] * k2[..., None] * inp.v[:, 2, :, None, :]
    assert max_rel(host(ck)[2], want, axes=(-2, -1)) < TOL_STEP


@pytest.mark.parametrize("precision", [gdn.GDN_PREC_BF16X3, gdn.GDN_PREC_BF16])
def test_reset_inside_chunks(oracle_mod, precision):
    """Resets at a chunk's first, middle and last token and in the ragged
    tail, with strong decay elsewhere."""
    inp = gdn_inputs.make_inputs(1204, B=2, T=150, g_scale=1.0)
    for t in (0, 37, 63, 64, 140):
        inp.g[:, t] = -200.0
    S, o = _prefill(inp, precision)
    S_ref, o_ref = oracle_mod.run_inputs(inp)
    es = max_rel(S, S_ref, axes=(-2, -1))
    eo = max_rel(o, o_ref, axes=(-2, -1))
    print(f"reset chunks {precision}: state {es:.3e} o {eo:.3e}")
    assert es < TOL_CHUNK[precision] and eo < TOL_CHUNK[precision]
    assert gdn.gdn_prefill_timeouts() == 0


@pytest.mark.parametrize("precision", [gdn.GDN_PREC_BF16X3, gdn.GDN_PREC_BF16])
def test_factored_flag_alternates(oracle_mod, precision):
    """Chunks that alternate between the factored exponentials (range of
    Gamma over the chunk at most 160) and one exp per element (a reset in
    the chunk): the kernel keeps the choice per chunk, next to that chunk's
    gate vectors, and the bf16 mode makes chunk c + 1's vectors while chunk
    c still reads its own."""
    inp = gdn_inputs.make_inputs(1206, B=2, T=200, g_scale=0.1)
    for t in (100, 195):  # chunks 1 and 3 of 0..3
        inp.g[:, t] = -200.0
    S, o = _prefill(inp, precision)
    S_ref, o_ref = oracle_mod.run_inputs(inp)
    es = max_rel(S, S_ref, axes=(-2, -1))
    eo = max_rel(o, o_ref, axes=(-2, -1))
    print(f"alternating factored chunks {precision}: state {es:.3e} o {eo:.3e}")
    assert es < TOL_CHUNK[precision] and eo < TOL_CHUNK[precision]
    assert gdn.gdn_prefill_timeouts() == 0


@pytest.mark.parametrize("precision", [gdn.GDN_PREC_BF16X3, gdn.GDN_PREC_BF16])
@pytest.mark.parametrize("g_const", [-2.4, -2.6])
def test_strong_uniform_decay_chunked(oracle_mod, precision, g_const):
    """A constant decay whose range over a 64-token chunk (63 |g|) is just
    under (151) and just over (164) the 160 up to which the kernel splits
    exp(Gamma_t - Gamma_s) into two per-token factors; either side must
    match the oracle."""
    inp = gdn_inputs.make_inputs(1205, B=2, T=130)
    inp.g[:] = g_const
    S, o = _prefill(inp, precision)
    S_ref, o_ref = oracle_mod.run_inputs(inp)
    es = max_rel(S, S_ref, axes=(-2, -1))
    eo = max_rel(o, o_ref, axes=(-2, -1))
    print(f"decay {g_const} {precision}: state {es:.3e} o {eo:.3e}")
    assert es < TOL_CHUNK[precision] and eo < TOL_CHUNK[precision]
    assert gdn.gdn_prefill_timeouts() == 0
