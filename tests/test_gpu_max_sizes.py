"""Launches whose buffers hold more than 2^31 elements.

Every kernel addresses its buffers with 64-bit offsets; these cases put
the last rows of a launch past element 2^31 of its buffers, so an offset
kept in 32 bits anywhere would read or write the wrong rows.

Long sequences (token buffers beyond 2^31 elements).  The
bulk of each sequence is drawn on the GPU (seeded; unit-norm q and k,
gates of the workload recipe).  The last two tokens come from
gdn_inputs, with a reset gate at the first of them (g = -200: exp(g) is 0
in fp32, so the state after it no longer depends on what came before).
Their outputs and the final state must then be those of the same two
tokens launched alone from any state:
- bit for bit on the token-serial kernels, whose result for a token
  depends only on the state and that token's inputs (a reset state is
  k tmp^T whatever the earlier state was);
- to the precision's tolerance against the oracle on the chunked path.

Sizes: 48 value heads (16 key heads); one sequence of 350,000 tokens for
the 8-column kernel (48 heads, fewer than SMs), four of 90,000 for the
head-per-CTA kernel (192 heads), two of 350,000 for the chunked prefill
(whose limit is T * vh < 2^31 per sequence).

Many sequences (state or checkpoint buffers beyond 2^31 elements): the
last sequence gets the same state and tokens as the first, so its results
must be the first's bit for bit, and the first's are checked against the
oracle.

Up to about 46 GB on the device.
"""

import numpy as np
import pytest
import torch

import gated_deltanet_linear_gb300 as gdn
import gdn_inputs
from oracle.ref64 import max_rel
from gpu_util import dev, empty, host

pytestmark = pytest.mark.gpu

KH, VH, D = 16, 48, 128
RESET_G = -200.0
TOL_MULTI = 1e-4
TOL_CHUNK = {gdn.GDN_PREC_BF16X3: 1e-4, gdn.GDN_PREC_BF16: 8 * 2.0 ** -9}


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.empty_cache()


def _long_inputs(seed, B, T):
    """q, k, v, g, beta of B sequences x T tokens on the device; tokens
    T-2 and T-1 are those of `tail` (returned), with the reset at T-2."""
    gen = torch.Generator(device="cuda").manual_seed(seed)

    def unit(x):
        return x / x.norm(dim=-1, keepdim=True)

    q = unit(torch.randn(B, T, KH, D, device="cuda", generator=gen))
    k = unit(torch.randn(B, T, KH, D, device="cuda", generator=gen))
    v = torch.randn(B, T, VH, D, device="cuda", generator=gen)
    g = -torch.nn.functional.softplus(
        torch.randn(B, T, VH, device="cuda", generator=gen))
    beta = torch.sigmoid(torch.randn(B, T, VH, device="cuda", generator=gen))
    tail = gdn_inputs.make_inputs(seed, B=B, T=2)
    tail.g[:, 0] = RESET_G
    for big, small in ((q, tail.q), (k, tail.k), (v, tail.v), (g, tail.g),
                       (beta, tail.beta)):
        big[:, T - 2:] = dev(small)
    assert B * T * VH * D > 2 ** 31
    return (q, k, v, g, beta), tail


def _tail_launch(tail):
    S = dev(tail.S)
    o = empty(tail.B, 2, VH, D)
    gdn.gdn_step_m(S, S, None, *(dev(x) for x in (tail.q, tail.k, tail.v,
                                                  tail.g, tail.beta)), o)
    return S, o


@pytest.mark.parametrize("B,T", [(1, 350_000), (4, 90_000)])
def test_token_serial_beyond_2_31_elements(oracle_mod, B, T):
    ins, tail = _long_inputs(7100 + B, B, T)
    S = dev(gdn_inputs.make_inputs(7200 + B, B=B, T=1).S)
    o = torch.empty(B, T, VH, D, device="cuda")
    gdn.gdn_step_m(S, S, None, *ins, o)
    o_tail = o[:, T - 2:].contiguous()
    assert torch.isfinite(o_tail).all()
    del ins, o
    torch.cuda.empty_cache()
    S2, o2 = _tail_launch(tail)
    assert torch.equal(S, S2)
    assert torch.equal(o_tail, o2)
    S_ref, o_ref = oracle_mod.run_inputs(tail)
    assert max_rel(host(S), S_ref, axes=(-2, -1)) < TOL_MULTI
    assert max_rel(host(o_tail), o_ref, axes=(-2, -1)) < TOL_MULTI
    assert gdn.gdn_wait_timeouts() == 0


@pytest.mark.parametrize("precision", [gdn.GDN_PREC_BF16X3, gdn.GDN_PREC_BF16])
def test_chunked_beyond_2_31_elements(oracle_mod, precision):
    B, T = 2, 350_000                      # last chunk: 48 tokens (ragged)
    ins, tail = _long_inputs(7300 + precision, B, T)
    S = torch.zeros(B, VH, D, D, device="cuda")
    o = torch.empty(B, T, VH, D, device="cuda")
    gdn.gdn_prefill(S, *ins, o, precision=precision)
    o_tail = o[:, T - 2:].contiguous()
    del ins, o
    torch.cuda.empty_cache()
    assert gdn.gdn_prefill_timeouts() == 0
    S_ref, o_ref = oracle_mod.run_inputs(tail)
    es = max_rel(host(S), S_ref, axes=(-2, -1))
    eo = max_rel(host(o_tail), o_ref, axes=(-2, -1))
    print(f"chunked {precision}, {B} x {T} tokens: state {es:.3e} o {eo:.3e}")
    assert es < TOL_CHUNK[precision] and eo < TOL_CHUNK[precision]


def _wide_inputs(seed, B, M):
    """B sequences x M tokens on the device, sequences 0 and B-1 both
    holding the state and tokens of `one` (returned, B = 1)."""
    gen = torch.Generator(device="cuda").manual_seed(seed)

    def unit(x):
        return x / x.norm(dim=-1, keepdim=True)

    S = torch.randn(B, VH, D, D, device="cuda", generator=gen).mul_(0.02)
    q = unit(torch.randn(B, M, KH, D, device="cuda", generator=gen))
    k = unit(torch.randn(B, M, KH, D, device="cuda", generator=gen))
    v = torch.randn(B, M, VH, D, device="cuda", generator=gen)
    g = -torch.nn.functional.softplus(
        torch.randn(B, M, VH, device="cuda", generator=gen))
    beta = torch.sigmoid(torch.randn(B, M, VH, device="cuda", generator=gen))
    one = gdn_inputs.make_inputs(seed, B=1, T=M)
    for big, small in ((S, one.S), (q, one.q), (k, one.k), (v, one.v),
                       (g, one.g), (beta, one.beta)):
        big[0] = dev(small)[0]
        big[B - 1] = dev(small)[0]
    return S, (q, k, v, g, beta), one


# (sequences, tokens, checkpoints): a state of 2,800 x 48 heads is 8.8 GB
# (more than 2^31 elements), for one token (32-column kernel) and two
# (head-per-CTA kernel); 400 x 48 heads x 8 tokens of checkpoints are 10 GB
# (8-column kernel)
WIDE = [(2800, 1, False), (2800, 2, False), (400, 8, True)]


@pytest.mark.parametrize("B,M,ckpt", WIDE)
def test_state_beyond_2_31_elements(oracle_mod, B, M, ckpt):
    S, ins, one = _wide_inputs(7400 + M, B, M)
    assert S.numel() * (M if ckpt else 1) > 2 ** 31
    o = torch.empty(B, M, VH, D, device="cuda")
    ck = torch.empty(M, B, VH, D, D, device="cuda") if ckpt else None
    if M == 1:
        gdn.gdn_step(S, *ins, o)
    else:
        gdn.gdn_step_m(S, S, ck, *ins, o)
    torch.cuda.synchronize()
    assert torch.equal(S[B - 1], S[0]) and torch.equal(o[B - 1], o[0])
    if ckpt:
        assert torch.equal(ck[:, B - 1], ck[:, 0])
    S_ref, o_ref = oracle_mod.run_inputs(one)
    tol = 1e-5 if M == 1 else TOL_MULTI
    assert max_rel(host(S[:1]), S_ref, axes=(-2, -1)) < tol
    assert max_rel(host(o[:1]), o_ref, axes=(-2, -1)) < tol
    assert gdn.gdn_wait_timeouts() == 0
    del S, ins, o, ck
    torch.cuda.empty_cache()


@pytest.mark.parametrize("precision", [gdn.GDN_PREC_BF16X3, gdn.GDN_PREC_BF16])
def test_chunked_state_beyond_2_31_elements(oracle_mod, precision):
    B, T = 2800, 70                        # two chunks, the second ragged
    S, ins, one = _wide_inputs(7500 + precision, B, T)
    o = torch.empty(B, T, VH, D, device="cuda")
    gdn.gdn_prefill(S, *ins, o, precision=precision)
    torch.cuda.synchronize()
    assert gdn.gdn_prefill_timeouts() == 0
    assert torch.equal(S[B - 1], S[0]) and torch.equal(o[B - 1], o[0])
    S_ref, o_ref = oracle_mod.run_inputs(one)
    es = max_rel(host(S[:1]), S_ref, axes=(-2, -1))
    eo = max_rel(host(o[:1]), o_ref, axes=(-2, -1))
    assert es < TOL_CHUNK[precision] and eo < TOL_CHUNK[precision]
    del S, ins, o
    torch.cuda.empty_cache()


def test_layer_step_beyond_2_31_elements(oracle_mod):
    """The layer step (convolution with history, normalisation, gates, then
    the update) over one sequence of 210,000 tokens, whose raw projections
    x hold more than 2^31 elements.  The last five rows of x, a and b come
    from gdn_inputs; a = 1e4 at token T-2 makes g about -1e4 there, a reset.
    The last two tokens then depend only on those five rows (three of
    convolution history and two tokens): a launch of the two tokens with
    the three rows as its history must give the same state, history and
    outputs bit for bit, and the oracle agrees with them."""
    T = 210_000
    L = gdn_inputs.make_layer_inputs(7600, B=1, T=5)
    conv_dim = L.x.shape[-1]
    assert T * conv_dim > 2 ** 31
    a_tail = L.a.copy()
    a_tail[:, 3] = 1e4
    gen = torch.Generator(device="cuda").manual_seed(7601)
    x = torch.randn(1, T, conv_dim, device="cuda", generator=gen)
    a = torch.randn(1, T, VH, device="cuda", generator=gen)
    b = torch.randn(1, T, VH, device="cuda", generator=gen)
    x[:, T - 5:] = dev(L.x)
    a[:, T - 5:] = dev(a_tail)
    b[:, T - 5:] = dev(L.b)
    w = [dev(t) for t in (L.conv_w, L.A_log, L.dt_bias)]

    def launch(S_in, hist_in, x_, a_, b_):
        M = x_.shape[1]
        S_out = torch.empty_like(S_in)
        hist_out = torch.empty_like(hist_in)
        o = torch.empty(1, M, VH, D, device="cuda")
        ws = torch.empty(gdn.gdn_layer_workspace(1, L.kh, VH, M),
                         dtype=torch.uint8, device="cuda")
        gdn.gdn_layer_step_m(S_in, S_out, None, hist_in, hist_out, x_, w[0],
                             a_, b_, w[1], w[2], o, L.kh, ws)
        torch.cuda.synchronize()
        return S_out, hist_out, o

    S_big, h_big, o_big = launch(dev(L.S), dev(L.hist), x, a, b)
    o_big = o_big[:, T - 2:].contiguous()
    del x, a, b
    torch.cuda.empty_cache()
    x5, a5, b5 = dev(L.x), dev(a_tail), dev(L.b)
    S2, h2, o2 = launch(dev(L.S), x5[:, :3].contiguous(), x5[:, 3:].contiguous(),
                        a5[:, 3:].contiguous(), b5[:, 3:].contiguous())
    assert torch.equal(S_big, S2) and torch.equal(h_big, h2)
    assert torch.equal(o_big, o2)
    S_ref, h_ref, o_ref = oracle_mod.run_layer(
        L.S, L.x[:, :3], L.x[:, 3:], L.conv_w, a_tail[:, 3:], L.b[:, 3:],
        L.A_log, L.dt_bias, L.kh)
    assert np.array_equal(host(h2), h_ref)
    assert max_rel(host(S2), S_ref, axes=(-2, -1)) < TOL_MULTI
    assert max_rel(host(o2), o_ref, axes=(-2, -1)) < TOL_MULTI
