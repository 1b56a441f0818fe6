"""Degenerate gates and empty batches on every update kernel.

The launches below reach each layout of the token-serial update: the
32-column single-token kernel (one token, no checkpoints), the head-per-CTA
kernel (several tokens, no checkpoints, at least one head per SM) and the
8-column kernel (checkpoints, or fewer heads than SMs).

- Identity gates (g = 0, so alpha = 1, and beta = 0) leave the state
  unchanged bit for bit, and o is S^T q (checked against fp64).
- A decay of g = -inf at one token (alpha = exp(-inf) = 0) resets the state
  to beta k v^T of that token, whatever came before; the result stays
  finite and agrees with the oracle.
- B = 0 is a no-op that returns GDN_OK on every entry point.
"""

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

# (B, M, checkpoints): 4 x 48 = 192 heads, at least one per SM of a GB300;
# one sequence, 48 heads, fewer
LAUNCHES = [(4, 1, False), (4, 3, False), (4, 3, True), (1, 3, False)]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _launch(inp, ckpt):
    S = dev(inp.S)
    o = empty(inp.B, inp.T, inp.vh, inp.vd)
    ck = empty(inp.T, *inp.S.shape) if ckpt else None
    ins = [dev(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta)]
    if inp.T == 1 and not ckpt:
        gdn.gdn_step(S, *ins, o)
    else:
        gdn.gdn_step_m(S, S, ck, *ins, o)
    torch.cuda.synchronize()
    return S, o, ck


@pytest.mark.parametrize("B,M,ckpt", LAUNCHES)
def test_identity_gates(B, M, ckpt):
    inp = gdn_inputs.make_inputs(3100 + 10 * B + M, B=B, T=M)
    inp.g[:] = 0.0
    inp.beta[:] = 0.0
    S, o, ck = _launch(inp, ckpt)
    assert torch.equal(S, dev(inp.S))
    if ckpt:
        for m in range(M):
            assert torch.equal(ck[m], dev(inp.S)), m
    rep = inp.vh // inp.kh
    q = np.repeat(inp.q.astype(np.float64), rep, axis=2)           # [B][M][vh][kd]
    want = np.einsum("bvkd,bmvk->bmvd", inp.S.astype(np.float64), q)
    assert max_rel(host(o), want, axes=(-1,)) < TOL_STEP


@pytest.mark.parametrize("B,M,ckpt", LAUNCHES)
def test_minus_infinity_decay_resets(oracle_mod, B, M, ckpt):
    inp = gdn_inputs.make_inputs(3200 + 10 * B + M, B=B, T=M)
    t = M - 1
    inp.g[:, t] = -np.inf
    S, o, ck = _launch(inp, ckpt)
    assert torch.isfinite(S).all() and torch.isfinite(o).all()
    rep = inp.vh // inp.kh
    kt = np.repeat(inp.k[:, t].astype(np.float64), rep, axis=1)    # [B][vh][kd]
    want = inp.beta[:, t, :, None, None] * kt[..., None] * inp.v[:, t, :, None, :]
    assert max_rel(host(S), want, axes=(-2, -1)) < TOL_STEP
    S_ref, o_ref = oracle_mod.run_inputs(inp)
    tol = TOL_STEP if M == 1 else TOL_MULTI
    assert max_rel(host(S), S_ref, axes=(-2, -1)) < tol
    assert max_rel(host(o), o_ref, axes=(-2, -1)) < tol


def test_empty_batch_every_entry_point():
    """B = 0 with empty tensors: every call returns without error."""
    S = empty(0, 48, 128, 128)
    q = empty(0, 4, 16, 128)
    v = empty(0, 4, 48, 128)
    g = empty(0, 4, 48)
    o = empty(0, 4, 48, 128)
    gdn.gdn_step_m(S, S, None, q, q, v, g, g, o)
    gdn.gdn_step_m(S, S, empty(4, 0, 48, 128, 128), q, q, v, g, g, o)
    for prec in (gdn.GDN_PREC_FP32, gdn.GDN_PREC_BF16X3, gdn.GDN_PREC_BF16):
        gdn.gdn_prefill(S, q, q, v, g, g, o, precision=prec)
    snap = empty(0, 48, 128, 128)
    gdn.gdn_mark(S, snap, 16)
    gdn.gdn_rollback(S, 4, 0, snap, None, 16)
    gdn.gdn_gated_rmsnorm_m(o, o.clone(), empty(128), o)
    torch.cuda.synchronize()
    assert gdn.gdn_wait_timeouts() == 0
