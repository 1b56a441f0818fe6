"""No launch writes outside its outputs.

Every output (and every in-place buffer) sits inside a larger allocation
whose guard bands, 16 KB on each side, hold a NaN bit pattern that no kernel
produces.  After the call the bands must hold the same bits, and the output
itself must hold no NaN (the inputs are finite).  One case per launch
route of the library:
- one token with device inputs (the 32-column kernel, four groups per CTA)
  and with page-locked host inputs and output (two groups per CTA);
- several tokens with at least one head per SM (head-per-CTA kernel), with
  fewer heads (8-column kernel), with host inputs, and with checkpoints;
- the prefill in its three precisions, on a ragged last chunk;
- mark, rollback, the layer step (including its caller workspace) and the
  gated RMSNorm.
"""

import numpy as np
import pytest
import torch

import gated_deltanet_linear_gb300 as gdn
import gdn_inputs
from gpu_util import dev, empty

pytestmark = pytest.mark.gpu

G = 4096            # guard elements (4 bytes each) on each side
PATTERN = 0x7FC0DEAD  # a quiet NaN with a payload


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


class Guarded:
    """A float32 tensor of `shape` inside a buffer with guard bands.  The
    tensor is initialised from `init` or left as the NaN pattern; `pinned`
    puts the buffer in page-locked host memory."""

    def __init__(self, shape, init=None, pinned=False):
        self.n = int(np.prod(shape))
        if pinned:
            self.base = torch.full((self.n + 2 * G,), PATTERN,
                                   dtype=torch.int32).pin_memory()
        else:
            self.base = torch.full((self.n + 2 * G,), PATTERN,
                                   dtype=torch.int32, device="cuda")
        self.t = self.base[G:G + self.n].view(torch.float32).view(*shape)
        if init is not None:
            self.t.copy_(torch.from_numpy(np.ascontiguousarray(init, np.float32)))

    def check(self, written=True):
        torch.cuda.synchronize()
        b = self.base.cpu()
        assert (b[:G] == PATTERN).all(), "write below the buffer"
        assert (b[G + self.n:] == PATTERN).all(), "write past the buffer"
        if written:
            assert not torch.isnan(b[G:G + self.n].view(torch.float32)).any()


def _tokens(inp, pinned=False):
    if pinned:
        return [torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
                for x in (inp.q, inp.k, inp.v, inp.g, inp.beta)]
    return [dev(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta)]


@pytest.mark.parametrize("pinned", [False, True])
def test_single_token(pinned):
    inp = gdn_inputs.make_inputs(5101, B=3, T=1)
    S = Guarded(inp.S.shape, inp.S)
    o = Guarded((inp.B, 1, inp.vh, 128), pinned=pinned)
    gdn.gdn_step(S.t, *_tokens(inp, pinned), o.t)
    S.check()
    o.check()


# (B, M, pinned inputs and output, checkpoints): 4 x 48 heads reach the
# head-per-CTA kernel, one sequence of 48 heads and the other cases the
# 8-column kernel
MULTI = [(4, 3, False, False), (1, 3, False, False), (2, 3, True, False),
         (2, 3, False, True)]


@pytest.mark.parametrize("B,M,pinned,ckpt", MULTI)
def test_multi_token(B, M, pinned, ckpt):
    inp = gdn_inputs.make_inputs(5102 + B, B=B, T=M)
    S_in = dev(inp.S)
    S_out = Guarded(inp.S.shape)
    o = Guarded((B, M, inp.vh, 128), pinned=pinned)
    ck = Guarded((M,) + inp.S.shape) if ckpt else None
    gdn.gdn_step_m(S_in, S_out.t, ck.t if ck else None, *_tokens(inp, pinned),
                   o.t)
    S_out.check()
    o.check()
    if ck:
        ck.check()
    # in place
    S = Guarded(inp.S.shape, inp.S)
    gdn.gdn_step_m(S.t, S.t, None, *_tokens(inp, pinned), o.t)
    S.check()
    o.check()


@pytest.mark.parametrize("precision", [gdn.GDN_PREC_FP32, gdn.GDN_PREC_BF16X3,
                                       gdn.GDN_PREC_BF16])
@pytest.mark.parametrize("T", [100, 64])
def test_prefill(precision, T):
    inp = gdn_inputs.make_inputs(5110 + T, B=2, T=T)
    S = Guarded(inp.S.shape, inp.S)
    o = Guarded((inp.B, T, inp.vh, 128))
    gdn.gdn_prefill(S.t, *_tokens(inp), o.t, precision=precision)
    S.check()
    o.check()
    assert gdn.gdn_prefill_timeouts() == 0


def test_mark_and_rollback():
    inp = gdn_inputs.make_inputs(5120, B=2, T=3)
    S_in = dev(inp.S)
    snap = Guarded(inp.S.shape)
    gdn.gdn_mark(S_in, snap.t, inp.kh)
    snap.check()
    ck = dev(np.stack([inp.S * (m + 2) for m in range(3)]))
    for m in (0, 2, 3):
        S = Guarded(inp.S.shape)
        gdn.gdn_rollback(S.t, 3, m, snap.t, ck, inp.kh)
        S.check()
        snap.check()


def test_layer_step_and_norm():
    L = gdn_inputs.make_layer_inputs(5130, B=3, T=2)
    B, M = L.x.shape[:2]
    vh = L.S.shape[1]
    S_out = Guarded(L.S.shape)
    hist_out = Guarded(L.hist.shape)
    o = Guarded((B, M, vh, 128))
    ck = Guarded((M,) + L.S.shape)
    ws_bytes = gdn.gdn_layer_workspace(B, L.kh, vh, M)
    assert ws_bytes % 16 == 0
    ws = Guarded((ws_bytes // 4,))
    ws_u8 = ws.t.view(torch.uint8)
    gdn.gdn_layer_step_m(dev(L.S), S_out.t, ck.t, dev(L.hist), hist_out.t,
                         dev(L.x), dev(L.conv_w), dev(L.a), dev(L.b),
                         dev(L.A_log), dev(L.dt_bias), o.t, L.kh, ws_u8)
    for buf in (S_out, hist_out, o, ck):
        buf.check()
    ws.check(written=False)
    z = dev(np.random.default_rng(5131).standard_normal((B, M, vh, 128),
                                                        dtype=np.float32))
    y = Guarded((B, M, vh, 128))
    gdn.gdn_gated_rmsnorm_m(o.t, z, dev(np.ones(128, np.float32)), y.t)
    y.check()
    o.check()
