"""Token inputs and outputs in page-locked host memory: the update kernel
reads q, k, v, g, beta and writes o over the host link, with the same bits
as device buffers; pageable host memory is refused before any launch."""

import ctypes

import numpy as np
import pytest
import torch

import gated_deltanet_linear_gb300 as gdn
import gdn_inputs
from gpu_util import dev, empty

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


CASES = [(hi, ho, ck) for hi in (True, False) for ho in (True, False)
         for ck in (False, True) if hi or ho or ck]


@pytest.mark.parametrize("host_in,host_out,ckpt", CASES)
@pytest.mark.parametrize("M", [1, 3])
def test_host_token_buffers_same_bits(host_in, host_out, ckpt, M):
    """Every combination of token buffers in host or device memory, one or
    three tokens, with or without checkpoints, against the device-memory
    launch without checkpoints: the same bits (the launches run different
    kernels: the 32-column single-token kernel with one or two column groups
    per CTA, the head-per-CTA kernel, the 8-column kernel)."""
    inp = gdn_inputs.make_inputs(1401 + M, B=5, T=M)
    xs = (inp.q, inp.k, inp.v, inp.g, inp.beta)
    d_in = [dev(x) for x in xs]
    ins = [_pinned(x) for x in xs] if host_in else d_in
    S_ref = dev(inp.S)
    o_ref = empty(inp.B, M, inp.vh, inp.vd)
    gdn.gdn_step_m(S_ref, S_ref, None, *d_in, o_ref)
    S = dev(inp.S)
    o = (torch.empty(inp.B, M, inp.vh, inp.vd).pin_memory() if host_out
         else empty(inp.B, M, inp.vh, inp.vd))
    ck = empty(M, *inp.S.shape) if ckpt else None
    if M == 1 and not ckpt:
        gdn.gdn_step(S, *ins, o)
    else:
        gdn.gdn_step_m(S, S, ck, *ins, o)
    torch.cuda.synchronize()
    assert torch.equal(S, S_ref)
    assert torch.equal(o.cpu(), o_ref.cpu())
    if ckpt:
        assert torch.equal(ck[M - 1], S_ref)


def test_pageable_host_memory_refused():
    lib = gdn.load()
    inp = gdn_inputs.make_inputs(1405, B=2, T=1)
    S = dev(inp.S)
    q, k, v, g, b = (dev(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    o_pageable = np.zeros((2, 1, 48, 128), np.float32)
    sh = gdn.Shape(2, 16, 48, 128, 128)
    P = lambda t: t.data_ptr()
    rc = lib.gdn_step(ctypes.byref(sh), P(S), P(q), P(k), P(v), P(g), P(b),
                      o_pageable.ctypes.data,
                      torch.cuda.current_stream().cuda_stream)
    assert rc in (gdn.GDN_EPTR, gdn.GDN_EALIGN)
    with pytest.raises(ValueError):
        gdn.gdn_step(S, q, k, v, g, b, torch.zeros(2, 1, 48, 128))
