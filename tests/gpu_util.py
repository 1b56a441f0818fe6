"""Helpers for the GPU tests: move seeded inputs to the device and run the
library's entry points on them."""

import numpy as np
import torch

import gated_deltanet_linear_gb300 as gdn


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def empty(*shape):
    return torch.empty(*shape, device="cuda", dtype=torch.float32)


def run_step(inp, S=None):
    """One gdn_step on token 0 of inp; returns (S_after, o) on the device."""
    S = dev(inp.S) if S is None else S
    t = inp.step(0) if inp.T != 1 else inp
    o = empty(inp.B, 1, inp.vh, inp.vd)
    gdn.gdn_step(S, dev(t.q), dev(t.k), dev(t.v), dev(t.g), dev(t.beta), o)
    return S, o


def run_single_steps(inp):
    """inp.T successive gdn_step calls; returns (S_T, o [B][T][vh][vd],
    states [T][...] after each token) on the device."""
    S = dev(inp.S)
    o = empty(inp.B, inp.T, inp.vh, inp.vd)
    states = []
    q, k, v, g, beta = (dev(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    for t in range(inp.T):
        ot = empty(inp.B, 1, inp.vh, inp.vd)
        gdn.gdn_step(S, q[:, t].contiguous(), k[:, t].contiguous(),
                     v[:, t].contiguous(), g[:, t].contiguous(),
                     beta[:, t].contiguous(), ot)
        o[:, t] = ot[:, 0]
        states.append(S.clone())
    return S, o, states


def run_step_m(inp, ckpt=True, inplace=False):
    S_in = dev(inp.S)
    S_out = S_in if inplace else torch.empty_like(S_in)
    ck = empty(inp.T, *inp.S.shape) if ckpt else None
    o = empty(inp.B, inp.T, inp.vh, inp.vd)
    gdn.gdn_step_m(S_in, S_out, ck, dev(inp.q), dev(inp.k), dev(inp.v),
                   dev(inp.g), dev(inp.beta), o)
    return S_in, S_out, ck, o
