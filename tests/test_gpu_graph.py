"""The entry points inside CUDA graphs: a decode step, a layer step followed
by the gated RMSNorm (whose kernels are chained by programmatic dependent
launch, which capture turns into graph edges), and a chunked prefill are
captured once and replayed; every replay gives the same bits as the same
calls made eagerly on the same inputs."""

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


def _capture(fn):
    """Warm up on a side stream, then capture fn() into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_decode_step_graph():
    inp = gdn_inputs.make_inputs(1301, B=8, T=1)
    q, k, v, g_, b = (dev(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    S0 = dev(inp.S)
    S = S0.clone()
    o = empty(inp.B, 1, inp.vh, inp.vd)
    graph = _capture(lambda: gdn.gdn_step(S, q, k, v, g_, b, o))
    # eager reference: two steps from S0
    S_ref = S0.clone()
    o_ref = torch.empty_like(o)
    for _ in range(2):
        gdn.gdn_step(S_ref, q, k, v, g_, b, o_ref)
    S.copy_(S0)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(S, S_ref) and torch.equal(o, o_ref)


def test_layer_step_and_norm_graph():
    B, M = 6, 2
    L = gdn_inputs.make_layer_inputs(1302, B=B, T=M)
    _, z, w = gdn_inputs.make_gate_norm_inputs(1303, B, M, 48)
    x, conv_w, a, b = dev(L.x), dev(L.conv_w), dev(L.a), dev(L.b)
    A_log, dt, zd, wd = dev(L.A_log), dev(L.dt_bias), dev(z), dev(w)
    S = dev(L.S)
    h = [dev(L.hist), torch.empty_like(dev(L.hist))]
    y = empty(B, M, 48, 128)
    ws = torch.empty(gdn.gdn_layer_workspace(B, L.kh, 48, M),
                     dtype=torch.uint8, device="cuda")

    def two_steps(S, h, y):
        # two layer steps passing the history forward, each normed in place
        for i in range(2):
            gdn.gdn_layer_step_m(S, S, None, h[i % 2], h[(i + 1) % 2], x,
                                 conv_w, a, b, A_log, dt, y, L.kh, ws)
            gdn.gdn_gated_rmsnorm_m(y, zd, wd, y)

    S_e, h_e, y_e = S.clone(), [t.clone() for t in h], torch.empty_like(y)
    two_steps(S_e, h_e, y_e)
    torch.cuda.synchronize()

    S_g, h_g, y_g = S.clone(), [t.clone() for t in h], torch.empty_like(y)
    graph = _capture(lambda: two_steps(S_g, h_g, y_g))
    S_g.copy_(S)
    h_g[0].copy_(h[0])
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(S_g, S_e) and torch.equal(y_g, y_e)
    assert torch.equal(h_g[0], h_e[0])


def test_chunked_prefill_graph():
    inp = gdn_inputs.make_inputs(1304, B=2, T=130)
    q, k, v, g_, b = (dev(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    S0 = dev(inp.S)
    S_e = S0.clone()
    o_e = empty(inp.B, inp.T, inp.vh, inp.vd)
    gdn.gdn_prefill(S_e, q, k, v, g_, b, o_e, precision=gdn.GDN_PREC_BF16X3)
    S_g = S0.clone()
    o_g = torch.empty_like(o_e)
    graph = _capture(lambda: gdn.gdn_prefill(S_g, q, k, v, g_, b, o_g,
                                              precision=gdn.GDN_PREC_BF16X3))
    S_g.copy_(S0)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(S_g, S_e) and torch.equal(o_g, o_e)
    assert gdn.gdn_prefill_timeouts() == 0
