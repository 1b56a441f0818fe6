"""Back-to-back launches that start behind the launch before them.

A single-token launch that fills the GPU, a verify launch without
checkpoints of at most 16 tokens, and the layer step's prologue start as
programmatic dependents of the kernel before them: their CTAs may be
resident before that kernel has ended, and they read (and write) nothing
until it has.  The decode loop is the case that tests this: each step reads
the state the step just before it wrote, with no other kernel in between.
Here every per-token buffer is prepared before the loop, the launches go
out back to back, and the results must equal one multi-token launch over
the same tokens bit for bit (the kernels share their arithmetic, so any
read of a state that was not yet final would show).

64 sequences x 48 heads (the grids fill every CTA slot of a GB300).
"""

import pytest
import torch

import gated_deltanet_linear_gb300 as gdn
import gdn_inputs
from gpu_util import dev, empty

pytestmark = pytest.mark.gpu

B, KH, VH, D = 64, 16, 48, 128


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _tokens(inp):
    return [dev(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta)]


def test_decode_steps_back_to_back():
    T = 12
    inp = gdn_inputs.make_inputs(8100, B=B, T=T)
    q, k, v, g, beta = _tokens(inp)
    per_tok = [tuple(x[:, t:t + 1].contiguous() for x in (q, k, v, g, beta))
               for t in range(T)]
    outs = [empty(B, 1, VH, D) for _ in range(T)]
    S = dev(inp.S)
    torch.cuda.synchronize()
    for t in range(T):
        gdn.gdn_step(S, *per_tok[t], outs[t])
    S_m = dev(inp.S)
    o_m = empty(B, T, VH, D)
    ck = empty(T, B, VH, D, D)
    gdn.gdn_step_m(S_m, S_m, ck, q, k, v, g, beta, o_m)
    torch.cuda.synchronize()
    assert torch.equal(S, S_m)
    for t in range(T):
        assert torch.equal(outs[t][:, 0], o_m[:, t]), t


@pytest.mark.parametrize("M", [2, 4])
def test_verify_launches_back_to_back(M):
    n = 4
    inp = gdn_inputs.make_inputs(8200 + M, B=B, T=n * M)
    q, k, v, g, beta = _tokens(inp)
    chunks = [tuple(x[:, i * M:(i + 1) * M].contiguous()
                    for x in (q, k, v, g, beta)) for i in range(n)]
    outs = [empty(B, M, VH, D) for _ in range(n)]
    S = dev(inp.S)
    torch.cuda.synchronize()
    for i in range(n):
        gdn.gdn_step_m(S, S, None, *chunks[i], outs[i])
    S_m = dev(inp.S)
    o_m = empty(B, n * M, VH, D)
    gdn.gdn_step_m(S_m, S_m, None, q, k, v, g, beta, o_m)
    torch.cuda.synchronize()
    assert torch.equal(S, S_m)
    for i in range(n):
        assert torch.equal(outs[i], o_m[:, i * M:(i + 1) * M]), i
    assert gdn.gdn_wait_timeouts() == 0


def test_layer_steps_back_to_back():
    T = 6
    L = gdn_inputs.make_layer_inputs(8300, B=B, T=T)
    x, a, b = dev(L.x), dev(L.a), dev(L.b)
    w = [dev(t) for t in (L.conv_w, L.A_log, L.dt_bias)]
    per_tok = [tuple(t_[:, m:m + 1].contiguous() for t_ in (x, a, b))
               for m in range(T)]
    ws = torch.empty(gdn.gdn_layer_workspace(B, L.kh, VH, T), dtype=torch.uint8,
                     device="cuda")
    # two state and two history buffers in turn, as a decode loop would
    S = [dev(L.S), torch.empty_like(dev(L.S))]
    hist = [dev(L.hist), torch.empty_like(dev(L.hist))]
    outs = [empty(B, 1, VH, D) for _ in range(T)]
    torch.cuda.synchronize()
    for m in range(T):
        i, j = m % 2, (m + 1) % 2
        gdn.gdn_layer_step_m(S[i], S[j], None, hist[i], hist[j], *per_tok[m][:1],
                             w[0], per_tok[m][1], per_tok[m][2], w[1], w[2],
                             outs[m], L.kh, ws)
    S_m, hist_m = torch.empty_like(S[0]), torch.empty_like(hist[0])
    o_m = empty(B, T, VH, D)
    gdn.gdn_layer_step_m(dev(L.S), S_m, None, dev(L.hist), hist_m, x, w[0], a, b,
                         w[1], w[2], o_m, L.kh, ws)
    torch.cuda.synchronize()
    assert torch.equal(S[T % 2], S_m) and torch.equal(hist[T % 2], hist_m)
    for m in range(T):
        assert torch.equal(outs[m][:, 0], o_m[:, m]), m


def test_two_streams_back_to_back():
    """Two batches decoded on two streams at once, each a run of
    back-to-back steps: every step on a stream starts behind the one
    before it on the same stream while the other stream's kernels run
    beside it.  Results equal the same steps run on one stream."""
    T = 6
    inps = [gdn_inputs.make_inputs(8400 + i, B=B, T=T) for i in range(2)]
    per_tok, states, outs = [], [], []
    for inp in inps:
        q, k, v, g, beta = _tokens(inp)
        per_tok.append([tuple(x[:, t:t + 1].contiguous()
                              for x in (q, k, v, g, beta)) for t in range(T)])
        states.append(dev(inp.S))
        outs.append([empty(B, 1, VH, D) for _ in range(T)])
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for t in range(T):
        for i in range(2):
            gdn.gdn_step(states[i], *per_tok[i][t], outs[i][t],
                         stream=streams[i])
    torch.cuda.synchronize()
    for i, inp in enumerate(inps):
        S = dev(inp.S)
        for t in range(T):
            o = empty(B, 1, VH, D)
            gdn.gdn_step(S, *per_tok[i][t], o)
            assert torch.equal(o, outs[i][t]), (i, t)
        torch.cuda.synchronize()
        assert torch.equal(S, states[i]), i


def test_decode_steps_back_to_back_in_a_graph():
    """Eight back-to-back full-grid steps captured in one CUDA graph (the
    programmatic dependencies between them become graph edges) and
    replayed: the same bits as the steps made eagerly."""
    T = 8
    inp = gdn_inputs.make_inputs(8500, B=B, T=T)
    q, k, v, g, beta = _tokens(inp)
    per_tok = [tuple(x[:, t:t + 1].contiguous() for x in (q, k, v, g, beta))
               for t in range(T)]
    outs = [empty(B, 1, VH, D) for _ in range(T)]
    S0 = dev(inp.S)
    S = S0.clone()

    def steps():
        for t in range(T):
            gdn.gdn_step(S, *per_tok[t], outs[t])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        steps()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        steps()
    S.copy_(S0)
    graph.replay()
    torch.cuda.synchronize()
    S_ref = S0.clone()
    for t in range(T):
        o = empty(B, 1, VH, D)
        gdn.gdn_step(S_ref, *per_tok[t], o)
        assert torch.equal(o, outs[t]), t
    assert torch.equal(S, S_ref)


def test_host_input_launches_back_to_back():
    """Two-token launches whose token inputs and outputs are page-locked
    host memory (the 8-column kernel, a full grid at 64 sequences, started
    behind the launch before it), back to back in place: the same bits as
    one launch over all tokens with device-resident inputs."""
    M, n = 2, 3
    inp = gdn_inputs.make_inputs(8600, B=B, T=n * M)
    host = [torch.from_numpy(x.copy()) for x in
            (inp.q, inp.k, inp.v, inp.g, inp.beta)]
    chunks = [tuple(x[:, i * M:(i + 1) * M].contiguous().pin_memory()
                    for x in host) for i in range(n)]
    outs = [torch.empty(B, M, VH, D).pin_memory() for _ in range(n)]
    S = dev(inp.S)
    torch.cuda.synchronize()
    for i in range(n):
        gdn.gdn_step_m(S, S, None, *chunks[i], outs[i])
    S_m = dev(inp.S)
    o_m = empty(B, n * M, VH, D)
    gdn.gdn_step_m(S_m, S_m, None, *_tokens(inp), o_m)
    torch.cuda.synchronize()
    assert torch.equal(S, S_m)
    for i in range(n):
        assert torch.equal(outs[i], o_m[:, i * M:(i + 1) * M].cpu()), i
