"""The CPU oracle against its pins (no GPU).

The pins live in oracle_pins.py; this file adds the checks that relate the
oracle's formulations to each other at the workloads' own sizes.
"""

import numpy as np
import pytest

import gdn_inputs
from oracle import ref64
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(oracle_mod, pin):
    pin(oracle_mod.run_f32)


def test_f32_matches_f64_matrix_decode(oracle_mod):
    """Single decode step, one sequence x 48 value heads, kd = vd = 128: the
    fp32 scalar oracle within 1e-6 normwise of the fp64 matrix form on every
    head (o and S)."""
    inp = gdn_inputs.make_workload("decode_b1")
    S32, o32 = oracle_mod.run_inputs(inp)
    S64, o64 = ref64.run_matrix(inp.S, inp.q, inp.k, inp.v, inp.g, inp.beta)
    assert ref64.max_rel(S32, S64, axes=(2, 3)) < 1e-6
    # o is a 128-term fp32 sum with cancellation (|o| is several times smaller
    # than sum |S q|).  Recursive summation of n terms errs by at most
    # ~n*u*sum|terms| (u = 2^-24); the inputs S_new carry a few ulps more.
    # Check every element against that bound with a factor 2 margin.
    u = 2.0 ** -24
    kd = inp.kd
    rep = inp.vh // inp.kh
    for vi in range(inp.vh):
        q = inp.q[0, 0, vi // rep].astype(np.float64)
        mag = np.abs(S64[0, vi]).T @ np.abs(q)           # sum_dk |S q|
        bound = 2 * (kd + 4) * u * mag
        assert np.all(np.abs(o32[0, 0, vi] - o64[0, 0, vi]) <= bound), vi
    # and the normwise figure stays at the fp32 level (a slip is O(1))
    assert ref64.max_rel(o32, o64, axes=(3,)) < 1e-5


def test_f32_matches_f64_matrix_chained(oracle_mod):
    """64 chained tokens on a subset of heads: fp32 oracle within 1e-5 of
    fp64 (the rounding of 64 fp32 steps)."""
    inp = gdn_inputs.make_workload("decode_b1_t64").heads([0], range(6))
    S32, o32 = oracle_mod.run_inputs(inp)
    S64, o64 = ref64.run_matrix(inp.S, inp.q, inp.k, inp.v, inp.g, inp.beta)
    assert ref64.max_rel(S32, S64, axes=(2, 3)) < 1e-5
    assert ref64.max_rel(o32, o64, axes=(0, 3)) < 1e-5


def test_matrix_form_matches_closed_form():
    """The fp64 step-by-step matrix form and the explicit product solution
    agree to fp64 rounding."""
    r = np.random.Generator(np.random.PCG64(5))
    kd, vd, T = 9, 5, 6
    S0 = r.standard_normal((kd, vd))
    k = r.standard_normal((T, kd))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = r.standard_normal((T, kd))
    v = r.standard_normal((T, vd))
    g = -np.abs(r.standard_normal(T))
    beta = r.uniform(0, 1, T)
    S = S0.copy()
    o = []
    for t in range(T):
        S, ot = ref64.step_matrix(S, q[t], k[t], v[t], g[t], beta[t])
        o.append(ot)
    ST, oT = ref64.closed_form(S0, q, k, v, g, beta)
    assert np.max(np.abs(S - ST)) < 1e-12
    assert np.max(np.abs(np.array(o) - oT)) < 1e-12


@pytest.mark.parametrize("T,chunk", [(10, 4), (64, 64), (150, 64), (7, 16)])
def test_chunked_form_matches_sequential(T, chunk):
    """The chunk-parallel form (including a ragged last chunk) equals the
    token-by-token recurrence in fp64."""
    r = np.random.Generator(np.random.PCG64(100 + T))
    kd, vd = 12, 10
    S0 = r.standard_normal((kd, vd)) * 0.1
    k = r.standard_normal((T, kd))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = r.standard_normal((T, kd))
    v = r.standard_normal((T, vd))
    g = -np.logaddexp(0, r.standard_normal(T))
    beta = 1 / (1 + np.exp(-r.standard_normal(T)))
    S = S0.copy()
    o = np.zeros((T, vd))
    for t in range(T):
        S, o[t] = ref64.step_matrix(S, q[t], k[t], v[t], g[t], beta[t])
    Sc, oc = ref64.chunked_head(S0, q, k, v, g, beta, chunk)
    assert ref64.max_rel(Sc, S) < 1e-11
    assert ref64.max_rel(oc, o) < 1e-11
    if T <= 10:
        ST, oT = ref64.closed_form(S0, q, k, v, g, beta)
        assert ref64.max_rel(Sc, ST) < 1e-11


def test_multi_token_equals_single_tokens(oracle_mod):
    """T tokens in one call are T single-token calls in sequence (bit-exact),
    and checkpoint t is the state after token t."""
    inp = gdn_inputs.make_inputs(7, B=2, T=5, kh=2, vh=4, kd=16, vd=8)
    S_all, o_all, ck = oracle_mod.run_inputs(inp, ckpt=True)
    S = inp.S
    for t in range(inp.T):
        st = inp.step(t)
        S, o = oracle_mod.run_f32(S, st.q, st.k, st.v, st.g, st.beta)
        assert np.array_equal(o[:, 0], o_all[:, t])
        assert np.array_equal(S, ck[t])
    assert np.array_equal(S, S_all)


def test_state_norm_bound(oracle_mod):
    """With alpha <= 1, beta in [0, 1] and |k| = 1 the transition
    alpha (I - beta k k^T) has spectral norm <= 1, so
    |S_t|_F <= |S_{t-1}|_F + beta_t |k_t| |v_t| at every token."""
    inp = gdn_inputs.make_inputs(8, B=1, T=300, kh=1, vh=2, kd=32, vd=16,
                                 s_std=1.0)
    _, _, ck = oracle_mod.run_inputs(inp, ckpt=True)
    prev = np.linalg.norm(inp.S.astype(np.float64), axis=(2, 3))
    for t in range(inp.T):
        cur = np.linalg.norm(ck[t].astype(np.float64), axis=(2, 3))
        inc = inp.beta[:, t].astype(np.float64) * np.linalg.norm(
            inp.v[:, t].astype(np.float64), axis=-1)
        assert np.all(cur <= prev + inc + 1e-4 * (1 + prev)), t
        prev = cur


def test_gqa_shared_key_head(oracle_mod):
    """Value heads in one key-head group with identical (S, v, g, beta) give
    identical results; a head of another group does not."""
    inp = gdn_inputs.make_inputs(9, B=1, T=3, kh=2, vh=6, kd=16, vd=8)
    S = inp.S.copy()
    v, g, beta = inp.v.copy(), inp.g.copy(), inp.beta.copy()
    for vi in (1, 2, 3):
        S[:, vi] = S[:, 0]
        v[:, :, vi] = v[:, :, 0]
        g[:, :, vi] = g[:, :, 0]
        beta[:, :, vi] = beta[:, :, 0]
    S1, o = oracle_mod.run_f32(S, inp.q, inp.k, v, g, beta)
    assert np.array_equal(o[:, :, 0], o[:, :, 1])
    assert np.array_equal(o[:, :, 0], o[:, :, 2])
    assert not np.array_equal(o[:, :, 0], o[:, :, 3])
    assert np.array_equal(S1[:, 0], S1[:, 2])


def test_input_recipe():
    """The generator's distributions: unit q/k rows, g < 0, beta in (0, 1),
    S std near 0.02; fixed seeds reproduce."""
    a = gdn_inputs.make_workload("decode_b1")
    b = gdn_inputs.make_workload("decode_b1")
    assert np.array_equal(a.S, b.S) and np.array_equal(a.v, b.v)
    assert np.allclose(np.linalg.norm(a.q, axis=-1), 1, atol=1e-6)
    assert np.allclose(np.linalg.norm(a.k, axis=-1), 1, atol=1e-6)
    assert np.all(a.g < 0) and np.all((a.beta > 0) & (a.beta < 1))
    assert abs(float(a.S.std()) - 0.02) < 1e-3
    assert a.S.shape == (1, 48, 128, 128) and a.q.shape == (1, 1, 16, 128)
