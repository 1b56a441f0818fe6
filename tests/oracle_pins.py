"""Checks that pin the CPU oracle to facts other than its own code.

Each pin takes a runner with the signature of ``oracle.run_f32`` and raises
AssertionError when the runner disagrees with what the definition and the
mathematics fix.  The same pins run against the real oracle
(test_oracle.py) and against deliberately broken copies of it
(test_oracle_mutants.py), which shows each plausible mistake is caught.

The definition pinned is the single token step of "Kestrel_VLLM - 24 · GDN
linear attention to GPU", section 4 / figure 1 step 5:
    alpha = exp(g); S *= alpha; kv = S^T k; tmp = (v - kv) beta;
    S += k tmp^T; o = S^T q (updated S); key head hh = vi / (vh / kh).
"""

from __future__ import annotations

import json
import os

import numpy as np

from oracle import ref64

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _rand_case(seed, B=1, T=1, kh=2, vh=6, kd=16, vd=12, s_std=0.3):
    r = _rng(seed)
    S = (r.standard_normal((B, vh, kd, vd)) * s_std).astype(np.float32)
    q = _unit(r.standard_normal((B, T, kh, kd))).astype(np.float32)
    k = _unit(r.standard_normal((B, T, kh, kd))).astype(np.float32)
    v = r.standard_normal((B, T, vh, vd)).astype(np.float32)
    g = (-np.logaddexp(0, r.standard_normal((B, T, vh)))).astype(np.float32)
    beta = (1 / (1 + np.exp(-r.standard_normal((B, T, vh))))).astype(np.float32)
    return S, q, k, v, g, beta


def pin_golden_tiny(run):
    """Hand-worked dyadic two-token example: exact in fp32."""
    with open(os.path.join(GOLDEN, "tiny_two_tokens.json")) as f:
        d = json.load(f)
    S0 = np.array(d["S0"], np.float32).reshape(1, 1, 2, 2)
    q = np.array(d["q"], np.float32).reshape(1, 2, 1, 2)
    k = np.array(d["k"], np.float32).reshape(1, 2, 1, 2)
    v = np.array(d["v"], np.float32).reshape(1, 2, 1, 2)
    g = np.array(d["g"], np.float32).reshape(1, 2, 1)
    beta = np.array(d["beta"], np.float32).reshape(1, 2, 1)
    S, o, ck = run(S0, q, k, v, g, beta, ckpt=True)
    assert np.array_equal(o.reshape(2, 2), np.array(d["o"], np.float32)), o
    exp_ck = np.array(d["S_after"], np.float32)
    assert np.array_equal(ck.reshape(2, 2, 2), exp_ck), ck
    assert np.array_equal(S.reshape(2, 2), exp_ck[-1])


def pin_identity(run):
    """alpha = 1 (g = 0) and beta = 0 leave S bit-exactly unchanged and give
    o = S^T q."""
    S, q, k, v, g, beta = _rand_case(11, B=2, T=3)
    g[:] = 0
    beta[:] = 0
    S1, o = run(S, q, k, v, g, beta)
    assert np.array_equal(S1, S), "state changed under alpha=1, beta=0"
    rep = S.shape[1] // q.shape[2]
    for b in range(S.shape[0]):
        for t in range(q.shape[1]):
            for vi in range(S.shape[1]):
                ref = S[b, vi].astype(np.float64).T @ q[b, t, vi // rep].astype(np.float64)
                assert ref64.max_rel(o[b, t, vi], ref) < 1e-6


def pin_beta1_readback(run):
    """beta = 1 and |k| = 1: after the update S^T k = v (to fp32 rounding plus
    the |k|^2 - 1 residue of the fp32 unit vector)."""
    S, q, k, v, g, beta = _rand_case(12, B=2, T=1)
    beta[:] = 1
    S1, _ = run(S, q, k, v, g, beta)
    rep = S.shape[1] // q.shape[2]
    for b in range(S.shape[0]):
        for vi in range(S.shape[1]):
            kk = k[b, 0, vi // rep].astype(np.float64)
            readback = S1[b, vi].astype(np.float64).T @ kk
            resid = abs(kk @ kk - 1.0)
            err = np.max(np.abs(readback - v[b, 0, vi]))
            assert err < 1e-5 + resid * np.max(np.abs(v[b, 0, vi])) * 2, err


def pin_zero_state(run):
    """S0 = 0, one token: S = beta k v^T and o = beta (q.k) v, with value head
    vi reading key head vi // rep (contiguous groups)."""
    S, q, k, v, g, beta = _rand_case(13, B=2, T=1, kh=2, vh=6)
    S[:] = 0
    S1, o = run(S, q, k, v, g, beta)
    rep = S.shape[1] // q.shape[2]
    for b in range(S.shape[0]):
        for vi in range(S.shape[1]):
            kk = k[b, 0, vi // rep].astype(np.float64)
            qq = q[b, 0, vi // rep].astype(np.float64)
            vv = v[b, 0, vi].astype(np.float64)
            bt = np.float64(beta[b, 0, vi])
            assert ref64.max_rel(S1[b, vi], bt * np.outer(kk, vv)) < 1e-6
            assert ref64.max_rel(o[b, 0, vi], bt * (qq @ kk) * vv) < 1e-6


def pin_alpha0(run):
    """g -> -inf (alpha = 0) forgets S0: S = beta k v^T for any S0."""
    S, q, k, v, g, beta = _rand_case(14, B=1, T=1)
    g[:] = -1.0e4
    S1, _ = run(S, q, k, v, g, beta)
    rep = S.shape[1] // q.shape[2]
    for vi in range(S.shape[1]):
        kk = k[0, 0, vi // rep].astype(np.float64)
        ref = np.float64(beta[0, 0, vi]) * np.outer(kk, v[0, 0, vi].astype(np.float64))
        assert ref64.max_rel(S1[0, vi], ref) < 1e-6


def pin_closed_form(run):
    """T = 1, 2, 3 against the explicit transition-matrix solution (fp64)."""
    for T in (1, 2, 3):
        S, q, k, v, g, beta = _rand_case(20 + T, B=1, T=T, kh=2, vh=4,
                                         kd=10, vd=7)
        S1, o = run(S, q, k, v, g, beta)
        rep = S.shape[1] // q.shape[2]
        for vi in range(S.shape[1]):
            hh = vi // rep
            ST, oT = ref64.closed_form(S[0, vi], q[0, :, hh], k[0, :, hh],
                                       v[0, :, vi], g[0, :, vi], beta[0, :, vi])
            assert ref64.max_rel(S1[0, vi], ST) < 2e-6, (T, vi)
            assert ref64.max_rel(o[0, :, vi], oT) < 2e-6, (T, vi)


def pin_alpha_value(run):
    """A non-trivial decay: g = ln(1/2) halves the state before the read-out
    (beta = 0 isolates it): S_1 = S0 / 2 and o = S_1^T q."""
    S, q, k, v, g, beta = _rand_case(15, B=1, T=1)
    g[:] = np.float32(np.log(0.5))
    beta[:] = 0
    S1, o = run(S, q, k, v, g, beta)
    assert ref64.max_rel(S1, S.astype(np.float64) * 0.5) < 1e-6
    rep = S.shape[1] // q.shape[2]
    for vi in range(S.shape[1]):
        ref = 0.5 * S[0, vi].astype(np.float64).T @ q[0, 0, vi // rep]
        assert ref64.max_rel(o[0, 0, vi], ref) < 1e-6


ALL_PINS = [pin_golden_tiny, pin_identity, pin_beta1_readback, pin_zero_state,
            pin_alpha0, pin_closed_form, pin_alpha_value]
