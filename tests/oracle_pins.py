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


# ------------------------------------------------------------ layer core
#
# The layer core around the recurrence ("24 · GDN linear attention to GPU",
# section 3 and figure 1 steps 2-5): depthwise causal conv1d + SiLU over the
# mixed q|k|v projection with a history of the last ck-1 inputs (oldest
# first), q/k scaled to unit L2 norm per key head, and the gates
# beta = sigmoid(b), g = -exp(A_log) * softplus(a + dt_bias).  Each pin
# below recomputes one of those steps in fp64 NumPy from its closed form and
# feeds the result to the already-pinned recurrence.


def _layer_case(seed, B=2, T=6, kh=2, vh=4, kd=8, vd=6, ck=4):
    r = _rng(seed)
    conv_dim = 2 * kh * kd + vh * vd
    S = (r.standard_normal((B, vh, kd, vd)) * 0.3).astype(np.float32)
    hist = r.standard_normal((B, ck - 1, conv_dim)).astype(np.float32)
    x = r.standard_normal((B, T, conv_dim)).astype(np.float32)
    w = (r.standard_normal((conv_dim, ck)) * 0.5).astype(np.float32)
    a = r.standard_normal((B, T, vh)).astype(np.float32)
    b = r.standard_normal((B, T, vh)).astype(np.float32)
    A_log = (r.standard_normal(vh) * 0.5).astype(np.float32)
    dt = (r.standard_normal(vh) * 0.5).astype(np.float32)
    return S, hist, x, w, a, b, A_log, dt, kh


def _layer_inputs64(hist, x, w, a, b, A_log, dt, kh, kd, vh, vd, eps=1e-6):
    """q, k, v, g, beta of every token from the closed forms (fp64)."""
    hist, x, w = (np.asarray(t, np.float64) for t in (hist, x, w))
    B, T, C = x.shape
    ck = w.shape[1]
    seq = np.concatenate([hist, x], axis=1)          # [B][ck-1+T][C]
    conv = np.zeros((B, T, C))
    for t in range(T):
        window = seq[:, t:t + ck]                    # oldest first
        conv[:, t] = np.einsum("bjc,cj->bc", window, w)
    act = conv / (1.0 + np.exp(-conv))               # SiLU
    q = act[:, :, :kh * kd].reshape(B, T, kh, kd)
    k = act[:, :, kh * kd:2 * kh * kd].reshape(B, T, kh, kd)
    v = act[:, :, 2 * kh * kd:].reshape(B, T, vh, vd)
    q = q / np.sqrt(np.sum(q * q, -1, keepdims=True) + eps)
    k = k / np.sqrt(np.sum(k * k, -1, keepdims=True) + eps)
    xa = np.asarray(a, np.float64) + np.asarray(dt, np.float64)
    g = -np.exp(np.asarray(A_log, np.float64)) * np.logaddexp(0.0, xa)
    beta = 1.0 / (1.0 + np.exp(-np.asarray(b, np.float64)))
    return q, k, v, g, beta, seq[:, -(ck - 1):] if ck > 1 else seq[:, :0]


def layer_pin_closed_forms(run_layer, run_f32):
    """Conv (general kernel, history carried across tokens), SiLU, norm and
    gates against their closed forms: the layer's o and S equal the pinned
    recurrence fed with fp64-derived q, k, v, g, beta (to fp32 rounding),
    and the final history is the last ck-1 inputs exactly."""
    S, hist, x, w, a, b, A_log, dt, kh = _layer_case(31)
    B, vh, kd, vd = S.shape
    S1, h1, o1 = run_layer(S, hist, x, w, a, b, A_log, dt, kh)
    q, k, v, g, beta, hist_ref = _layer_inputs64(hist, x, w, a, b, A_log, dt,
                                                 kh, kd, vh, vd)
    S2, o2 = run_f32(S, q, k, v, g, beta)
    assert ref64.max_rel(o1, o2, axes=(-2, -1)) < 2e-5
    assert ref64.max_rel(S1, S2, axes=(-2, -1)) < 2e-5
    assert np.array_equal(h1, hist_ref.astype(np.float32))


def layer_pin_identity_conv(run_layer, run_f32):
    """conv_w = (0, ..., 0, 1) makes the convolution the identity: q, k, v
    are SiLU of the raw input, unit-normalised for q and k."""
    S, hist, x, w, a, b, A_log, dt, kh = _layer_case(32)
    w[:] = 0
    w[:, -1] = 1
    B, vh, kd, vd = S.shape
    _, _, o1 = run_layer(S, hist, x, w, a, b, A_log, dt, kh)
    x64 = x.astype(np.float64)
    act = x64 / (1 + np.exp(-x64))
    q = act[:, :, :kh * kd].reshape(B, -1, kh, kd)
    k = act[:, :, kh * kd:2 * kh * kd].reshape(B, -1, kh, kd)
    v = act[:, :, 2 * kh * kd:].reshape(B, -1, vh, vd)
    q = q / np.linalg.norm(q, axis=-1, keepdims=True)
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    g = -np.exp(A_log.astype(np.float64)) * np.logaddexp(0, a.astype(np.float64) + dt)
    beta = 1 / (1 + np.exp(-b.astype(np.float64)))
    _, o2 = run_f32(S, q, k, v, g, beta)
    assert ref64.max_rel(o1, o2, axes=(-2, -1)) < 2e-5


def layer_pin_softplus_branches(run_layer, run_f32):
    """a + dt_bias beyond +-20 selects the linear and exponential branches:
    g = -exp(A_log) * xa and -exp(A_log) * exp(xa) respectively."""
    S, hist, x, w, a, b, A_log, dt, kh = _layer_case(33, T=2)
    a[:, 0] = 25.0 - dt      # xa = 25
    a[:, 1] = -25.0 - dt     # xa = -25
    A_log[:] = np.float32(np.log(0.01))   # keep g = -0.25 visible in alpha
    B, vh, kd, vd = S.shape
    S1, _, o1 = run_layer(S, hist, x, w, a, b, A_log, dt, kh)
    q, k, v, _, beta, _ = _layer_inputs64(hist, x, w, a, b, A_log, dt, kh,
                                          kd, vh, vd)
    g = np.empty((B, 2, vh))
    g[:, 0] = -np.exp(A_log.astype(np.float64)) * 25.0
    g[:, 1] = -np.exp(A_log.astype(np.float64)) * np.exp(-25.0)
    S2, o2 = run_f32(S, q, k, v, g, beta)
    assert ref64.max_rel(S1, S2, axes=(-2, -1)) < 2e-5
    assert ref64.max_rel(o1, o2, axes=(-2, -1)) < 2e-5


def layer_pin_gate_values(run_layer, run_f32):
    """a = -dt_bias, b = 0, A_log = 0: softplus(0) = ln 2 and sigmoid(0) =
    1/2, so g = -ln 2 (alpha = 1/2) and beta = 1/2 for every head."""
    S, hist, x, w, a, b, A_log, dt, kh = _layer_case(34, T=3)
    a[:] = -dt
    b[:] = 0
    A_log[:] = 0
    B, vh, kd, vd = S.shape
    S1, _, o1 = run_layer(S, hist, x, w, a, b, A_log, dt, kh)
    q, k, v, _, _, _ = _layer_inputs64(hist, x, w, a, b, A_log, dt, kh, kd,
                                       vh, vd)
    g = np.full((B, 3, vh), -np.log(2.0))
    beta = np.full((B, 3, vh), 0.5)
    S2, o2 = run_f32(S, q, k, v, g, beta)
    assert ref64.max_rel(S1, S2, axes=(-2, -1)) < 2e-5


LAYER_PINS = [layer_pin_closed_forms, layer_pin_identity_conv,
              layer_pin_softplus_branches, layer_pin_gate_values]


# ---------------------------------------------------------------------------
# Gated RMSNorm on the recurrence output (one value head's vd channels at a
# time).  Each pin takes run_gate_norm(o, z, w, eps) -> y.  The values are
# closed forms: a row of +-1 has RMS exactly 1, and at z = ln 3 the sigmoid
# is exactly 3/4, so the SiLU gate is 0.75 ln 3.

_SILU_LN3 = 0.75 * np.log(3.0)


def _pm_ones(B, T, vh, vd, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.where(rng.standard_normal((B, T, vh, vd)) < 0, -1.0, 1.0)


def gate_norm_pin_unit_row(run_gate_norm):
    """o = +-1 (RMS 1), z = ln 3, w = 1, eps = 0: y = +-0.75 ln 3."""
    o = _pm_ones(2, 3, 4, 128, 41)
    z = np.full_like(o, np.log(3.0))
    y = run_gate_norm(o, z, np.ones(128), eps=0.0)
    assert np.allclose(y, o * _SILU_LN3, rtol=2e-6, atol=0)


def gate_norm_pin_per_channel(run_gate_norm):
    """Per-channel weight and gate: w[c] = 2^(c mod 5 - 2) and z[c] cycling
    through ln 3, -ln 3, 0 (SiLU 0.75 ln 3, -0.25 ln 3, 0) on a +-1 row."""
    vd = 128
    o = _pm_ones(1, 2, 3, vd, 42)
    c = np.arange(vd)
    w = 2.0 ** (c % 5 - 2)
    zc = np.array([np.log(3.0), -np.log(3.0), 0.0])[c % 3]
    sc = np.array([_SILU_LN3, -0.25 * np.log(3.0), 0.0])[c % 3]
    y = run_gate_norm(o, np.broadcast_to(zc, o.shape), w, eps=0.0)
    assert np.allclose(y, o * w * sc, rtol=2e-6, atol=1e-30)


def gate_norm_pin_eps_placement(run_gate_norm):
    """A constant row o = 0.01 with eps = 1e-4: RMS sqrt(1e-4 + 1e-4), so
    o * r = 1/sqrt 2; an all-zero row gives y = 0."""
    o = np.full((1, 1, 2, 128), 0.01)
    o[0, 0, 1] = 0.0
    z = np.full_like(o, np.log(3.0))
    y = run_gate_norm(o, z, np.ones(128), eps=1e-4)
    assert np.allclose(y[0, 0, 0], _SILU_LN3 / np.sqrt(2.0), rtol=2e-6)
    assert np.all(y[0, 0, 1] == 0.0)


def gate_norm_pin_row_scaling(run_gate_norm):
    """eps = 0: scaling a whole (sequence, token, head) row by a power of two
    (a different one per row) or negating it changes y by nothing or by its
    sign, bit for bit; each row is normalised on its own."""
    rng = np.random.Generator(np.random.PCG64(43))
    o = rng.standard_normal((2, 2, 3, 128)).astype(np.float32)
    z = rng.standard_normal(o.shape).astype(np.float32)
    w = rng.uniform(0.5, 2.0, 128).astype(np.float32)
    y = run_gate_norm(o, z, w, eps=0.0)
    scale = np.float32(2.0) ** np.arange(-6, 6).reshape(2, 2, 3, 1)
    ys = run_gate_norm(o * scale, z, w, eps=0.0)
    yn = run_gate_norm(-o, z, w, eps=0.0)
    assert np.array_equal(ys, y)
    assert np.array_equal(yn, -y)


GATE_NORM_PINS = [gate_norm_pin_unit_row, gate_norm_pin_per_channel,
                  gate_norm_pin_eps_placement, gate_norm_pin_row_scaling]
