"""Double-precision formulations of the gated delta-rule update (test
infrastructure only: nothing in the product imports this module).

Three independent restatements, used to pin the fp32 scalar oracle and to
check the chunked derivation the tensor-core prefill implements:

1. ``step_matrix``: one token in matrix form.  Expanding the per-element
   definition ("Kestrel_VLLM - 24 · GDN linear attention to GPU", section 4,
   the delta-recurrence kernel; figure 1 step 5):
       S' = alpha*S;  kv = S'^T k;  tmp = beta*(v - kv);  S'' = S' + k tmp^T
   gives  S'' = alpha (I - beta k k^T) S + beta k v^T  and  o = S''^T q.

2. ``closed_form``: the solution of that linear recurrence after T tokens as
   explicit products of the per-token transition matrices,
       S_T = P(T,1) S_0 + sum_s P(T,s+1) beta_s k_s v_s^T,
       P(t,s) = A_t A_{t-1} ... A_s,  A_t = alpha_t (I - beta_t k_t k_t^T),
   with o_t = S_t^T q_t.  Written without any per-token state update.

3. ``chunked``: the chunk-parallel form of the same recurrence (derived
   here; the articles process tokens strictly one after another, "34 ·
   batched M rows", section 3.6).  With Gamma_t = sum_{s<=t} g_s inside a
   chunk, gamma_t = exp(Gamma_t), and S0 the state entering the chunk:
       A[t,s]  = beta_t exp(Gamma_t - Gamma_s) (k_t . k_s),   s < t
       (I + A) Delta = diag(beta) (V - diag(gamma) K S0)
       O   = diag(gamma) Q S0 + (L o (Q K^T)) Delta,
             L[t,s] = exp(Gamma_t - Gamma_s) for s <= t, else 0
       S_C = gamma_{C-1} S0 + K^T diag(exp(Gamma_{C-1} - Gamma_s)) Delta
   It follows from delta_t = beta_t (v_t - alpha_t S_{t-1}^T k_t) and
   S_t = gamma_t S0 + sum_{s<=t} (gamma_t / gamma_s) k_s delta_s^T.

Shapes follow the library layouts: S [B][vh][kd][vd], q/k [B][T][kh][kd],
v [B][T][vh][vd], g/beta [B][T][vh].  Value head vi reads key head
vi // (vh // kh).
"""

from __future__ import annotations

import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def step_matrix(S, q, k, v, g, beta):
    """One token for one head in fp64.  S [kd][vd]; q, k [kd]; v [vd]."""
    S, q, k, v = _f64(S), _f64(q), _f64(k), _f64(v)
    alpha = np.exp(np.float64(g))
    beta = np.float64(beta)
    kd = S.shape[0]
    A = alpha * (np.eye(kd) - beta * np.outer(k, k))
    S_new = A @ S + beta * np.outer(k, v)
    return S_new, S_new.T @ q


def run_matrix(S, q, k, v, g, beta, ckpt: bool = False):
    """All heads, T tokens, fp64 matrix form.  Returns (S_T, o[, ckpt])."""
    S = _f64(S).copy()
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    B, vh = S.shape[:2]
    T, kh = q.shape[1], q.shape[2]
    rep = vh // kh
    o = np.zeros(v.shape, dtype=np.float64)
    ck = np.zeros((T,) + S.shape, dtype=np.float64) if ckpt else None
    for b in range(B):
        for vi in range(vh):
            hh = vi // rep
            for t in range(T):
                S[b, vi], o[b, t, vi] = step_matrix(
                    S[b, vi], q[b, t, hh], k[b, t, hh], v[b, t, vi],
                    g[b, t, vi], beta[b, t, vi])
                if ckpt:
                    ck[t, b, vi] = S[b, vi]
    return (S, o, ck) if ckpt else (S, o)


def closed_form(S0, q, k, v, g, beta):
    """One head over T tokens via explicit transition-matrix products.

    S0 [kd][vd]; q, k [T][kd]; v [T][vd]; g, beta [T].
    Returns (S_T, o [T][vd]).
    """
    S0, q, k, v, g, beta = map(_f64, (S0, q, k, v, g, beta))
    T, kd = k.shape
    A = [np.exp(g[t]) * (np.eye(kd) - beta[t] * np.outer(k[t], k[t]))
         for t in range(T)]

    def P(t_hi, t_lo):  # A_{t_hi} ... A_{t_lo}, identity when empty
        M = np.eye(kd)
        for t in range(t_lo, t_hi + 1):
            M = A[t] @ M
        return M

    o = np.zeros((T, S0.shape[1]))
    S_t = None
    for t in range(T):
        S_t = P(t, 0) @ S0
        for s in range(t + 1):
            S_t = S_t + P(t, s + 1) @ (beta[s] * np.outer(k[s], v[s]))
        o[t] = S_t.T @ q[t]
    return (S_t if T else S0.copy()), o


def chunked_head(S0, q, k, v, g, beta, chunk: int = 64):
    """One head over T tokens via the chunk-parallel form (fp64).

    S0 [kd][vd]; q, k [T][kd]; v [T][vd]; g, beta [T].
    Returns (S_T, o [T][vd]).  The last chunk may be shorter.
    """
    S = _f64(S0).copy()
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    T = k.shape[0]
    o = np.zeros((T, S.shape[1]))
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        K, Q, V = k[c0:c1], q[c0:c1], v[c0:c1]
        G = np.cumsum(g[c0:c1])
        bt = beta[c0:c1]
        n = c1 - c0
        D = G[:, None] - G[None, :]                 # Gamma_t - Gamma_s
        tri_strict = np.tril(np.ones((n, n)), -1)
        tri = np.tril(np.ones((n, n)))
        decay = np.exp(np.where(tri > 0, D, -np.inf))  # L[t, s]
        A = bt[:, None] * decay * tri_strict * (K @ K.T)
        gam = np.exp(G)
        rhs = bt[:, None] * (V - gam[:, None] * (K @ S))
        Delta = np.linalg.solve(np.eye(n) + A, rhs)
        o[c0:c1] = gam[:, None] * (Q @ S) + (decay * (Q @ K.T)) @ Delta
        w = np.exp(G[-1] - G)
        S = gam[-1] * S + K.T @ (w[:, None] * Delta)
    return S, o


def run_chunked(S, q, k, v, g, beta, chunk: int = 64):
    """All heads via ``chunked_head``.  Returns (S_T, o)."""
    S = _f64(S).copy()
    B, vh = S.shape[:2]
    kh = q.shape[2]
    rep = vh // kh
    o = np.zeros(v.shape, dtype=np.float64)
    for b in range(B):
        for vi in range(vh):
            hh = vi // rep
            S[b, vi], o[b, :, vi] = chunked_head(
                S[b, vi], q[b, :, hh], k[b, :, hh], v[b, :, vi],
                g[b, :, vi], beta[b, :, vi], chunk)
    return S, o


def max_rel(x, ref, axes=None):
    """Normwise relative error max|x - ref| / max|ref|.

    The error measure of "24 · GDN linear attention to GPU", section 6 (the
    f32 oracle check: max_abs_err / max_abs_ref).  With ``axes`` it is taken
    per slice over those axes and the worst slice is returned.
    """
    x, ref = _f64(x), _f64(ref)
    err = np.abs(x - ref)
    if axes is None:
        den = np.max(np.abs(ref))
        return float(np.max(err) / den) if den > 0 else float(np.max(err))
    num = np.max(err, axis=axes)
    den = np.max(np.abs(ref), axis=axes)
    r = np.where(den > 0, num / np.where(den > 0, den, 1.0), num)
    return float(np.max(r))
