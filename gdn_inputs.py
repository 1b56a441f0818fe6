"""Seeded synthetic inputs for the gated delta-rule state update.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests. It holds no arithmetic of the method itself: it only draws
random tensors with the shapes and value distributions of the decode and
prefill workloads and returns them as contiguous fp32 NumPy arrays in the
library's canonical layouts.

Layouts (row-major, fp32):
  S        [B][vh][kd][vd]     one state per (sequence, value head)
  q, k     [B][T][kh][kd]      T tokens per call (T = 1 for a single step)
  v        [B][T][vh][vd]
  g, beta  [B][T][vh]

Distributions (drawn in fp64 with NumPy's PCG64, transformed in fp64, cast to
fp32 once):
  S     ~ N(0, 0.02^2)  (std 0.02), or zeros for prefill
  q, k  ~ N(0, 1) per element, then each (b, t, key-head) row scaled to unit
          L2 norm
  v     ~ N(0, 1)
  g     = -softplus(x) * g_scale,  x ~ N(0, 1)   (log-domain decay, < 0)
  beta  = sigmoid(x),              x ~ N(0, 1)

Draw order from a single generator: S, q, k, v, g-source, beta-source.
"""

from __future__ import annotations

import dataclasses

import numpy as np

# Seeds of the named workloads: workload i uses SEED_BASE + i.
SEED_BASE = 20261202


@dataclasses.dataclass
class GDNInputs:
    S: np.ndarray
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    B: int
    T: int
    kh: int
    vh: int
    kd: int
    vd: int
    seed: int

    def step(self, t: int) -> "GDNInputs":
        """The inputs of token t alone (T = 1), as contiguous arrays."""
        sl = slice(t, t + 1)
        return GDNInputs(
            S=self.S, q=np.ascontiguousarray(self.q[:, sl]),
            k=np.ascontiguousarray(self.k[:, sl]),
            v=np.ascontiguousarray(self.v[:, sl]),
            g=np.ascontiguousarray(self.g[:, sl]),
            beta=np.ascontiguousarray(self.beta[:, sl]),
            B=self.B, T=1, kh=self.kh, vh=self.vh, kd=self.kd, vd=self.vd,
            seed=self.seed)

    def tokens(self, t0: int, t1: int) -> "GDNInputs":
        """Tokens t0..t1-1 as contiguous arrays (T = t1 - t0)."""
        sl = slice(t0, t1)
        return GDNInputs(
            S=self.S, q=np.ascontiguousarray(self.q[:, sl]),
            k=np.ascontiguousarray(self.k[:, sl]),
            v=np.ascontiguousarray(self.v[:, sl]),
            g=np.ascontiguousarray(self.g[:, sl]),
            beta=np.ascontiguousarray(self.beta[:, sl]),
            B=self.B, T=t1 - t0, kh=self.kh, vh=self.vh, kd=self.kd,
            vd=self.vd, seed=self.seed)

    def heads(self, b_idx, vi_idx) -> "GDNInputs":
        """Restrict to sequences b_idx and value heads vi_idx.

        vi_idx must be whole groups of value heads that share a key head
        (contiguous runs of rep = vh // kh heads starting at a multiple of
        rep), so the head mapping stays valid; the key heads kept are those
        groups' key heads in the same order.
        """
        b_idx = np.asarray(b_idx, dtype=np.int64)
        vi_idx = np.asarray(vi_idx, dtype=np.int64)
        rep = self.vh // self.kh
        if len(vi_idx) % rep or np.any(vi_idx.reshape(-1, rep)[:, 0] % rep) or \
           np.any(np.diff(vi_idx.reshape(-1, rep), axis=1) != 1):
            raise ValueError("vi_idx must be whole key-head groups")
        kh_idx = vi_idx.reshape(-1, rep)[:, 0] // rep
        return GDNInputs(
            S=np.ascontiguousarray(self.S[b_idx][:, vi_idx]),
            q=np.ascontiguousarray(self.q[b_idx][:, :, kh_idx]),
            k=np.ascontiguousarray(self.k[b_idx][:, :, kh_idx]),
            v=np.ascontiguousarray(self.v[b_idx][:, :, vi_idx]),
            g=np.ascontiguousarray(self.g[b_idx][:, :, vi_idx]),
            beta=np.ascontiguousarray(self.beta[b_idx][:, :, vi_idx]),
            B=len(b_idx), T=self.T, kh=len(kh_idx), vh=len(vi_idx),
            kd=self.kd, vd=self.vd, seed=self.seed)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / n


def make_inputs(seed: int, B: int, T: int, kh: int = 16, vh: int = 48,
                kd: int = 128, vd: int = 128, s_std: float = 0.02,
                zero_state: bool = False, g_scale: float = 1.0) -> GDNInputs:
    """Draw one workload's inputs (see the module docstring)."""
    if vh % kh:
        raise ValueError("vh must be a multiple of kh")
    rng = np.random.Generator(np.random.PCG64(seed))
    if zero_state:
        S = np.zeros((B, vh, kd, vd), dtype=np.float32)
    else:
        S = (rng.standard_normal((B, vh, kd, vd)) * s_std).astype(np.float32)
    q = _unit_rows(rng.standard_normal((B, T, kh, kd))).astype(np.float32)
    k = _unit_rows(rng.standard_normal((B, T, kh, kd))).astype(np.float32)
    v = rng.standard_normal((B, T, vh, vd)).astype(np.float32)
    xg = rng.standard_normal((B, T, vh))
    g = (-np.logaddexp(0.0, xg) * g_scale).astype(np.float32)
    xb = rng.standard_normal((B, T, vh))
    beta = (1.0 / (1.0 + np.exp(-xb))).astype(np.float32)
    return GDNInputs(S=S, q=q, k=k, v=v, g=g, beta=beta, B=B, T=T, kh=kh,
                     vh=vh, kd=kd, vd=vd, seed=seed)


# The named workloads (sizes from the decode / verify / prefill scenarios).
WORKLOADS = {
    "decode_b1": dict(B=1, T=1),                 # one decode step, one sequence
    "decode_b1_t64": dict(B=1, T=64),            # 64 chained decode steps
    "decode_b64": dict(B=64, T=1),               # batched decode, HBM-bound
    "verify_b32": dict(B=32, T=8),               # M-step verify, M in {2,4,8}
    "prefill_b8_t4096": dict(B=8, T=4096, zero_state=True, g_scale=0.1),
}

WORKLOAD_SEED = {name: SEED_BASE + i for i, name in enumerate(WORKLOADS)}


def make_workload(name: str, **overrides) -> GDNInputs:
    kw = dict(WORKLOADS[name])
    kw.update(overrides)
    return make_inputs(WORKLOAD_SEED[name], **kw)


@dataclasses.dataclass
class LayerInputs:
    S: np.ndarray        # [B][vh][kd][vd]
    hist: np.ndarray     # [B][ck-1][conv_dim]
    x: np.ndarray        # [B][T][conv_dim]
    conv_w: np.ndarray   # [conv_dim][ck]
    a: np.ndarray        # [B][T][vh]
    b: np.ndarray        # [B][T][vh]
    A_log: np.ndarray    # [vh]
    dt_bias: np.ndarray  # [vh]
    kh: int
    T: int


def make_layer_inputs(seed: int, B: int, T: int, kh: int = 16, vh: int = 48,
                      kd: int = 128, vd: int = 128, ck: int = 4,
                      s_std: float = 0.02) -> LayerInputs:
    """Raw inputs of the layer core (before convolution, normalisation and
    gates), drawn in this order from one PCG64 generator:
      S ~ N(0, s_std^2); hist, x ~ N(0, 1) (raw projections);
      conv_w ~ N(0, 1/ck) (unit-variance convolution outputs);
      a, b ~ N(0, 1);
      A_log = log(U(1, 16)) per head and dt_bias = softplus^-1(dt) with
      dt = exp(U(log 1e-3, log 1e-1)) per head, a common initialisation of
      such gates (no trained weights are available)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    conv_dim = 2 * kh * kd + vh * vd
    S = (rng.standard_normal((B, vh, kd, vd)) * s_std).astype(np.float32)
    hist = rng.standard_normal((B, ck - 1, conv_dim)).astype(np.float32)
    x = rng.standard_normal((B, T, conv_dim)).astype(np.float32)
    conv_w = (rng.standard_normal((conv_dim, ck)) / np.sqrt(ck)).astype(np.float32)
    a = rng.standard_normal((B, T, vh)).astype(np.float32)
    b = rng.standard_normal((B, T, vh)).astype(np.float32)
    A_log = np.log(rng.uniform(1.0, 16.0, vh)).astype(np.float32)
    dt = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), vh))
    dt_bias = (dt + np.log(-np.expm1(-dt))).astype(np.float32)
    return LayerInputs(S=S, hist=hist, x=x, conv_w=conv_w, a=a, b=b,
                       A_log=A_log, dt_bias=dt_bias, kh=kh, T=T)


def make_gate_norm_inputs(seed: int, B: int, T: int, vh: int = 48,
                          vd: int = 128):
    """Inputs of the gated RMSNorm on the update's output, drawn in this
    order from one PCG64 generator:
      o = N(0, 1) * s per (b, t, head) row, s = exp(U(log 1e-3, log 10))
          (rows of very different scale, as outputs of different heads are);
      z ~ N(0, 1) (the gate projection);
      w = 1 + 0.1 N(0, 1) per channel (around the usual all-ones start).
    Returns (o, z, w) as fp32 arrays [B][T][vh][vd], [B][T][vh][vd], [vd]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    s = np.exp(rng.uniform(np.log(1e-3), np.log(10.0), (B, T, vh, 1)))
    o = (rng.standard_normal((B, T, vh, vd)) * s).astype(np.float32)
    z = rng.standard_normal((B, T, vh, vd)).astype(np.float32)
    w = (1.0 + 0.1 * rng.standard_normal(vd)).astype(np.float32)
    return o, z, w
