"""CPU oracle of the gated delta-rule state update.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline / reference legs may import this package.  The CUDA
library and its Python binding never import, link or call it, and share no
code with it: the two agree only through the seeded inputs of ``gdn_inputs``.

Contents
  gdn_ref.c  scalar fp32 implementation of the single-token step in the exact
             order of the articles' delta-recurrence kernel, applied token by
             token (see that file's header for the citations).  Built by
             ``build()`` into _build/libgdn_oracle.so.
  ref64.py   fp64 restatements: matrix form, explicit closed form of the
             linear recurrence, and the chunk-parallel form.
  gdn_ref.c also holds the layer core around the recurrence (conv1d + SiLU
             with rolling history, q/k normalisation, gate computation),
             ``run_layer``, and the gated RMSNorm on its output,
             ``run_gate_norm``.

Pins (each checked by tests that do not use the oracle's own code):
  run_f32     pinned by closed forms (alpha = 1 & beta = 0 identity, beta = 1
              read-back, zero-state rank-1, alpha = 0 reset), a hand-worked
              dyadic example, brute-force closed form for T = 1..3, and the
              fp64 matrix form.
  ref64.*     the matrix form and the closed form are pinned against each
              other and against the same closed-form special cases; the
              chunked form is pinned against the closed form.
  run_layer   pinned by closed forms of each step (identity convolution,
              SiLU/softplus/sigmoid values, unit norms, the +-20 softplus
              branches, history shift) and by equality with run_f32 when the
              layer steps are bypassed by construction.
  run_gate_norm pinned by closed forms: unit RMS of y / (w silu(z)), a
              +-1 row with silu(ln 3) = 0.75 ln 3, the eps placement on a
              constant row, per-channel weights, scale invariance and odd
              symmetry in o.
"""

from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_SRC = os.path.join(_HERE, "gdn_ref.c")

_lib = None


def build(force: bool = False) -> str:
    """Compile gdn_ref.c with gcc (fp32, no contraction, OpenMP if present)."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler found for the oracle")
    base = [cc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    r = subprocess.run(base[:-1] + ["-fopenmp", "-lm"], capture_output=True,
                       text=True)
    if r.returncode != 0:  # no OpenMP runtime: single-threaded build
        r = subprocess.run(base, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        fp = ctypes.POINTER(ctypes.c_float)
        lib.gdn_oracle_run.argtypes = [ctypes.c_int] * 6 + [fp] * 8
        lib.gdn_oracle_run.restype = ctypes.c_int
        lib.gdn_oracle_threads.restype = ctypes.c_int
        lib.gdn_oracle_layer.argtypes = [ctypes.c_int] * 7 + [ctypes.c_float] + [fp] * 10
        lib.gdn_oracle_layer.restype = ctypes.c_int
        lib.gdn_oracle_set_threads.argtypes = [ctypes.c_int]
        lib.gdn_oracle_gate_norm.argtypes = [ctypes.c_int] * 4 + \
            [ctypes.c_float] + [fp] * 4
        lib.gdn_oracle_gate_norm.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _f32c(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def threads() -> int:
    return _load().gdn_oracle_threads()


def set_threads(n: int) -> None:
    _load().gdn_oracle_set_threads(int(n))


def run_f32(S, q, k, v, g, beta, ckpt: bool = False):
    """Advance all heads over T tokens with the scalar fp32 oracle.

    S [B][vh][kd][vd]; q, k [B][T][kh][kd]; v [B][T][vh][vd]; g, beta
    [B][T][vh].  Returns (S_T, o) or (S_T, o, ckpt) with ckpt [T][B][vh][kd][vd],
    ckpt[t] = state after token t.  Inputs are not modified.
    """
    lib = _load()
    S = _f32c(S).copy()
    q, k, v, g, beta = map(_f32c, (q, k, v, g, beta))
    B, vh, kd, vd = S.shape
    T, kh = q.shape[1], q.shape[2]
    if q.shape != (B, T, kh, kd) or k.shape != q.shape or \
            v.shape != (B, T, vh, vd) or g.shape != (B, T, vh) or \
            beta.shape != g.shape:
        raise ValueError("inconsistent oracle input shapes")
    o = np.zeros((B, T, vh, vd), dtype=np.float32)
    ck = np.zeros((T, B, vh, kd, vd), dtype=np.float32) if ckpt else None
    rc = lib.gdn_oracle_run(B, T, kh, vh, kd, vd, _ptr(S), _ptr(q), _ptr(k),
                            _ptr(v), _ptr(g), _ptr(beta), _ptr(o), _ptr(ck))
    if rc != 0:
        raise RuntimeError(f"gdn_oracle_run failed ({rc})")
    return (S, o, ck) if ckpt else (S, o)


def run_layer(S, hist, x, conv_w, a, b, A_log, dt_bias, kh, eps=1e-6,
              ckpt: bool = False):
    """The layer core (conv1d + SiLU with history, q/k normalisation, gates,
    recurrence) over T tokens.  Shapes: S [B][vh][kd][vd], hist
    [B][ck-1][conv_dim], x [B][T][conv_dim], conv_w [conv_dim][ck], a, b
    [B][T][vh], A_log, dt_bias [vh].  Returns (S_T, hist_T, o[, ckpt])."""
    lib = _load()
    S = _f32c(S).copy()
    hist = _f32c(hist).copy()
    x, conv_w, a, b, A_log, dt_bias = map(_f32c, (x, conv_w, a, b, A_log, dt_bias))
    B, vh, kd, vd = S.shape
    T = x.shape[1]
    ck = conv_w.shape[1]
    if x.shape != (B, T, 2 * kh * kd + vh * vd) or hist.shape != (B, ck - 1, x.shape[2]):
        raise ValueError("inconsistent layer shapes")
    o = np.zeros((B, T, vh, vd), dtype=np.float32)
    ck_ = np.zeros((T, B, vh, kd, vd), dtype=np.float32) if ckpt else None
    rc = lib.gdn_oracle_layer(B, T, kh, vh, kd, vd, ck, float(eps), _ptr(S),
                              _ptr(hist), _ptr(x), _ptr(conv_w), _ptr(a), _ptr(b),
                              _ptr(A_log), _ptr(dt_bias), _ptr(o), _ptr(ck_))
    if rc != 0:
        raise RuntimeError(f"gdn_oracle_layer failed ({rc})")
    return (S, hist, o, ck_) if ckpt else (S, hist, o)


def run_gate_norm(o, z, w, eps=1e-6):
    """Gated RMSNorm of the recurrence output per (sequence, token, value
    head): o, z [B][T][vh][vd], w [vd].  Returns y, same shape as o."""
    lib = _load()
    o, z, w = map(_f32c, (o, z, w))
    if o.ndim != 4 or z.shape != o.shape or w.shape != (o.shape[3],):
        raise ValueError("inconsistent gate-norm shapes")
    B, T, vh, vd = o.shape
    y = np.zeros_like(o)
    rc = lib.gdn_oracle_gate_norm(B, T, vh, vd, float(eps), _ptr(o), _ptr(z),
                                  _ptr(w), _ptr(y))
    if rc != 0:
        raise RuntimeError(f"gdn_oracle_gate_norm failed ({rc})")
    return y


def run_inputs(inp, ckpt: bool = False):
    """``run_f32`` on a ``gdn_inputs.GDNInputs``."""
    return run_f32(inp.S, inp.q, inp.k, inp.v, inp.g, inp.beta, ckpt=ckpt)
