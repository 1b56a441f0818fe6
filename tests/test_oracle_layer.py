"""The layer-core oracle (conv1d + SiLU, q/k normalisation, gates around the
recurrence) against its pins, and planted slips in it caught by them."""

import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_ref.c")


@pytest.mark.parametrize("pin", oracle_pins.LAYER_PINS, ids=lambda p: p.__name__)
def test_layer_pin(oracle_mod, pin):
    pin(oracle_mod.run_layer, oracle_mod.run_f32)


LAYER_MUTANTS = {
    "a_b_swapped": ("gate_softplus(a[row * vh + h] + dt_bias[h])",
                    "gate_softplus(b[row * vh + h] + dt_bias[h])"),
    "history_newest_first": ("win[(size_t)j * C + ch];",
                             "win[(size_t)(ck - 1 - j) * C + ch];"),
    "no_history_shift": ("memcpy(hs, rows + (size_t)T * C, sizeof(float) * nh * C);",
                         "(void)0;"),
    "no_silu": ("act[ch] = y * logistic(y);  /* SiLU */", "act[ch] = y;"),
    "softplus_branch": ("if (x > 20.0f) return x;", "if (x > 20.0f) return 20.0f;"),
    "no_norm_eps_sqrt": ("const float nrm = sqrtf(ss + eps);",
                         "const float nrm = ss + eps;"),
    "k_head_offset": ("r < (size_t)kh ? qu + r * (size_t)kd",
                      "r < (size_t)kh ? ku + r * (size_t)kd"),
    "window_one_row_late": ("const float *win = rows + (size_t)t * C;",
                            "const float *win = rows + (size_t)(t + (t > 0)) * C;"),
}


def _runners(tmp, name):
    src = open(SRC).read()
    old, new = LAYER_MUTANTS[name]
    assert src.count(old) == 1, name
    path = os.path.join(tmp, "m.c")
    open(path, "w").write(src.replace(old, new))
    so = os.path.join(tmp, "m.so")
    cc = shutil.which("gcc") or shutil.which("cc")
    subprocess.run([cc, "-O2", "-std=c11", "-ffp-contract=off", "-fPIC",
                    "-shared", path, "-o", so, "-lm"], check=True)
    lib = ctypes.CDLL(so)
    fp = ctypes.POINTER(ctypes.c_float)
    lib.gdn_oracle_layer.argtypes = [ctypes.c_int] * 7 + [ctypes.c_float] + [fp] * 10
    lib.gdn_oracle_layer.restype = ctypes.c_int
    P = lambda a: a.ctypes.data_as(fp)

    def run_layer(S, hist, x, w, a, b, A_log, dt, kh, eps=1e-6):
        S = np.ascontiguousarray(S, np.float32).copy()
        hist = np.ascontiguousarray(hist, np.float32).copy()
        x, w, a, b, A_log, dt = (np.ascontiguousarray(t, np.float32)
                                 for t in (x, w, a, b, A_log, dt))
        B, vh, kd, vd = S.shape
        T = x.shape[1]
        o = np.zeros((B, T, vh, vd), np.float32)
        rc = lib.gdn_oracle_layer(B, T, kh, vh, kd, vd, w.shape[1], eps, P(S),
                                  P(hist), P(x), P(w), P(a), P(b), P(A_log),
                                  P(dt), P(o), None)
        assert rc == 0
        return S, hist, o
    return run_layer


@pytest.mark.skipif(shutil.which("gcc") is None and shutil.which("cc") is None,
                    reason="no C compiler")
@pytest.mark.parametrize("name", sorted(LAYER_MUTANTS))
def test_layer_mutant_is_caught(oracle_mod, name):
    with tempfile.TemporaryDirectory() as tmp:
        run_layer = _runners(tmp, name)
        failed = []
        with np.errstate(all="ignore"):
            for pin in oracle_pins.LAYER_PINS:
                try:
                    pin(run_layer, oracle_mod.run_f32)
                except AssertionError:
                    failed.append(pin.__name__)
        assert failed, f"layer mutant {name} passed every pin"
