"""The gated-RMSNorm oracle against its closed-form pins, and planted slips
in it caught by them."""

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


@pytest.mark.parametrize("pin", oracle_pins.GATE_NORM_PINS,
                         ids=lambda p: p.__name__)
def test_gate_norm_pin(oracle_mod, pin):
    pin(oracle_mod.run_gate_norm)


GATE_NORM_MUTANTS = {
    "sum_not_mean": ("const float ms = ss / (float)vd;",
                     "const float ms = ss;"),
    "eps_outside_sqrt": ("const float rinv = 1.0f / sqrtf(ms + eps);",
                         "const float rinv = 1.0f / (sqrtf(ms) + eps);"),
    "sigmoid_gate": ("const float gate = zrow[c] / (1.0f + expf(-zrow[c]));",
                     "const float gate = 1.0f / (1.0f + expf(-zrow[c]));"),
    "weight_reversed": ("const float nw = n * w[c];",
                        "const float nw = n * w[vd - 1 - c];"),
    "no_weight": ("const float nw = n * w[c];", "const float nw = n;"),
    "first_row_rms": ("const float p = orow[c] * orow[c];",
                      "const float p = o[c] * o[c];"),
    "gate_of_next_channel": ("const float gate = zrow[c] / (1.0f + expf(-zrow[c]));",
                             "const float gate = zrow[(c + 1) % vd] / (1.0f + expf(-zrow[(c + 1) % vd]));"),
}


def _runner(tmp, name):
    src = open(SRC).read()
    old, new = GATE_NORM_MUTANTS[name]
    assert src.count(old) == 1, name
    path = os.path.join(tmp, "m.c")
    open(path, "w").write(src.replace(old, new))
    so = os.path.join(tmp, "m.so")
    cc = shutil.which("gcc") or shutil.which("cc")
    subprocess.run([cc, "-O2", "-std=c11", "-ffp-contract=off", "-fPIC",
                    "-shared", path, "-o", so, "-lm"], check=True)
    lib = ctypes.CDLL(so)
    fp = ctypes.POINTER(ctypes.c_float)
    lib.gdn_oracle_gate_norm.argtypes = [ctypes.c_int] * 4 + [ctypes.c_float] + [fp] * 4
    lib.gdn_oracle_gate_norm.restype = ctypes.c_int
    P = lambda a: a.ctypes.data_as(fp)

    def run_gate_norm(o, z, w, eps=1e-6):
        o, z, w = (np.ascontiguousarray(t, np.float32) for t in (o, z, w))
        y = np.zeros_like(o)
        B, T, vh, vd = o.shape
        assert lib.gdn_oracle_gate_norm(B, T, vh, vd, eps, P(o), P(z), P(w),
                                        P(y)) == 0
        return y
    return run_gate_norm


@pytest.mark.skipif(shutil.which("gcc") is None and shutil.which("cc") is None,
                    reason="no C compiler")
@pytest.mark.parametrize("name", sorted(GATE_NORM_MUTANTS))
def test_gate_norm_mutant_is_caught(name):
    with tempfile.TemporaryDirectory() as tmp:
        run = _runner(tmp, name)
        failed = []
        with np.errstate(all="ignore"):
            for pin in oracle_pins.GATE_NORM_PINS:
                try:
                    pin(run)
                except AssertionError:
                    failed.append(pin.__name__)
        assert failed, f"gate-norm mutant {name} passed every pin"
