"""Every plausible slip in the oracle is caught by at least one pin.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
in a temporary directory), builds it, and runs the pins of oracle_pins.py
against the broken build: at least one pin must fail.  The real oracle
passes all of them (test_oracle.py), so the pins discriminate.
"""

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

MUTANTS = {
    "delta_sign": ("const float d = v[dv] - kv[dv];",
                   "const float d = kv[dv] - v[dv];"),
    "o_from_old_state": ("const float p = t * qq;",
                         "const float p = (t - u) * qq;"),
    "interleaved_heads": ("hh = vi / rep;", "hh = vi % kh;"),
    "no_decay": ("const float t = row[dv] * alpha;",
                 "const float t = row[dv];"),
    "decay_after_readout": ("const float p = t * kk;",
                            "const float p = (t / alpha) * kk;"),
    "decay_sign": ("const float alpha = expf(g);",
                   "const float alpha = expf(-g);"),
    "no_beta": ("kv[dv] = d * beta;", "kv[dv] = d;"),
    "transposed_update": ("const float u = kk * kv[dv];",
                          "const float u = k[dv % kd] * kv[dk % vd];"),
    "missing_rank1": ("const float t = row[dv] + u;",
                      "const float t = row[dv];"),
}


def _build_mutant(name, tmp):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(tmp, f"{name}.so")
    cc = shutil.which("gcc") or shutil.which("cc")
    subprocess.run([cc, "-O2", "-std=c11", "-ffp-contract=off", "-fPIC",
                    "-shared", path, "-o", so, "-lm"], check=True)
    lib = ctypes.CDLL(so)
    fp = ctypes.POINTER(ctypes.c_float)
    lib.gdn_oracle_run.argtypes = [ctypes.c_int] * 6 + [fp] * 8
    lib.gdn_oracle_run.restype = ctypes.c_int
    return lib


def _runner(lib):
    def ptr(a):
        return None if a is None else a.ctypes.data_as(
            ctypes.POINTER(ctypes.c_float))

    def run(S, q, k, v, g, beta, ckpt=False):
        S = np.ascontiguousarray(S, np.float32).copy()
        q, k, v, g, beta = (np.ascontiguousarray(x, np.float32)
                            for x in (q, k, v, g, beta))
        B, vh, kd, vd = S.shape
        T, kh = q.shape[1], q.shape[2]
        o = np.zeros((B, T, vh, vd), np.float32)
        ck = np.zeros((T, B, vh, kd, vd), np.float32) if ckpt else None
        rc = lib.gdn_oracle_run(B, T, kh, vh, kd, vd, ptr(S), ptr(q), ptr(k),
                                ptr(v), ptr(g), ptr(beta), ptr(o), ptr(ck))
        assert rc == 0
        return (S, o, ck) if ckpt else (S, o)
    return run


@pytest.mark.skipif(shutil.which("gcc") is None and shutil.which("cc") is None,
                    reason="no C compiler")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    with tempfile.TemporaryDirectory() as tmp:
        run = _runner(_build_mutant(name, tmp))
        failed = []
        with np.errstate(all="ignore"):
            for pin in oracle_pins.ALL_PINS:
                try:
                    pin(run)
                except AssertionError:
                    failed.append(pin.__name__)
        assert failed, f"mutant {name} passed every pin"
