"""Plant plausible mistakes in copies of the fp64 reference and check the pins catch them.

Each mutant is a text edit of ``oracle/gla_oracle.c`` compiled into a temporary
library on the CPU; the committed oracle is never modified.  A mutant survives
only if the recurrence still agrees with the numpy attention form, the
hand-worked example and the zero-key closed form, so every mutant below must
fail at least one of them.
"""
import ctypes
import json
import math
import os
import subprocess

import numpy as np
import pytest

from test_oracle_pins import GOLDEN, attention_form_numpy, rand_case

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "gla_oracle.c")

MUTANTS = {
    "readout_before_update": (
        "                Si[j] = lam * Si[j] + ki * (double)vt[j];   /* S_t = lam S_{t-1} + k_t^T v_t */\n"
        "                ot[j] += qi * Si[j];                        /* o_t = q_t S_t                 */\n",
        "                ot[j] += qi * Si[j];\n"
        "                Si[j] = lam * Si[j] + ki * (double)vt[j];\n"),
    "decay_on_new_term": ("Si[j] = lam * Si[j] + ki * (double)vt[j];", "Si[j] = lam * (Si[j] + ki * (double)vt[j]);"),
    "q_k_swapped": ("const double ki = kt[i], qi = qt[i];", "const double ki = qt[i], qi = kt[i];"),
    "squared_decay": ("const double lam = exp(J->log_decay[h]);\n    double *S", "const double lam = exp(2.0 * J->log_decay[h]);\n    double *S"),
    "first_head_decay": ("const double lam = exp(J->log_decay[h]);\n    double *S", "const double lam = exp(J->log_decay[0]);\n    double *S"),
    "h0_dropped": ("    if (J->h0) memcpy(S, J->h0 + ((size_t)s * H + h) * dk * dv, sizeof(double) * dk * dv);\n    for (int64_t t = 0;",
                   "    for (int64_t t = 0;"),
    "v_column_reversed": ("ki * (double)vt[j];   /*", "ki * (double)vt[dv - 1 - j];   /*"),
}


def _build(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so), str(path), "-lm"])
    lib = ctypes.CDLL(str(so))
    lib.gla_oracle_recurrent.restype = ctypes.c_int
    return lib


def _recurrent(lib, q, k, v, ld, h0):
    B, T, H, dk = q.shape
    dv = v.shape[3]
    q, k, v = (np.ascontiguousarray(x, np.float32) for x in (q, k, v))
    ld = np.ascontiguousarray(ld, np.float64)
    h0 = None if h0 is None else np.ascontiguousarray(h0, np.float64)
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((B, H, dk, dv))
    starts = np.arange(B, dtype=np.int64) * T
    lens = np.full(B, T, dtype=np.int64)
    P = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    rc = lib.gla_oracle_recurrent(P(q), P(k), P(v), P(ld), P(h0), P(o), P(hT), P(starts), P(lens),
                                  ctypes.c_int(B), ctypes.c_int(H), ctypes.c_int(dk), ctypes.c_int(dv),
                                  None, ctypes.c_int(0), ctypes.c_int(1))
    assert rc == 0
    return o, hT


def _pins_pass(lib):
    q, k, v, ld, h0 = rand_case(B=2, T=19, H=3, dk=4, dv=6, seed=11)
    o, hT = _recurrent(lib, q, k, v, ld, h0)
    o_ref, hT_ref = attention_form_numpy(q, k, v, ld, h0)
    ok = max(np.max(np.abs(o - o_ref)) / np.max(np.abs(o_ref)),
             np.max(np.abs(hT - hT_ref)) / np.max(np.abs(hT_ref))) < 1e-12
    g = json.load(open(os.path.join(GOLDEN, "worked_example_2x2.json")))
    for case in g["cases"]:
        o2, h2 = _recurrent(lib, np.array(g["q"], np.float32)[None, :, None], np.array(g["k"], np.float32)[None, :, None],
                            np.array(g["v"], np.float32)[None, :, None], np.array([math.log(case["lam"])]),
                            np.array(g["h0"], np.float64)[None, None])
        ok = ok and np.allclose(o2[0, :, 0], case["o"], atol=1e-14) and np.allclose(h2[0, 0], case["hT"], atol=1e-14)
    k0 = np.zeros_like(k)
    o3, h3 = _recurrent(lib, q, k0, v, ld, h0)
    T = q.shape[1]
    g3 = np.exp(np.arange(1, T + 1)[None, :, None] * ld[None, None, :])
    o3_ref = g3[..., None] * np.einsum("bthd,bhde->bthe", q.astype(np.float64), h0)
    ok = ok and np.allclose(o3, o3_ref, rtol=1e-12, atol=1e-14)
    return bool(ok)


def test_unmodified_copy_passes(tmp_path):
    lib = _build(tmp_path, "identity", "#include <math.h>", "#include <math.h>")
    assert _pins_pass(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _build(tmp_path, name, old, new)
    assert not _pins_pass(lib), f"mutant {name} survived the pins"
