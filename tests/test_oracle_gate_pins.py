"""Pins of the oracle's output gate (page "线性注意力模型如何实现固定推理状态", section "i14 与 Laplace 3B 架构",
QKVG projection: the gate g_t acts on the mixer output).  The page gives no formula; the oracle's reading is
o * SiLU(g) (kind 0) or o * sigmoid(g) (kind 1).  These tests pin that code to a library logistic function,
to values fixed by the definitions and to identities that a dropped factor, a sign slip or swapped kinds
would break."""
import numpy as np
import pytest
from scipy.special import expit

import oracle


def _inputs(n=4096, seed=0):
    rng = np.random.default_rng(seed)
    o = rng.standard_normal(n)
    g = (rng.standard_normal(n) * 4).astype(np.float32)
    return o, g


def test_gate_matches_library_logistic():
    o, g = _inputs()
    gd = g.astype(np.float64)
    np.testing.assert_allclose(oracle.output_gate(o, g, oracle.GATE_SILU), o * gd * expit(gd), rtol=1e-13, atol=0)
    np.testing.assert_allclose(oracle.output_gate(o, g, oracle.GATE_SIGMOID), o * expit(gd), rtol=1e-13, atol=0)


def test_gate_special_values():
    o = np.array([1.5, -2.0, 3.25])
    zero = np.zeros(3, dtype=np.float32)
    assert np.all(oracle.output_gate(o, zero, oracle.GATE_SILU) == 0.0)         # SiLU(0) = 0
    np.testing.assert_allclose(oracle.output_gate(o, zero, oracle.GATE_SIGMOID), o / 2, rtol=0, atol=0)
    big = np.full(3, 40.0, dtype=np.float32)                                      # gate fully open
    np.testing.assert_allclose(oracle.output_gate(o, big, oracle.GATE_SILU), o * 40.0, rtol=1e-15)
    np.testing.assert_allclose(oracle.output_gate(o, big, oracle.GATE_SIGMOID), o, rtol=1e-15)
    assert np.all(np.abs(oracle.output_gate(o, -big, oracle.GATE_SIGMOID)) < 1e-16)  # gate shut


def test_gate_identities():
    o, g = _inputs(seed=1)
    gd = g.astype(np.float64)
    # sigmoid(g) + sigmoid(-g) = 1 and SiLU(g) - SiLU(-g) = g
    np.testing.assert_allclose(oracle.output_gate(o, g, 1) + oracle.output_gate(o, -g, 1), o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.output_gate(o, g, 0) - oracle.output_gate(o, -g, 0), o * gd, rtol=1e-12,
                               atol=1e-12)
    # linear in o
    np.testing.assert_allclose(oracle.output_gate(3.0 * o, g, 0), 3.0 * oracle.output_gate(o, g, 0), rtol=1e-14)


def test_gate_rejects_bad_arguments():
    o, g = _inputs(16)
    with pytest.raises(ValueError):
        oracle.output_gate(o, g, 2)
    with pytest.raises(ValueError):
        oracle.output_gate(o, g[:8], 0)
