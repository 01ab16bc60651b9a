"""Pins for the fp64 reference of the causal depthwise Conv1d (width 4) + SiLU.

Checked against what the mathematics fixes: numpy's full convolution of each channel with its
kernel (a library routine, with the causal alignment written out here) followed by z * sigmoid(z)
evaluated with scipy's expit; the impulse response (a unit input returns the kernel taps in order);
SiLU's closed values (SiLU(0) = 0, odd part z/2); resume from the returned state; packing; and
planted mistakes in copies of the C source.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
from scipy.special import expit

import oracle

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "gla_oracle.c")


def case(B=2, T=29, D=6, seed=0, bias=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, T, D)).astype(np.float32)
    w = rng.standard_normal((D, 4))
    b = rng.standard_normal(D) if bias else None
    return x, w, b


def numpy_conv_silu(x, w, b, state=None):
    B, T, D = x.shape
    y = np.zeros((B, T, D))
    for bb in range(B):
        for c in range(D):
            hist = np.zeros(3) if state is None else state[bb, c]
            seq = np.concatenate([hist, x[bb, :, c].astype(np.float64)])
            # full convolution with the flipped taps: output index t + 3 sees inputs t .. t+3 of seq,
            # i.e. x_{t-3} .. x_t, weighted by w[c, 0] .. w[c, 3]
            full = np.convolve(seq, w[c][::-1], mode="full")
            z = full[3:3 + T] + (0.0 if b is None else b[c])
            y[bb, :, c] = z * expit(z)
    return y


@pytest.mark.parametrize("bias", [True, False])
def test_matches_numpy_convolution(bias):
    x, w, b = case(bias=bias)
    y, _ = oracle.conv1d_silu(x, w, b)
    assert np.max(np.abs(y - numpy_conv_silu(x, w, b))) < 1e-12


def test_with_incoming_state():
    x, w, b = case(seed=3)
    st = np.random.default_rng(9).standard_normal((2, 6, 3))
    y, _ = oracle.conv1d_silu(x, w, b, st)
    assert np.max(np.abs(y - numpy_conv_silu(x, w, b, st))) < 1e-12


def test_impulse_response_is_the_kernel():
    """A unit impulse at t = 0 with no bias: z_t = w[c, 3 - t] for t < 4, then 0."""
    D = 3
    x = np.zeros((1, 7, D), np.float32)
    x[0, 0] = 1.0
    w = np.random.default_rng(1).standard_normal((D, 4))
    y, _ = oracle.conv1d_silu(x, w)
    for t in range(7):
        z = w[:, 3 - t] if t < 4 else np.zeros(D)
        assert np.allclose(y[0, t], z / (1 + np.exp(-z)), atol=1e-15)


def test_silu_closed_values():
    """All-zero taps give z = b: SiLU(0) = 0 and SiLU(z) - SiLU(-z) = z."""
    x = np.random.default_rng(2).standard_normal((1, 5, 4)).astype(np.float32)
    w = np.zeros((4, 4))
    b = np.array([0.0, 1.5, -1.5, 3.0])
    y, _ = oracle.conv1d_silu(x, w, b)
    assert np.all(y[0, :, 0] == 0.0)
    assert np.allclose(y[0, :, 1] - y[0, :, 2], 1.5, atol=1e-15)


@pytest.mark.parametrize("split", [1, 2, 3, 17])
def test_resume_from_state(split):
    x, w, b = case(B=1, T=30, seed=4)
    full, st_full = oracle.conv1d_silu(x, w, b)
    a, st = oracle.conv1d_silu(x[:, :split], w, b)
    c, st2 = oracle.conv1d_silu(x[:, split:], w, b, st)
    assert np.array_equal(np.concatenate([a, c], axis=1), full) and np.array_equal(st2, st_full)


def test_short_sequence_state_keeps_older_inputs():
    x, w, b = case(B=1, T=2, D=2, seed=5)
    st_in = np.random.default_rng(6).standard_normal((1, 2, 3))
    _, st = oracle.conv1d_silu(x, w, b, st_in)
    assert np.array_equal(st[0, :, 0], st_in[0, :, 2]) and np.array_equal(st[0, :, 1:], x[0].T.astype(np.float64))


def test_packed_equals_separate():
    rng = np.random.default_rng(7)
    lens = [4, 0, 1, 13, 2]
    D = 5
    x = rng.standard_normal((1, sum(lens), D)).astype(np.float32)
    w = rng.standard_normal((D, 4))
    b = rng.standard_normal(D)
    st = rng.standard_normal((len(lens), D, 3))
    cu = np.concatenate([[0], np.cumsum(lens)])
    y, so = oracle.conv1d_silu(x, w, b, st, cu_seqlens=cu)
    for s, (a, e) in enumerate(zip(cu[:-1], cu[1:])):
        ys, ss = oracle.conv1d_silu(x[:, a:e], w, b, st[s:s + 1])
        assert np.array_equal(y[:, a:e], ys) and np.array_equal(so[s:s + 1], ss)


MUTANTS = {
    "taps_reversed": ("z += w[(size_t)c * 4 + k] * hist[k];", "z += w[(size_t)c * 4 + 2 - k] * hist[k];"),
    "current_tap_missing": ("z += w[(size_t)c * 4 + 3] * xt;", ""),
    "sigmoid_not_silu": ("y[(size_t)(r0 + t) * D + c] = z / (1.0 + exp(-z));", "y[(size_t)(r0 + t) * D + c] = 1.0 / (1.0 + exp(-z));"),
    "history_not_shifted": ("                hist[0] = hist[1];\n", ""),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_conv_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so), str(path), "-lm"])
    lib = ctypes.CDLL(str(so))
    lib.gla_oracle_conv1d_silu.restype = ctypes.c_int
    x, w, b = case(B=1, T=12, D=3, seed=8)
    xf = np.ascontiguousarray(x, np.float32)
    y = np.zeros((1, 12, 3))
    so_ = np.zeros((1, 3, 3))
    starts, lens = np.array([0], np.int64), np.array([12], np.int64)
    P = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    rc = lib.gla_oracle_conv1d_silu(P(xf), P(np.ascontiguousarray(w)), P(np.ascontiguousarray(b)), None, P(so_), P(y),
                                    P(starts), P(lens), ctypes.c_int(1), ctypes.c_int(3))
    assert rc == 0
    assert np.max(np.abs(y - numpy_conv_silu(x, w, b))) > 1e-6, f"mutant {name} survived"
