"""Pins for the fp64 reference backward, independent of the backward itself.

The backward (gradients of L = sum(dout * o) + sum(dhT * hT) through the recurrence) is checked
against what the mathematics fixes:
  - reverse-mode differentiation by torch autograd (float64, CPU) of a recurrence written out here;
  - exact finite differences: L is linear in each of q, k, v and h0 separately, so a central
    difference along a random direction equals the directional derivative up to rounding;
  - Euler's identity for the q-linear part: sum(dq * q) = sum(dout * o);
  - the vanishing-decay closed form (each state holds only its own token);
  - packing (a ragged batch equals its sequences run one by one) and chain selection.
Mutants planted in copies of the C source (on the CPU) must each fail at least one pin.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from test_oracle_pins import rand_case

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "gla_oracle.c")


def bwd_case(B=2, T=37, H=3, dk=5, dv=7, seed=3, int_vals=False):
    q, k, v, ld, h0 = rand_case(B, T, H, dk, dv, seed=seed, int_vals=int_vals)
    rng = np.random.default_rng(seed + 100)
    do = rng.standard_normal((B, T, H, dv)).astype(np.float32)
    dhT = rng.standard_normal((B, H, dk, dv))
    return q, k, v, do, ld, h0, dhT


def loss_from_forward(q, k, v, do, ld, h0, dhT):
    o, hT = oracle.recurrent(q, k, v, ld, h0)
    return float(np.sum(do.astype(np.float64) * o) + (np.sum(dhT * hT) if dhT is not None else 0.0)), o


def torch_autograd(q, k, v, do, ld, h0, dhT):
    """float64 autograd of S_t = lam S_{t-1} + k_t^T v_t, o_t = q_t S_t, written independently."""
    Q, K, V = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    S0 = torch.tensor(h0, dtype=torch.float64, requires_grad=True)
    lam = torch.exp(torch.tensor(ld, dtype=torch.float64))
    B, T, H, _ = q.shape
    outs = []
    S = S0
    for t in range(T):
        S = lam[None, :, None, None] * S + K[:, t, :, :, None] * V[:, t, :, None, :]
        outs.append(torch.einsum("bhd,bhde->bhe", Q[:, t], S))
    O = torch.stack(outs, dim=1)
    L = (O * torch.tensor(do, dtype=torch.float64)).sum() + (S * torch.tensor(dhT, dtype=torch.float64)).sum()
    L.backward()
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy(), S0.grad.numpy()


def test_backward_matches_torch_autograd():
    q, k, v, do, ld, h0, dhT = bwd_case(B=2, T=23, H=2, dk=4, dv=6)
    got = oracle.backward(q, k, v, do, ld, h0, dhT)
    ref = torch_autograd(q, k, v, do, ld, h0, dhT)
    for g, r, name in zip(got, ref, ("dq", "dk", "dv", "dh0")):
        assert oracle.rel_err(g, r) < 1e-12, name


@pytest.mark.parametrize("T", [1, 63, 64, 65, 150])
def test_backward_exact_directional_derivatives(T):
    """Central differences along random directions; exact because L is linear in each input alone."""
    # small-integer inputs and dyadic directions keep every perturbed input exact in float32
    q, k, v, do, ld, h0, dhT = bwd_case(B=1, T=T, H=2, dk=3, dv=5, seed=T, int_vals=True)
    dq, dk, dv, dh0 = oracle.backward(q, k, v, do, ld, h0, dhT)
    rng = np.random.default_rng(7 + T)
    for name, grad in (("q", dq), ("k", dk), ("v", dv), ("h0", dh0)):
        d = rng.integers(-4, 5, grad.shape).astype(np.float64) / 8.0
        args = dict(q=q, k=k, v=v, h0=h0)
        base = args[name].astype(np.float64)
        plus, minus = dict(args), dict(args)
        dt = np.float64 if name == "h0" else np.float32
        plus[name] = (base + d).astype(dt)
        minus[name] = (base - d).astype(dt)
        lp, _ = loss_from_forward(plus["q"], plus["k"], plus["v"], do, ld, plus["h0"], dhT)
        lm, _ = loss_from_forward(minus["q"], minus["k"], minus["v"], do, ld, minus["h0"], dhT)
        fd = (lp - lm) / 2.0
        an = float(np.sum(grad * d))
        assert abs(fd - an) <= 1e-9 * max(1.0, abs(an)), (name, fd, an)


def test_euler_identity_for_q():
    q, k, v, do, ld, h0, dhT = bwd_case(B=2, T=40, H=3, dk=4, dv=5, seed=9)
    dq, _, _, _ = oracle.backward(q, k, v, do, ld, h0, dhT)
    _, o = loss_from_forward(q, k, v, do, ld, h0, None)
    lhs = float(np.sum(dq * q.astype(np.float64)))
    rhs = float(np.sum(do.astype(np.float64) * o))
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs))


def test_vanishing_decay_closed_form():
    """lambda = e^-80: S_t = k_t^T v_t, so dq_t = (do_t.v_t) k_t, dk_t = (v_t.do_t) q_t, dv_t = (k_t.q_t) do_t."""
    q, k, v, do, ld, h0, dhT = bwd_case(B=1, T=9, H=1, dk=3, dv=4, seed=5)
    ld = np.array([-80.0])
    dq, dk, dv, dh0 = oracle.backward(q, k, v, do, ld, h0, None)
    Q, K, V, D = (x[0, :, 0].astype(np.float64) for x in (q, k, v, do))
    dv_dot = np.sum(D * V, axis=1, keepdims=True)
    assert np.allclose(dq[0, :, 0], dv_dot * K, rtol=1e-12, atol=1e-12)
    assert np.allclose(dk[0, :, 0], dv_dot * Q, rtol=1e-12, atol=1e-12)
    assert np.allclose(dv[0, :, 0], np.sum(K * Q, axis=1, keepdims=True) * D, rtol=1e-12, atol=1e-12)
    assert np.max(np.abs(dh0)) < 1e-30


def test_packed_backward_equals_separate_sequences():
    rng = np.random.default_rng(4)
    lens = [5, 0, 70, 1, 33]
    H, dk, dv = 2, 3, 4
    tot = sum(lens)
    q = rng.standard_normal((1, tot, H, dk)).astype(np.float32)
    k = rng.standard_normal((1, tot, H, dk)).astype(np.float32)
    v = rng.standard_normal((1, tot, H, dv)).astype(np.float32)
    do = rng.standard_normal((1, tot, H, dv)).astype(np.float32)
    h0 = rng.standard_normal((len(lens), H, dk, dv))
    dhT = rng.standard_normal((len(lens), H, dk, dv))
    ld = np.log([0.8, 0.97])
    cu = np.concatenate([[0], np.cumsum(lens)])
    dq, dk_, dv_, dh0 = oracle.backward(q, k, v, do, ld, h0, dhT, cu_seqlens=cu)
    for s, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        if b == a:
            assert np.allclose(dh0[s], dhT[s])  # an empty sequence passes dhT straight through
            continue
        r = oracle.backward(q[:, a:b], k[:, a:b], v[:, a:b], do[:, a:b], ld, h0[s:s + 1], dhT[s:s + 1])
        assert np.array_equal(dq[:, a:b], r[0]) and np.array_equal(dk_[:, a:b], r[1])
        assert np.array_equal(dv_[:, a:b], r[2]) and np.array_equal(dh0[s:s + 1], r[3])


def test_backward_units_subset_and_threads_agree():
    q, k, v, do, ld, h0, dhT = bwd_case(B=3, T=20, H=2, dk=3, dv=4, seed=12)
    full = oracle.backward(q, k, v, do, ld, h0, dhT, nthreads=1)
    part = oracle.backward(q, k, v, do, ld, h0, dhT, units=[(2, 1), (0, 0)], nthreads=4)
    assert np.array_equal(part[0][2, :, 1], full[0][2, :, 1]) and np.array_equal(part[2][0, :, 0], full[2][0, :, 0])
    assert np.array_equal(part[3][2, 1], full[3][2, 1])
    assert not np.any(part[0][1])  # chains not selected stay untouched (zeros)


# ---- mutants: plausible mistakes in the backward must fail a pin ---------------------------------
MUTANTS = {
    "readout_gradient_dropped": (
        "            for (int i = 0; i < dk; ++i)               /* G += q_t^T do_t */\n"
        "                for (int j = 0; j < dv; ++j) G[(size_t)i * dv + j] += (double)qt[i] * (double)dot[j];\n"
        "            for (int i = 0; i < dk; ++i) {             /* dq_t = do_t S_t^T;  dk_t = v_t G^T */",
        "            for (int i = 0; i < dk; ++i) {             /* dq_t = do_t S_t^T;  dk_t = v_t G^T */"),
    "missing_decay_of_G": ("for (size_t e = 0; e < sz; ++e) G[e] *= lam;", "for (size_t e = 0; e < sz; ++e) G[e] *= 1.0;"),
    "dq_uses_previous_state": ("const double *St = blk + (size_t)(t - t0) * sz;",
                               "const double *St = (t > t0) ? blk + (size_t)(t - t0 - 1) * sz : ck + (size_t)b * sz;"),
    "dk_from_q": ("ak += (double)vt[j] * G[(size_t)i * dv + j];", "ak += (double)dot[j] * G[(size_t)i * dv + j];"),
    "dhT_ignored": ("    if (J->dhT) memcpy(G, J->dhT + ((size_t)s * H + h) * sz, sizeof(double) * sz);\n", ""),
    "checkpoint_off_by_one": ("if (t % kCkpt == 0) memcpy(ck + (size_t)(t / kCkpt) * sz, S, sizeof(double) * sz);",
                              "if (t % kCkpt == 1 || t == 0) memcpy(ck + (size_t)(t / kCkpt) * sz, S, sizeof(double) * sz);"),
}


def _mutant_backward(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so), str(path), "-lm"])
    lib = ctypes.CDLL(str(so))
    lib.gla_oracle_backward.restype = ctypes.c_int
    return lib


def _call(lib, q, k, v, do, ld, h0, dhT):
    B, T, H, dk = q.shape
    dv = v.shape[3]
    q, k, v, do = (np.ascontiguousarray(x, np.float32) for x in (q, k, v, do))
    ld = np.ascontiguousarray(ld, np.float64)
    h0, dhT = np.ascontiguousarray(h0, np.float64), np.ascontiguousarray(dhT, np.float64)
    dq, dk_ = np.zeros((B, T, H, dk)), np.zeros((B, T, H, dk))
    dv_, dh0 = np.zeros((B, T, H, dv)), np.zeros((B, H, dk, dv))
    starts = np.arange(B, dtype=np.int64) * T
    lens = np.full(B, T, dtype=np.int64)
    P = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    c = ctypes.c_int
    rc = lib.gla_oracle_backward(P(q), P(k), P(v), P(do), P(ld), P(h0), P(dhT), P(dq), P(dk_), P(dv_), P(dh0),
                                 P(starts), P(lens), c(B), c(H), c(dk), c(dv), None, c(0), c(1))
    assert rc == 0
    return dq, dk_, dv_, dh0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_backward_mutant_is_caught(tmp_path, name):
    lib = _mutant_backward(tmp_path, name, *MUTANTS[name])
    q, k, v, do, ld, h0, dhT = bwd_case(B=1, T=70, H=2, dk=3, dv=4, seed=21)
    got = _call(lib, q, k, v, do, ld, h0, dhT)
    ref = torch_autograd(q, k, v, do, ld, h0, dhT)
    worst = max(oracle.rel_err(g, r) for g, r in zip(got, ref))
    assert worst > 1e-6, f"mutant {name} survived the autograd pin"
