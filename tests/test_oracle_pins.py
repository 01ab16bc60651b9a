"""Pins for the fp64 reference, independent of the reference itself.

Each test checks the oracle against something the mathematics fixes: the
unrolled attention form evaluated with numpy matmuls, exact prefix sums,
a geometric-series closed form, degenerate decays, invariants (causality,
linearity, column separability, resume, packing) and a hand-worked example.
Together they catch a dropped term, a wrong decay exponent, a read-out taken
before the update, or a transposed state.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from gated_linear_rnn_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(B=2, T=37, H=3, dk=5, dv=7, seed=1, h0=True, int_vals=False):
    rng = np.random.default_rng(seed)
    if int_vals:
        q = rng.integers(-3, 4, (B, T, H, dk)).astype(np.float32)
        k = rng.integers(-3, 4, (B, T, H, dk)).astype(np.float32)
        v = rng.integers(-3, 4, (B, T, H, dv)).astype(np.float32)
        s0 = rng.integers(-3, 4, (B, H, dk, dv)).astype(np.float64) if h0 else None
    else:
        q = rng.standard_normal((B, T, H, dk)).astype(np.float32)
        k = rng.standard_normal((B, T, H, dk)).astype(np.float32)
        v = rng.standard_normal((B, T, H, dv)).astype(np.float32)
        s0 = rng.standard_normal((B, H, dk, dv)) if h0 else None
    ld = np.log(1.0 - np.geomspace(1 / 4, 1 / 64, H))
    return q, k, v, ld, s0


def attention_form_numpy(q, k, v, ld, h0):
    """O = ((Q K^T) .* D) V + diag(lam^(t+1)) Q h0 and hT, per (b, h), via numpy matmuls."""
    B, T, H, dk = q.shape
    dv = v.shape[3]
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((B, H, dk, dv))
    t = np.arange(T)
    diff = t[:, None] - t[None, :]
    for b in range(B):
        for h in range(H):
            Q = q[b, :, h].astype(np.float64)
            K = k[b, :, h].astype(np.float64)
            V = v[b, :, h].astype(np.float64)
            D = np.where(diff >= 0, np.exp(np.maximum(diff, 0) * ld[h]), 0.0)
            o[b, :, h] = ((Q @ K.T) * D) @ V
            w = np.exp((T - 1 - t) * ld[h])
            hT[b, h] = K.T @ (w[:, None] * V)
            if h0 is not None:
                o[b, :, h] += np.exp((t + 1) * ld[h])[:, None] * (Q @ h0[b, h])
                hT[b, h] += math.exp(T * ld[h]) * h0[b, h]
    return o, hT


@pytest.mark.parametrize("with_h0", [False, True])
def test_recurrence_matches_attention_form(with_h0):
    q, k, v, ld, h0 = rand_case(h0=with_h0)
    o, hT = oracle.recurrent(q, k, v, ld, h0)
    o_ref, hT_ref = attention_form_numpy(q, k, v, ld, h0)
    assert oracle.rel_err(o, o_ref) < 1e-12
    assert oracle.rel_err(hT, hT_ref) < 1e-12


def test_quadratic_c_matches_attention_form():
    q, k, v, ld, h0 = rand_case(seed=2)
    o, hT = oracle.quadratic(q, k, v, ld, h0)
    o_ref, hT_ref = attention_form_numpy(q, k, v, ld, h0)
    assert oracle.rel_err(o, o_ref) < 1e-12
    assert oracle.rel_err(hT, hT_ref) < 1e-12


def test_lambda_one_is_exact_prefix_sum():
    """lam = 1: S_t = S_0 + sum_{s<=t} k_s^T v_s exactly (integer data, fp64 exact)."""
    q, k, v, _, h0 = rand_case(B=1, T=40, H=2, dk=4, dv=6, int_vals=True)
    ld = np.zeros(2)
    o, hT = oracle.recurrent(q, k, v, ld, h0)
    outer = np.einsum("bthd,bthe->bthde", k.astype(np.float64), v.astype(np.float64))
    S = np.cumsum(outer, axis=1) + h0[:, None]
    o_ref = np.einsum("bthd,bthde->bthe", q.astype(np.float64), S)
    assert np.array_equal(o, o_ref)
    assert np.array_equal(hT, S[:, -1])


def test_scalar_geometric_series():
    """dk = dv = 1, q = k = v = 1: o_t = sum_{s<=t} lam^(t-s) = (1 - lam^(t+1)) / (1 - lam)."""
    T = 300
    ones = np.ones((1, T, 1, 1), dtype=np.float32)
    for lam in (0.5, 0.9, 0.999):
        o, hT = oracle.recurrent(ones, ones, ones, np.array([math.log(lam)]))
        t = np.arange(T)
        ref = (1 - lam ** (t + 1)) / (1 - lam)
        assert np.max(np.abs(o[0, :, 0, 0] - ref) / ref) < 1e-12
        assert abs(hT[0, 0, 0, 0] - ref[-1]) / ref[-1] < 1e-12


def test_vanishing_decay_keeps_only_diagonal():
    """lam -> 0: o_t = (q_t . k_t) v_t and hT = k_{T-1}^T v_{T-1}."""
    q, k, v, _, h0 = rand_case(B=1, T=9, H=2, dk=3, dv=4)
    ld = np.full(2, -80.0)
    o, hT = oracle.recurrent(q, k, v, ld, h0)
    qk = np.einsum("bthd,bthd->bth", q.astype(np.float64), k.astype(np.float64))
    assert oracle.rel_err(o, qk[..., None] * v) < 1e-12
    last = np.einsum("bhd,bhe->bhde", k[:, -1].astype(np.float64), v[:, -1].astype(np.float64))
    assert oracle.rel_err(hT, last) < 1e-12


def test_zero_keys_only_decay_the_initial_state():
    """k = 0: o_t = lam^(t+1) q_t h0 and hT = lam^T h0."""
    q, k, v, ld, h0 = rand_case(B=2, T=17, H=3, dk=4, dv=5)
    k[:] = 0
    o, hT = oracle.recurrent(q, k, v, ld, h0)
    T = q.shape[1]
    g = np.exp(np.arange(1, T + 1)[None, :, None] * ld[None, None, :])
    o_ref = g[..., None] * np.einsum("bthd,bhde->bthe", q.astype(np.float64), h0)
    assert oracle.rel_err(o, o_ref) < 1e-13
    assert oracle.rel_err(hT, np.exp(T * ld)[None, :, None, None] * h0) < 1e-13


def test_linear_in_v_and_columns_separable():
    q, k, v, ld, h0 = rand_case(seed=3)
    v2 = np.random.default_rng(9).standard_normal(v.shape).astype(np.float32)
    o1, s1 = oracle.recurrent(q, k, v, ld, h0)
    o2, s2 = oracle.recurrent(q, k, v2, ld, None)
    o12, s12 = oracle.recurrent(q, k, (v.astype(np.float64) + v2).astype(np.float32), ld, h0)
    vsum = v.astype(np.float64) + v2
    # only exact when v + v2 is representable; compare against the fp64 sum via the attention form
    o_ref, s_ref = attention_form_numpy(q, k, vsum, ld, h0)
    assert oracle.rel_err(o1 + o2, o_ref) < 1e-12
    assert oracle.rel_err(s1 + s2, s_ref) < 1e-12
    assert oracle.rel_err(o12, o_ref) < 1e-6  # float32 rounding of v + v2
    cols = [1, 4, 6]
    oc, sc = oracle.recurrent(q, k, v[..., cols], ld, h0[..., cols])
    assert np.array_equal(oc, o1[..., cols])
    assert np.array_equal(sc, s1[..., cols])


def test_causality_last_position():
    q, k, v, ld, h0 = rand_case(seed=4)
    o1, _ = oracle.recurrent(q, k, v, ld, h0)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[:, -1] += 5
    k2[:, -1] -= 3
    v2[:, -1] *= -2
    o2, _ = oracle.recurrent(q2, k2, v2, ld, h0)
    assert np.array_equal(o1[:, :-1], o2[:, :-1])
    assert not np.array_equal(o1[:, -1], o2[:, -1])


def test_resume_from_final_state():
    q, k, v, ld, h0 = rand_case(T=50, seed=5)
    o, hT = oracle.recurrent(q, k, v, ld, h0)
    T1 = 23
    oa, ha = oracle.recurrent(q[:, :T1], k[:, :T1], v[:, :T1], ld, h0)
    ob, hb = oracle.recurrent(q[:, T1:], k[:, T1:], v[:, T1:], ld, ha)
    assert np.array_equal(np.concatenate([oa, ob], axis=1), o)
    assert np.array_equal(hb, hT)


def test_packed_batch_equals_separate_sequences():
    rng = np.random.default_rng(6)
    lens = [5, 1, 0, 17, 9]
    H, dk, dv = 2, 3, 4
    total = sum(lens)
    q = rng.standard_normal((1, total, H, dk)).astype(np.float32)
    k = rng.standard_normal((1, total, H, dk)).astype(np.float32)
    v = rng.standard_normal((1, total, H, dv)).astype(np.float32)
    h0 = rng.standard_normal((len(lens), H, dk, dv))
    ld = np.log([0.9, 0.6])
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, hT = oracle.recurrent(q, k, v, ld, h0, cu_seqlens=cu)
    for s, L in enumerate(lens):
        a, b = cu[s], cu[s + 1]
        os_, hs = oracle.recurrent(q[:, a:b], k[:, a:b], v[:, a:b], ld, h0[s:s + 1])
        assert np.array_equal(o[:, a:b], os_)
        assert np.array_equal(hT[s], hs[0])
    assert np.array_equal(hT[2], h0[2])  # empty sequence: hT = h0


@pytest.mark.parametrize("T", [96, 50])
def test_chunked_form_matches_recurrence_for_every_chunk(T):
    q, k, v, ld, h0 = rand_case(B=1, T=T, H=2, dk=4, dv=6, seed=7)
    o, hT = oracle.recurrent(q, k, v, ld, h0)
    chunks = [c for c in range(1, T + 1) if T % c == 0] + [5, 7, 64, 128, T + 3]
    for C in sorted(set(chunks)):
        oc, hc = oracle.chunked(q, k, v, ld, C, h0)
        assert oracle.rel_err(oc, o) < 1e-12, C
        assert oracle.rel_err(hc, hT) < 1e-12, C


def test_decode_step_is_one_token_of_the_recurrence():
    rng = np.random.default_rng(8)
    N, H, dk, dv = 5, 3, 4, 6
    q = rng.standard_normal((N, H, dk)).astype(np.float32)
    k = rng.standard_normal((N, H, dk)).astype(np.float32)
    v = rng.standard_normal((N, H, dv)).astype(np.float32)
    st = rng.standard_normal((N, H, dk, dv))
    ld = np.log([0.99, 0.5, 0.1])
    o, st2 = oracle.decode_step(q, k, v, ld, st)
    o_ref, hT_ref = oracle.recurrent(q[:, None], k[:, None], v[:, None], ld, st)
    assert np.array_equal(o, o_ref[:, 0])
    assert np.array_equal(st2, hT_ref)
    lam = np.exp(ld)[None, :, None, None]
    assert oracle.rel_err(st2, lam * st + np.einsum("nhd,nhe->nhde", k.astype(np.float64), v.astype(np.float64))) < 1e-14


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "worked_example_2x2.json")))
    q = np.array(g["q"], np.float32)[None, :, None, :]
    k = np.array(g["k"], np.float32)[None, :, None, :]
    v = np.array(g["v"], np.float32)[None, :, None, :]
    h0 = np.array(g["h0"], np.float64)[None, None]
    for case in g["cases"]:
        ld = np.array([math.log(case["lam"])])
        o, hT = oracle.recurrent(q, k, v, ld, h0)
        np.testing.assert_allclose(o[0, :, 0], np.array(case["o"]), rtol=0, atol=1e-14)
        np.testing.assert_allclose(hT[0, 0], np.array(case["hT"]), rtol=0, atol=1e-14)
        for form in (oracle.quadratic,):
            o2, h2 = form(q, k, v, ld, h0)
            np.testing.assert_allclose(o2[0, :, 0], np.array(case["o"]), rtol=0, atol=1e-14)
            np.testing.assert_allclose(h2[0, 0], np.array(case["hT"]), rtol=0, atol=1e-14)


def test_units_subset_and_threads_agree():
    q, k, v, ld, h0 = rand_case(B=3, T=20, H=4, seed=10)
    o, hT = oracle.recurrent(q, k, v, ld, h0, nthreads=1)
    o4, hT4 = oracle.recurrent(q, k, v, ld, h0, nthreads=4)
    assert np.array_equal(o, o4) and np.array_equal(hT, hT4)
    units = [(2, 1), (0, 3)]
    ou, hu = oracle.recurrent(q, k, v, ld, h0, units=units)
    for b, h in units:
        assert np.array_equal(ou[b, :, h], o[b, :, h])
        assert np.array_equal(hu[b, h], hT[b, h])
    assert np.all(ou[1] == 0)


def test_rejects_bad_arguments():
    q, k, v, ld, h0 = rand_case(B=1, T=4, H=2)
    with pytest.raises(ValueError):
        oracle.recurrent(q, k, v, ld[:1])
    with pytest.raises(ValueError):
        oracle.chunked(q, k, v, ld, 0)
    with pytest.raises(ValueError):
        oracle.recurrent(q, k, v, ld, units=[(5, 0)])
    with pytest.raises(ValueError):
        oracle.recurrent(q, k, v, ld, cu_seqlens=[0, 3, 2])


def test_workload_decays_follow_the_geometric_rule():
    """log(1 - lam_h) evenly spaced from log(1/32) to log(1/4096) across 16 heads."""
    ld = I.log_decays(16).double().numpy()
    one_minus = -np.expm1(ld)
    steps = np.diff(np.log(one_minus))
    assert np.allclose(steps, steps[0], rtol=1e-5)
    assert abs(one_minus[0] - 1 / 32) < 1e-8 and abs(one_minus[-1] - 1 / 4096) < 1e-9
    ld2 = I.log_decays(2, 1 / 32, 1 / 512).double().numpy()
    assert np.allclose(-np.expm1(ld2), [1 / 32, 1 / 512], rtol=1e-6)
