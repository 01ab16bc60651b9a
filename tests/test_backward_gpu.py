"""GPU parity of the backward (gla_chunk_bwd / gla_chunk_bwd_f32) against the fp64 reference backward.

Bar per gradient tensor (dq, dk, dv, dh0 separately): max|gpu - ref| / max|ref| <= 1e-2 for bf16
inputs (f32 accumulate, bf16 gradients) and <= 1e-4 for f32 inputs.  The reference differentiates
the recurrence one token at a time; the GPU runs three chunked recurrences, so agreement also
checks the chunked backward formulas.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_linear_rnn_gb300 import build as B
from gated_linear_rnn_gb300 import gla
from gated_linear_rnn_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "f32": 1e-4}
NAMES = ("dq", "dk", "dv", "dh0")


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build_library()
    gla.load()
    torch.cuda.set_device(0)
    yield
    assert gla.gla_last_device_status() == 0


def gpu_backward(d, chunk):
    cu = None if d["cu_seqlens"] is None else d["cu_seqlens"].cuda()
    grads = gla.chunk_bwd(d["q"], d["k"], d["v"], d["dout"], d["log_decay"], d["h0"], d["dhT"], chunk=chunk,
                          cu_seqlens=cu)
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    return [g.float().cpu().numpy() for g in grads]


def select(x, units, cu, state=False):
    """Rows (or states) of the sampled (sequence, head) chains, concatenated."""
    parts = []
    for s, h in units:
        if state:
            parts.append(x[s, h])
        elif cu is None:
            parts.append(x[s, :, h])
        else:
            parts.append(x[0, int(cu[s]):int(cu[s + 1]), h])
    return np.concatenate([p.reshape(-1) for p in parts])


def check_backward(w, chunk=None, units=None, seed=0, dhT_std=0.02, **kw):
    d = I.make_backward(w, device="cuda", seed=seed, dhT_std=dhT_std, **kw)
    chunk = chunk or w.chunk
    got = gpu_backward(d, chunk)
    ref = oracle.backward(d["q"], d["k"], d["v"], d["dout"], d["log_decay"], d["h0"], d["dhT"],
                          cu_seqlens=d["cu_seqlens"], units=units)
    errs = {}
    for name, g, r in zip(NAMES, got, ref):
        if units is not None:
            g, r = select(g, units, d["cu_seqlens"], name == "dh0"), select(r, units, d["cu_seqlens"], name == "dh0")
        errs[name] = oracle.rel_err(g, r)
    tol = TOL[w.dtype]
    assert all(e <= tol for e in errs.values()), errs
    return errs


def test_backward_tiny_f32():
    check_backward(I.WORKLOADS["tiny_f32"])


@pytest.mark.parametrize("chunk", [16, 32, 64, 128])
def test_backward_f32_chunks_and_ragged_tail(chunk):
    w = I.scaled(I.WORKLOADS["tiny_f32"], T=203, B=2, H=3, h0_std=0.02)
    check_backward(w, chunk=chunk)


@pytest.mark.parametrize("dk,dv", [(64, 128), (96, 192), (128, 64), (32, 256)])
def test_backward_bf16_head_sizes(dk, dv):
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=300, H=2, dk=dk, dv=dv, h0_std=0.02)
    check_backward(w)


def test_backward_bf16_no_h0_no_dhT():
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=257, H=4)
    check_backward(w, dhT_std=0.0)


def test_backward_ragged_packed_with_empty_sequence():
    w = I.scaled(I.WORKLOADS["ragged"], H=4, h0_std=0.02)
    check_backward(w, lengths=[130, 0, 1, 384, 77, 256])


@pytest.mark.parametrize("lo,hi", [(0.5, 0.25), (1e-6, 1e-7)])
def test_backward_decay_extremes(lo, hi):
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=1, T=384, H=2, h0_std=0.02, decay_lo=lo, decay_hi=hi)
    check_backward(w)


def test_backward_is_deterministic():
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=256, H=4, h0_std=0.02)
    d = I.make_backward(w, device="cuda", seed=5)
    a = gpu_backward(d, 128)
    b = gpu_backward(d, 128)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_backward_layer_workload_full_size():
    """The layer workload at full size (B8 T2048 H16 dk96 dv192): every chain's dq, dk, dv and dh0."""
    check_backward(I.WORKLOADS["layer_bf16"], seed=1)


def test_backward_matches_forward_linearisation():
    """sum(dq * q) = sum(dout * out) (the output is linear in q), using the GPU's own forward."""
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=320, H=2, h0_std=0.02)
    d = I.make_backward(w, device="cuda", seed=9, dhT_std=0.0)
    out, _ = gla.chunk_fwd(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], chunk=128)
    dq = gpu_backward(d, 128)[0]
    lhs = float(np.sum(dq.astype(np.float64) * d["q"].float().cpu().numpy()))
    rhs = float(np.sum(d["dout"].float().cpu().numpy().astype(np.float64) * out.float().cpu().numpy()))
    assert abs(lhs - rhs) <= 2e-2 * max(1.0, abs(rhs))


@pytest.mark.parametrize("T,H,lo,hi", [(4096, 2, 1 / 32, 1 / 4096), (4000, 3, 1 / 32, 1 / 4096), (3000, 2, 0.6, 1 / 4096)])
def test_backward_segmented_state_passes(T, H, lo, hi):
    """Few long chains: both state passes run segmented (segment end states from zero, a scan, then
    every segment from its start state); T = 4000 leaves a short last segment and a partial last
    chunk, the last case mixes heads the SIMT recurrences own."""
    w = I.scaled(I.WORKLOADS["long_bf16"], B=1, T=T, H=H, h0_std=0.02, decay_lo=lo, decay_hi=hi)
    check_backward(w, seed=T)


def rel_err_rows(got, ref, rows=4096):
    """max|got - ref| / max|ref| over a full-size gradient, in blocks of the token axis."""
    num = den = 0.0
    for a in range(0, ref.shape[1], rows):
        g = got[:, a:a + rows].float().cpu().numpy().astype(np.float64)
        r = ref[:, a:a + rows]
        num = max(num, float(np.max(np.abs(g - r))))
        den = max(den, float(np.max(np.abs(r))))
    return num / den if den else num


@pytest.mark.parametrize("name", ["long_bf16", "ragged"])
def test_backward_long_and_ragged_workloads_full_size(name):
    """The backward at the long-context size (B1 T32768 H16 with h0 and dhT: both state passes segmented) and
    at the ragged packed batch (64 sequences of U[1, 8192] tokens): every chain's dq, dk, dv and dh0."""
    w = I.WORKLOADS[name]
    d = I.make_backward(w, device="cuda", seed=2, dhT_std=0.02)
    cu = None if d["cu_seqlens"] is None else d["cu_seqlens"].cuda()
    grads = gla.chunk_bwd(d["q"], d["k"], d["v"], d["dout"], d["log_decay"], d["h0"], d["dhT"], chunk=128,
                          cu_seqlens=cu)
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    ref = oracle.backward(d["q"], d["k"], d["v"], d["dout"], d["log_decay"], d["h0"], d["dhT"],
                          cu_seqlens=d["cu_seqlens"])
    errs = {n: rel_err_rows(g, r) for n, g, r in zip(NAMES[:3], grads[:3], ref[:3])}
    errs["dh0"] = oracle.rel_err(grads[3].cpu().numpy(), ref[3])
    assert all(e <= TOL["bf16"] for e in errs.values()), errs
