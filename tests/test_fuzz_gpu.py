"""Seeded random parity sweep of the forward and the backward against the fp64 reference.

Each case draws its shape (head sizes inside and outside the tensor-core envelopes, sequence
lengths from 1 to a few chunks, dense or packed), its decays (mild, strong or mixed heads) and
whether h0 / dhT are present from a generator seeded with the case number, so a failure names a
reproducible case.  Same bars as the other parity tests: 1e-2 (bf16 inputs), 1e-4 (f32 inputs).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_linear_rnn_gb300 import build as B
from gated_linear_rnn_gb300 import gla
from gated_linear_rnn_gb300 import inputs as I

pytestmark = pytest.mark.gpu

N_CASES = 24


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build_library()
    gla.load()
    torch.cuda.set_device(0)
    yield
    assert gla.gla_last_device_status() == 0


def draw(case):
    rng = np.random.default_rng(1000 + case)
    dk = int(rng.choice([32, 64, 96, 128]))
    dv = int(rng.choice([64, 128, 192]))
    H = int(rng.integers(1, 4))
    chunk = int(rng.choice([128, 128, 64]))
    ragged = bool(rng.integers(0, 2))
    dtype = "bf16" if rng.random() < 0.8 else "f32"
    decay = rng.choice(["mild", "strong", "mixed"])
    if decay == "mild":
        lo, hi = 1 / 32, 1 / 4096
    elif decay == "strong":
        lo, hi = 0.6, 0.3
    else:
        lo, hi = 0.6, 1 / 4096
    w = I.scaled(I.WORKLOADS["layer_bf16"], dtype=dtype, H=H, dk=dk, dv=dv, chunk=chunk, decay_lo=lo, decay_hi=hi,
                 h0_std=0.02 if rng.random() < 0.6 else 0.0)
    if ragged:
        lens = [int(x) for x in rng.integers(0, 3 * 128 + 40, int(rng.integers(1, 5)))]
        if sum(lens) == 0:
            lens[0] = 1
        kw = {"lengths": lens}
    else:
        kw = {"B": int(rng.integers(1, 3)), "T": int(rng.integers(1, 3 * 128 + 40))}
    dhT_std = 0.02 if rng.random() < 0.5 else 0.0
    return w, kw, dhT_std


@pytest.mark.parametrize("case", range(N_CASES))
def test_fuzz_forward_and_backward(case):
    w, kw, dhT_std = draw(case)
    tol = 1e-2 if w.dtype == "bf16" else 1e-4
    d = I.make_backward(w, device="cuda", seed=case, dhT_std=dhT_std, **kw)
    cu = None if d["cu_seqlens"] is None else d["cu_seqlens"].cuda()
    out, hT = gla.chunk_fwd(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], chunk=w.chunk, cu_seqlens=cu)
    grads = gla.chunk_bwd(d["q"], d["k"], d["v"], d["dout"], d["log_decay"], d["h0"], d["dhT"], chunk=w.chunk,
                          cu_seqlens=cu)
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], cu_seqlens=d["cu_seqlens"])
    g_ref = oracle.backward(d["q"], d["k"], d["v"], d["dout"], d["log_decay"], d["h0"], d["dhT"],
                            cu_seqlens=d["cu_seqlens"])
    errs = {"out": oracle.rel_err(out.float().cpu().numpy(), o_ref), "hT": oracle.rel_err(hT.cpu().numpy(), h_ref)}
    for name, g, r in zip(("dq", "dk", "dv", "dh0"), grads, g_ref):
        errs[name] = oracle.rel_err(g.float().cpu().numpy(), r)
    assert all(e <= tol for e in errs.values()), (case, w.dtype, w.dk, w.dv, w.H, w.chunk, kw, errs)


@pytest.mark.parametrize("case", range(12))
def test_fuzz_gated_forward(case):
    """The forward with the output gate (bf16 only) over the same seeded draws, both gate forms."""
    w, kw, _ = draw(case)
    w = I.scaled(w, dtype="bf16")
    kind = case % 2
    d = I.make_prefill(w, device="cuda", seed=case, **kw)
    cu = d["cu_seqlens"]
    cu_dev = None if cu is None else cu.cuda()
    nseq = d["q"].shape[0] if cu is None else cu.numel() - 1
    out = torch.empty(d["q"].shape[:3] + (w.dv,), dtype=torch.bfloat16, device="cuda")
    hT = torch.empty(nseq, w.H, w.dk, w.dv, device="cuda")
    g = I.make_gate(out.shape, device="cuda", seed=case)
    gla.gla_chunk_fwd_gated(d["q"], d["k"], d["v"], g, d["log_decay"], d["h0"], out, hT, w.chunk, cu_dev,
                            gate_kind=kind)
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], cu_seqlens=cu)
    eo = oracle.rel_err(out.float().cpu().numpy(), oracle.output_gate(o_ref, g, kind))
    eh = oracle.rel_err(hT.cpu().numpy(), h_ref)
    assert eo <= 1e-2 and eh <= 1e-2, (case, kind, w.dk, w.dv, w.H, w.chunk, kw, eo, eh)
