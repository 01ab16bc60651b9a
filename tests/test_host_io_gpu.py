"""GPU parity of gla_chunk_fwd_host: the chunked forward on host arrays, copies overlapped by groups.

The entry point cuts the work into groups (of whole sequences, or, for few long sequences, ranges of
whole chunks of rows of every sequence, each started from the state the previous range left) and runs
copy-in, compute and copy-out of consecutive groups on three streams.  Checks: results against the
fp64 reference (same 1e-2 bar as the device entry point), bit-identity with the device entry point
called on the same groups (the kernels are deterministic and a group is computed as a call of its
own), pageable host memory, missing h0 / hT, the full layer workload (eight groups of one sequence)
and the full long-context workload (eight time ranges).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_linear_rnn_gb300 import build as B
from gated_linear_rnn_gb300 import gla
from gated_linear_rnn_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build_library()
    gla.load()
    torch.cuda.set_device(0)
    yield
    assert gla.gla_last_device_status() == 0


def host_forward(d, chunk, pinned=True, with_h0=True, with_hT=True):
    def h(t):
        t = t.cpu().contiguous()
        return t.pin_memory() if pinned else t
    q, k, v, ld = h(d["q"]), h(d["k"]), h(d["v"]), h(d["log_decay"])
    h0 = h(d["h0"]) if (with_h0 and d["h0"] is not None) else None
    out = torch.empty(q.shape[:3] + (v.shape[-1],), dtype=torch.bfloat16)
    hT = torch.empty(q.shape[0], q.shape[2], q.shape[3], v.shape[-1]) if with_hT else None
    if pinned:
        out = out.pin_memory()
        hT = hT.pin_memory() if hT is not None else None
    s = torch.cuda.Stream()
    gla.gla_chunk_fwd_host(q, k, v, ld, h0, out, hT, chunk, stream=s)
    s.synchronize()
    assert gla.gla_last_device_status() == 0
    return out, hT


def host_groups(B, T, H, dk, dv, chunk, with_h0=True, with_hT=True):
    """How gla_chunk_fwd_host cuts the work, by the rule its header states: at most 8 groups, none under
    8 MiB of copies unless the batch is smaller; whole sequences, or ranges of whole chunks when those
    make more groups.  Returns ("sequences", sequences per group) or ("ranges", rows per range)."""
    max_groups, min_bytes = 8, 8 << 20
    cdiv = lambda a, b: -(-a // b)
    seq_b = T * H * (2 * dk + 2 * dv) * 2 + (int(with_h0) + int(with_hT)) * H * dk * dv * 4
    per_group = cdiv(B, max_groups)
    if per_group < cdiv(min_bytes, seq_b):
        per_group = min(cdiv(min_bytes, seq_b), B)
    ngroups = cdiv(B, per_group)
    nch = cdiv(T, chunk)
    chunk_b = B * chunk * H * (2 * dk + 2 * dv) * 2
    per = cdiv(nch, max_groups)
    if per < cdiv(min_bytes, chunk_b):
        per = min(cdiv(min_bytes, chunk_b), nch)
    return ("ranges", per * chunk) if cdiv(nch, per) > ngroups else ("sequences", per_group)


def chained_device_forward(d, chunk, rows):
    """The device entry point over consecutive ranges of `rows` rows of every sequence, each range started
    from the state the previous one left."""
    T = d["q"].shape[1]
    h, outs = d["h0"], []
    for t0 in range(0, T, rows):
        sl = slice(t0, t0 + rows)
        o, h = gla.chunk_fwd(d["q"][:, sl].contiguous(), d["k"][:, sl].contiguous(), d["v"][:, sl].contiguous(),
                             d["log_decay"], h, chunk=chunk)
        outs.append(o)
    torch.cuda.synchronize()
    return torch.cat(outs, dim=1).cpu(), h.cpu()


def device_forward(d, chunk, b0=0, b1=None, with_h0=True):
    sl = slice(b0, b1)
    h0 = d["h0"][sl].contiguous() if (with_h0 and d["h0"] is not None) else None
    out, hT = gla.chunk_fwd(d["q"][sl].contiguous(), d["k"][sl].contiguous(), d["v"][sl].contiguous(),
                            d["log_decay"], h0, chunk=chunk)
    torch.cuda.synchronize()
    return out.cpu(), hT.cpu()


@pytest.mark.parametrize("dk,dv,chunk", [(96, 192, 128), (64, 128, 64), (128, 256, 128)])
def test_host_forward_matches_reference_and_device_call(dk, dv, chunk):
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=3, T=300, H=4, dk=dk, dv=dv, h0_std=0.02)
    d = I.make_prefill(w, device="cuda", seed=3)
    out, hT = host_forward(d, chunk)
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"])
    assert oracle.rel_err(out.float().numpy(), o_ref) <= 1e-2
    assert oracle.rel_err(hT.numpy(), h_ref) <= 1e-2
    # one group (the batch is under the group size): the same launch as the device entry point
    od, hd = device_forward(d, chunk)
    assert torch.equal(out, od) and torch.equal(hT, hd)


def test_host_forward_pageable_memory_and_no_states():
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=257, H=3)
    d = I.make_prefill(w, device="cuda", seed=4)
    out, _ = host_forward(d, 128, pinned=False, with_h0=False, with_hT=False)
    o_ref, _ = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], None)
    assert oracle.rel_err(out.float().numpy(), o_ref) <= 1e-2


def test_host_forward_layer_workload_eight_groups():
    """B8 T2048 H16 dk96 dv192: 39 MB of copies per sequence, so every sequence is its own group.
    Each group must equal the device entry point on that one sequence bit for bit, and every chain
    must match the reference."""
    w = I.WORKLOADS["layer_bf16"]
    d = I.make_prefill(w, device="cuda", seed=6)
    out, hT = host_forward(d, 128)
    for b in (0, 3, 7):
        od, hd = device_forward(d, 128, b, b + 1)
        assert torch.equal(out[b:b + 1], od) and torch.equal(hT[b:b + 1], hd), b
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"])
    assert oracle.rel_err(out.float().numpy(), o_ref) <= 1e-2
    assert oracle.rel_err(hT.numpy(), h_ref) <= 1e-2


def test_host_forward_rejects_device_tensors():
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=1, T=64, H=2)
    d = I.make_prefill(w, device="cuda", seed=1)
    out = torch.empty(1, 64, 2, w.dv, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        gla.gla_chunk_fwd_host(d["q"], d["k"], d["v"], d["log_decay"], None, out, None, 128)


@pytest.mark.parametrize("B_,chunk", [(1, 128), (2, 128), (1, 64), (1, 32)])
def test_host_forward_time_ranges_match_chained_device_calls(B_, chunk):
    """Few long sequences (T = 64 chunks of 128 + 100 rows): the work is cut in time, in whole chunks.  The
    result must equal the device entry point called range by range with the state carried over, bit for
    bit, and the reference within the bar (chunk 32 runs the SIMT kernel, the others the tensor cores)."""
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=B_, T=64 * 128 + 100, H=4, h0_std=0.02)
    kind, rows = host_groups(B_, w.T, w.H, w.dk, w.dv, chunk)
    assert kind == "ranges" and rows % chunk == 0 and rows < w.T, (kind, rows)
    d = I.make_prefill(w, device="cuda", seed=11)
    out, hT = host_forward(d, chunk)
    oc, hc = chained_device_forward(d, chunk, rows)
    assert torch.equal(out, oc) and torch.equal(hT, hc)
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"])
    assert oracle.rel_err(out.float().numpy(), o_ref) <= 1e-2
    assert oracle.rel_err(hT.numpy(), h_ref) <= 1e-2


def test_host_forward_time_ranges_pageable_memory_and_no_states():
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=1, T=4000, H=2)
    assert host_groups(1, w.T, w.H, w.dk, w.dv, 128, False, False)[0] == "ranges"
    d = I.make_prefill(w, device="cuda", seed=12)
    out, _ = host_forward(d, 128, pinned=False, with_h0=False, with_hT=False)
    o_ref, _ = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], None)
    assert oracle.rel_err(out.float().numpy(), o_ref) <= 1e-2


def test_host_forward_long_workload_eight_time_ranges():
    """B1 T32768 H16 with h0: eight ranges of 4,096 rows, every chain against the reference, and the
    result equal to the chained device calls bit for bit."""
    w = I.WORKLOADS["long_bf16"]
    assert host_groups(w.B, w.T, w.H, w.dk, w.dv, 128) == ("ranges", 4096)
    d = I.make_prefill(w, device="cuda", seed=13)
    out, hT = host_forward(d, 128)
    oc, hc = chained_device_forward(d, 128, 4096)
    assert torch.equal(out, oc) and torch.equal(hT, hc)
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"])
    assert oracle.rel_err(out.float().numpy(), o_ref) <= 1e-2
    assert oracle.rel_err(hT.numpy(), h_ref) <= 1e-2
