"""GPU parity of the paged decode step (gla_decode_step_paged) against the fp64 reference.

The batch rows name pages of a state pool through a slot table (a permutation with padding rows);
each row's output and page must match one reference decode step of that page, pages not named must
stay bit-identical, padding rows must produce zeros, and a CUDA graph of a fixed-width padded call
must replay correctly with new slot tables.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_linear_rnn_gb300 import build as B
from gated_linear_rnn_gb300 import gla
from gated_linear_rnn_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = 1e-2  # bf16 q, k, v, out; f32 state


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build_library()
    gla.load()
    torch.cuda.set_device(0)
    yield
    assert gla.gla_last_device_status() == 0


def make_case(N, nslots, seed, pad_rows=()):
    w = I.scaled(I.WORKLOADS["decode"], B=N)
    d = I.make_decode(w, device="cuda", seed=seed)
    g = torch.Generator().manual_seed(seed)
    pool = torch.randn((nslots, w.H, w.dk, w.dv), generator=g).mul_(0.02).cuda()
    slots = torch.randperm(nslots, generator=g)[:N].to(torch.int32)
    for r in pad_rows:
        slots[r] = -1
    return d, pool, slots.cuda()


def reference(d, pool0, slots):
    """One reference decode step per non-padding row, on that row's page."""
    s = slots.cpu().numpy()
    rows = np.nonzero(s >= 0)[0]
    o_ref = np.zeros((d["q"].shape[0],) + d["v"].shape[1:])
    pool_ref = pool0.copy()
    if rows.size:
        o, st = oracle.decode_step(d["q"][rows], d["k"][rows], d["v"][rows], d["log_decay"], pool0[s[rows]])
        o_ref[rows] = o
        pool_ref[s[rows]] = st
    return o_ref, pool_ref


def test_paged_matches_reference_with_padding():
    d, pool, slots = make_case(N=200, nslots=300, seed=3, pad_rows=(0, 17, 199))
    pool0 = pool.cpu().numpy().astype(np.float64)
    out = torch.empty_like(d["v"])
    gla.gla_decode_step_paged(d["q"], d["k"], d["v"], d["log_decay"], pool, slots, out)
    torch.cuda.synchronize()
    o_ref, pool_ref = reference(d, pool0, slots)
    o = out.float().cpu().numpy()
    assert oracle.rel_err(o, o_ref) <= TOL
    assert oracle.rel_err(pool.cpu().numpy(), pool_ref) <= 1e-5  # f32 state, one fma per element
    for r in (0, 17, 199):
        assert not o[r].any()  # padding rows: zero output
    untouched = np.setdiff1d(np.arange(300), slots.cpu().numpy())
    assert np.array_equal(pool.cpu().numpy()[untouched], pool0[untouched].astype(np.float32))
    assert gla.gla_last_device_status() == 0


def test_paged_with_identity_slots_equals_plain_decode():
    d, pool, _ = make_case(N=64, nslots=64, seed=4)
    ident = torch.arange(64, dtype=torch.int32, device="cuda")
    st_plain = pool.clone()
    out_p, out_d = torch.empty_like(d["v"]), torch.empty_like(d["v"])
    gla.gla_decode_step_paged(d["q"], d["k"], d["v"], d["log_decay"], pool, ident, out_p)
    gla.gla_decode_step(d["q"], d["k"], d["v"], d["log_decay"], st_plain, out_d)
    torch.cuda.synchronize()
    assert torch.equal(out_p, out_d) and torch.equal(pool, st_plain)


def test_paged_graph_replay_with_new_slots():
    """Capture one fixed-width padded call; replay it with rewritten slots and inputs."""
    N, nslots = 48, 96
    d, pool, slots = make_case(N=N, nslots=nslots, seed=5, pad_rows=(3,))
    q, k, v = d["q"].clone(), d["k"].clone(), d["v"].clone()
    out = torch.empty_like(v)
    ld = d["log_decay"]
    # warm up on a side stream, then capture
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    scratch = pool.clone()
    with torch.cuda.stream(s):
        gla.gla_decode_step_paged(q, k, v, ld, scratch, slots, out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gla.gla_decode_step_paged(q, k, v, ld, pool, slots, out)
    torch.cuda.synchronize()
    for it in range(3):
        d2, _, slots2 = make_case(N=N, nslots=nslots, seed=10 + it, pad_rows=(it, N - 1))
        q.copy_(d2["q"]), k.copy_(d2["k"]), v.copy_(d2["v"]), slots.copy_(slots2)
        pool0 = pool.cpu().numpy().astype(np.float64)
        graph.replay()
        torch.cuda.synchronize()
        o_ref, pool_ref = reference({"q": q.cpu(), "k": k.cpu(), "v": v.cpu(), "log_decay": ld.cpu()}, pool0, slots)
        assert oracle.rel_err(out.float().cpu().numpy(), o_ref) <= TOL
        assert oracle.rel_err(pool.cpu().numpy(), pool_ref) <= 1e-5
    assert gla.gla_last_device_status() == 0


def test_slot_beyond_pool_is_reported_and_skipped():
    d, pool, slots = make_case(N=8, nslots=16, seed=6)
    slots[2] = 16  # one past the pool
    pool0 = pool.clone()
    out = torch.empty_like(d["v"])
    gla.gla_decode_step_paged(d["q"], d["k"], d["v"], d["log_decay"], pool, slots, out)
    torch.cuda.synchronize()
    assert gla.STATUS[gla.gla_last_device_status()] == "GLA_ERR_DEVICE_ARG"
    assert not out[2].float().any()
    named = set(slots.cpu().tolist()) - {16}
    others = [i for i in range(16) if i not in named]
    assert torch.equal(pool[others], pool0[others])


def test_paged_decode_workload_full_size():
    """The bench's paged leg: N1280 x H16 states 96 x 192 as a pool read through a seeded permutation of the
    pages; every output and every page against the reference step."""
    w = I.WORKLOADS["decode"]
    d = I.make_decode(w, device="cuda", seed=0)
    pool = d["state"]
    slots = torch.randperm(w.B, generator=torch.Generator().manual_seed(7)).to(torch.int32).cuda()
    pool0 = pool.cpu().numpy().astype(np.float64)
    out = torch.empty_like(d["v"])
    gla.gla_decode_step_paged(d["q"], d["k"], d["v"], d["log_decay"], pool, slots, out)
    torch.cuda.synchronize()
    o_ref, pool_ref = reference(d, pool0, slots)
    assert oracle.rel_err(out.float().cpu().numpy(), o_ref) <= TOL
    assert oracle.rel_err(pool.cpu().numpy(), pool_ref) <= 1e-5
    assert gla.gla_last_device_status() == 0
