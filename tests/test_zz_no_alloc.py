"""gla_chunk_fwd_noalloc: the forward for callers that may not let a library allocate device memory.

Some callers cannot have the library allocate: a host whose memory manager owns the whole device
pool, a serving loop with a fixed memory budget, a plugin host that only hands out the input and
output buffers.  For them the long-sequence schedule keeps its segment states in a fixed scratch
array that is part of the library image instead of taking memory with cudaMallocAsync.

The no-alloc entry point runs the same kernels and the same schedule as gla_chunk_fwd; only the
address of the segment-state scratch differs.  So the tests call it through the C ABI twice in a row
on shapes whose schedule does use that scratch and require results bit-identical to gla_chunk_fwd
(a wrong segment offset or start state would show up as a difference, however small).  One case cuts
a single chain into as many segments as the GPU has room for, the most scratch any problem takes on
this GPU; its result is also held to the fp64 reference.  Another checks that a call leaves the
device's free memory unchanged.  GLA_ERR_SCRATCH_LIMIT cannot be produced on a 152-SM GB300: every
shape the tensor-core kernel takes fits the array there (a compile-time assertion in the library
checks that bound).

This file is collected last so that a failing run that stops at the first failure has already run
every other test; it passes alone in a fresh process as well.
"""
import pytest
import torch

import oracle
from gated_linear_rnn_gb300 import build as B
from gated_linear_rnn_gb300 import gla
from gated_linear_rnn_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = 1e-2  # bf16 inputs, f32 accumulate


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build_library()
    gla.load()
    torch.cuda.set_device(0)
    yield


def outputs(d, w, entry):
    nseq = d["q"].shape[0]
    out = torch.empty(d["q"].shape[:3] + (w.dv,), dtype=torch.bfloat16, device="cuda")
    hT = torch.empty(nseq, w.H, w.dk, w.dv, dtype=torch.float32, device="cuda")
    entry(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], out, hT, 128)
    return out, hT


@pytest.mark.parametrize("B_,H,T", [(1, 4, 2048), (1, 16, 32768)])
def test_noalloc_matches_allocating_entry_point_twice(B_, H, T):
    w = I.scaled(I.WORKLOADS["long_bf16"], B=B_, T=T, H=H, h0_std=0.02)
    for call, seed in enumerate((21, 22)):  # two calls in a row, different data each time
        d = I.make_prefill(w, device="cuda", seed=seed)
        launches = gla.gla_kernel_launches()
        o_n, h_n = outputs(d, w, gla.gla_chunk_fwd_noalloc)
        torch.cuda.synchronize()
        assert gla.gla_kernel_launches() - launches == 3, "shape should take the segmented schedule"
        assert gla.gla_last_device_status() == 0
        o_a, h_a = outputs(d, w, gla.gla_chunk_fwd)
        torch.cuda.synchronize()
        assert torch.equal(o_n, o_a) and torch.equal(h_n, h_a), f"call {call}: results differ"


def test_noalloc_most_segments_matches_and_follows_the_reference():
    """One chain long enough to be cut over every SM (the largest segment-state scratch on this GPU), twice."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = sms * 4 * 128 - 28  # one segment of 4 chunks per SM, the last chunk partial (100 tokens)
    w = I.scaled(I.WORKLOADS["long_bf16"], B=1, T=T, H=1, h0_std=0.02)
    for seed in (24, 25):
        d = I.make_prefill(w, device="cuda", seed=seed)
        o_n, h_n = outputs(d, w, gla.gla_chunk_fwd_noalloc)
        o_a, h_a = outputs(d, w, gla.gla_chunk_fwd)
        torch.cuda.synchronize()
        assert gla.gla_last_device_status() == 0
        assert torch.equal(o_n, o_a) and torch.equal(h_n, h_a)
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"])
    assert oracle.rel_err(o_n.float().cpu().numpy(), o_ref) <= TOL
    assert oracle.rel_err(h_n.cpu().numpy(), h_ref) <= TOL


def test_noalloc_call_takes_no_device_memory():
    w = I.scaled(I.WORKLOADS["long_bf16"], B=1, T=4096, H=4, h0_std=0.02)
    d = I.make_prefill(w, device="cuda", seed=23)
    outputs(d, w, gla.gla_chunk_fwd_noalloc)  # the first call on a device looks up the scratch address
    out = torch.empty(d["q"].shape[:3] + (w.dv,), dtype=torch.bfloat16, device="cuda")
    hT = torch.empty(1, w.H, w.dk, w.dv, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    gla.gla_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], out, hT, 128)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert gla.gla_last_device_status() == 0
