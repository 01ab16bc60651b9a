"""gla_chunk_fwd_noalloc: the forward for callers that may not let a library allocate device memory.

Some callers cannot have the library allocate: a host whose memory manager owns the whole device
pool, a serving loop with a fixed memory budget, a plugin host that only hands out the input and
output buffers.  For them the long-sequence schedule keeps its segment states in a fixed scratch
array that is part of the library image instead of taking memory with cudaMallocAsync.

The test calls the new entry point through the C ABI twice in a row, on shapes whose schedule
does use that scratch, and checks each result against gla_chunk_fwd within the bf16 tolerance
of the other parity tests.  It also checks that a call leaves the device's free memory unchanged.
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
        eo = oracle.rel_err(o_n.float().cpu().numpy(), o_a.float().cpu().numpy())
        eh = oracle.rel_err(h_n.cpu().numpy(), h_a.cpu().numpy())
        assert eo <= TOL and eh <= TOL, f"call {call}: out {eo:.3e} hT {eh:.3e}"


def test_noalloc_call_takes_no_device_memory():
    w = I.scaled(I.WORKLOADS["long_bf16"], B=1, T=4096, H=4, h0_std=0.02)
    d = I.make_prefill(w, device="cuda", seed=23)
    outputs(d, w, gla.gla_chunk_fwd_noalloc)  # the first call on a device looks up the scratch address
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    out = torch.empty(d["q"].shape[:3] + (w.dv,), dtype=torch.bfloat16, device="cuda")
    hT = torch.empty(1, w.H, w.dk, w.dv, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    gla.gla_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], out, hT, 128)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert gla.gla_last_device_status() == 0
