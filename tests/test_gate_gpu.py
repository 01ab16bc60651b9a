"""GPU parity of the output gate fused into the forward and the decode step (gla_chunk_fwd_gated,
gla_decode_step_gated, gla_decode_step_paged_gated) against the fp64 reference: the oracle's recurrence
followed by its output gate (page "线性注意力模型如何实现固定推理状态", section "i14 与 Laplace 3B 架构",
QKVG projection: the gate g_t acts on the mixer output).

Bar: max|gpu - ref| / max|ref| <= 1e-2 per tensor (bf16 inputs and outputs, f32 accumulate); the final
state must not depend on the gate.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_linear_rnn_gb300 import build as B
from gated_linear_rnn_gb300 import gla
from gated_linear_rnn_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = 1e-2
KINDS = [gla.GATE_SILU, gla.GATE_SIGMOID]


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build_library()
    gla.load()
    torch.cuda.set_device(0)
    yield
    assert gla.gla_last_device_status() == 0


def check_gated_prefill(w, kind, seed, chunk=128, lengths=None, log_decay=None):
    d = I.make_prefill(w, device="cuda", seed=seed, lengths=lengths)
    if log_decay is not None:
        d["log_decay"] = torch.tensor(log_decay, device="cuda")
    cu = d["cu_seqlens"]
    cu_dev = None if cu is None else cu.cuda()
    nseq = d["q"].shape[0] if cu is None else cu.numel() - 1
    out = torch.empty(d["q"].shape[:3] + (w.dv,), dtype=torch.bfloat16, device="cuda")
    g = I.make_gate(out.shape, device="cuda", seed=seed)
    hT = torch.empty(nseq, w.H, w.dk, w.dv, device="cuda")
    gla.gla_chunk_fwd_gated(d["q"], d["k"], d["v"], g, d["log_decay"], d["h0"], out, hT, chunk, cu_dev,
                            gate_kind=kind)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], cu_seqlens=cu)
    ref = oracle.output_gate(o_ref, g, kind)
    eo = oracle.rel_err(out.float().cpu().numpy(), ref)
    eh = oracle.rel_err(hT.cpu().numpy(), h_ref)
    assert eo <= TOL and eh <= TOL, f"out {eo:.3e} hT {eh:.3e}"
    return out, hT


@pytest.mark.parametrize("kind", KINDS)
def test_gated_prefill_tensor_cores(kind):
    """The tensor-core path: several chunks, a ragged tail, an initial state."""
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=300, H=4, h0_std=0.02)
    check_gated_prefill(w, kind, seed=21)


@pytest.mark.parametrize("dk,dv,chunk", [(48, 80, 128), (96, 192, 32), (96, 192, 64), (64, 64, 128), (64, 128, 128),
                                          (128, 128, 128)])
def test_gated_prefill_other_shapes(dk, dv, chunk):
    """Head sizes and chunk lengths outside the tensor-core envelope (48 x 80, chunk 32) run the SIMT kernel;
    chunk 64 runs on the tensor cores as two chunks per tile, (64, 64) on the tensor cores with one 64-column
    gate group per warp, (64, 128) and (128, 128) with two (the layer's dv 192 has three)."""
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=1, T=260, H=2, dk=dk, dv=dv, h0_std=0.1)
    check_gated_prefill(w, gla.GATE_SILU, seed=22, chunk=chunk)


def test_gated_prefill_packed_with_empty_sequences():
    w = I.scaled(I.WORKLOADS["ragged"], H=3)
    check_gated_prefill(w, gla.GATE_SIGMOID, seed=23, lengths=[0, 1, 127, 128, 129, 300, 0, 257])


def test_gated_prefill_strong_decays():
    """The direct decay form of the tensor-core kernel (lambda < e^-0.3) with the gate."""
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=390, H=2, h0_std=0.1)
    check_gated_prefill(w, gla.GATE_SILU, seed=24, log_decay=[-0.45, -1.7])


def test_gated_prefill_segmented_long_sequence():
    """Few long chains take the segmented schedule; the gate is applied in its full pass."""
    w = I.scaled(I.WORKLOADS["long_bf16"], B=1, T=4096, H=4, h0_std=0.02)
    check_gated_prefill(w, gla.GATE_SILU, seed=25)


def test_gated_prefill_leaves_the_state_and_matches_the_ungated_output():
    """hT is bit-identical to the ungated forward's, and the gated output is the ungated output times the gate
    factor formed in bf16 pairs (O rounded to bf16, the factor times the row factor rounded to bf16, their
    product rounded), so it agrees with the ungated output times the factor to within four bf16 roundings
    (the reference's own output rounding included)."""
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=256, H=4, h0_std=0.02)
    d = I.make_prefill(w, device="cuda", seed=26)
    out_g, hT_g = check_gated_prefill(w, gla.GATE_SIGMOID, seed=26)
    out, hT = gla.chunk_fwd(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], chunk=128)
    torch.cuda.synchronize()
    assert torch.equal(hT, hT_g)
    g = I.make_gate(out.shape, device="cuda", seed=26)
    expect = out.float() * torch.sigmoid(g.float())
    assert (out_g.float() - expect).abs().max().item() <= 2 ** -6 * expect.abs().max().item()


@pytest.mark.parametrize("kind", KINDS)
def test_gated_decode_step(kind):
    w = I.scaled(I.WORKLOADS["decode"], B=40)
    d = I.make_decode(w, device="cuda", seed=27)
    g = I.make_gate((40, w.H, w.dv), device="cuda", seed=27)
    state = d["state"].clone()
    out = torch.empty(40, w.H, w.dv, dtype=torch.bfloat16, device="cuda")
    gla.gla_decode_step_gated(d["q"], d["k"], d["v"], g, d["log_decay"], state, out, gate_kind=kind)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.decode_step(d["q"], d["k"], d["v"], d["log_decay"], d["state"])
    assert oracle.rel_err(out.float().cpu().numpy(), oracle.output_gate(o_ref, g, kind)) <= TOL
    assert oracle.rel_err(state.cpu().numpy(), s_ref) <= 1e-5


def test_gated_paged_decode_with_padding_rows():
    w = I.scaled(I.WORKLOADS["decode"], B=24)
    d = I.make_decode(w, device="cuda", seed=28)
    gen = torch.Generator().manual_seed(28)
    nslots = 64
    pool = torch.randn((nslots, w.H, w.dk, w.dv), generator=gen).mul_(0.02).cuda()
    slots = torch.randperm(nslots, generator=gen)[:24].to(torch.int32)
    slots[[3, 17]] = -1
    slots = slots.cuda()
    g = I.make_gate((24, w.H, w.dv), device="cuda", seed=28)
    pool0 = pool.clone()
    out = torch.empty(24, w.H, w.dv, dtype=torch.bfloat16, device="cuda")
    gla.gla_decode_step_paged_gated(d["q"], d["k"], d["v"], g, d["log_decay"], pool, slots, out,
                                    gate_kind=gla.GATE_SILU)
    torch.cuda.synchronize()
    sl = slots.cpu().numpy()
    live = np.nonzero(sl >= 0)[0]
    o_ref, s_ref = oracle.decode_step(d["q"][live], d["k"][live], d["v"][live], d["log_decay"],
                                      pool0[torch.as_tensor(sl[live]).long().cuda()])
    ref = oracle.output_gate(o_ref, g[live], gla.GATE_SILU)
    assert oracle.rel_err(out[live].float().cpu().numpy(), ref) <= TOL
    assert oracle.rel_err(pool[torch.as_tensor(sl[live]).long().cuda()].cpu().numpy(), s_ref) <= 1e-5
    assert torch.count_nonzero(out[[3, 17]]).item() == 0


def test_gate_arguments_are_checked():
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=1, T=128, H=2)
    d = I.make_prefill(w, device="cuda", seed=29)
    out = torch.empty(1, 128, 2, w.dv, dtype=torch.bfloat16, device="cuda")
    g = I.make_gate(out.shape, device="cuda", seed=29)
    with pytest.raises(gla.GLAError):
        gla.gla_chunk_fwd_gated(d["q"], d["k"], d["v"], g, d["log_decay"], None, out, None, 128, gate_kind=2)
    rc = gla.load().gla_chunk_fwd_gated(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), None, 0,
                                        d["log_decay"].data_ptr(), None, out.data_ptr(), None, 1, 128, 2, w.dk,
                                        w.dv, 128, None, None)
    assert rc == -1  # GLA_ERR_ARG: no gate


@pytest.mark.parametrize("kind", KINDS)
def test_gated_prefill_layer_workload_full_size(kind):
    """The bench's gated leg at full size (B8 T2048 H16 dk96 dv192, g ~ N(0, 2^2)): every chain's gated
    output and final state against the reference."""
    check_gated_prefill(I.WORKLOADS["layer_bf16"], kind, seed=0)
