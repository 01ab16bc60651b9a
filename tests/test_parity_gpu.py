"""GPU parity: every CUDA path against the fp64 reference, through the C ABI.

Bar (per tensor, O and the final state separately): max|gpu - ref| / max|ref|
<= 1e-2 for bf16 inputs (f32 accumulate) and <= 1e-4 for f32 inputs.
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


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build_library()
    gla.load()
    torch.cuda.set_device(0)
    yield
    assert gla.gla_last_device_status() == 0


def run_prefill(d, chunk):
    out, hT = gla.chunk_fwd(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], chunk=chunk,
                            cu_seqlens=d["cu_dev"])
    torch.cuda.synchronize()
    return out, hT


def with_dev_cu(d):
    d["cu_dev"] = None if d["cu_seqlens"] is None else d["cu_seqlens"].cuda()
    return d


def rel_err_rows(got, ref, rows=4096):
    """max|got - ref| / max|ref| over the whole tensor, taken over blocks of the token axis (a full-size
    output widened to float64 in one piece would need several times the host memory)."""
    num = den = 0.0
    for a in range(0, ref.shape[1], rows):
        g = got[:, a:a + rows].float().cpu().numpy().astype(np.float64)
        r = ref[:, a:a + rows]
        num = max(num, float(np.max(np.abs(g - r))))
        den = max(den, float(np.max(np.abs(r))))
    return num / den if den else num


def check_prefill(w, chunk=None, units=None, seed=0, **kw):
    d = with_dev_cu(I.make_prefill(w, device="cuda", seed=seed, **kw))
    chunk = chunk or w.chunk
    out, hT = run_prefill(d, chunk)
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"],
                                    cu_seqlens=d["cu_seqlens"], units=units)
    if units is None and o_ref.size > (1 << 26):
        # full-size workloads: every chain, element by element, compared block by block
        eo, eh = rel_err_rows(out, o_ref), oracle.rel_err(hT.cpu().numpy(), h_ref)
        tol = TOL[w.dtype]
        assert eo <= tol and eh <= tol, f"out {eo:.3e} hT {eh:.3e} (tol {tol})"
        assert torch.isfinite(out).all() and torch.isfinite(hT).all()
        return eo, eh
    o = out.float().cpu().numpy()
    h = hT.cpu().numpy()
    if units is not None:
        # compare only the sampled chains
        sel_o, sel_r, sel_h, sel_hr = [], [], [], []
        cu = d["cu_seqlens"]
        for s, hh in units:
            if cu is None:
                sel_o.append(o[s, :, hh]); sel_r.append(o_ref[s, :, hh])
            else:
                a, b = int(cu[s]), int(cu[s + 1])
                sel_o.append(o[0, a:b, hh]); sel_r.append(o_ref[0, a:b, hh])
            sel_h.append(h[s, hh]); sel_hr.append(h_ref[s, hh])
        o, o_ref = np.concatenate(sel_o), np.concatenate(sel_r)
        h, h_ref = np.stack(sel_h), np.stack(sel_hr)
    eo, eh = oracle.rel_err(o, o_ref), oracle.rel_err(h, h_ref)
    tol = TOL[w.dtype]
    assert eo <= tol and eh <= tol, f"out {eo:.3e} hT {eh:.3e} (tol {tol})"
    assert np.isfinite(o).all() and np.isfinite(h).all()
    return eo, eh


# ---- the small fp32 workload, whole ----
def test_tiny_f32_workload():
    check_prefill(I.WORKLOADS["tiny_f32"])


@pytest.mark.parametrize("chunk", [16, 32, 64, 128])
def test_f32_chunks_ragged_tail(chunk):
    w = I.scaled(I.WORKLOADS["tiny_f32"], B=2, T=200, H=3, h0_std=0.5)
    check_prefill(w, chunk=chunk, seed=1)


# ---- bf16: several chunks and a ragged tail, every chunk size ----
@pytest.mark.parametrize("chunk", [16, 32, 64, 128])
def test_bf16_layer_shapes_small(chunk):
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=300, H=4, h0_std=0.02)
    check_prefill(w, chunk=chunk, seed=2)


@pytest.mark.parametrize("dk,dv", [(32, 64), (64, 64), (64, 128), (128, 192), (96, 128), (128, 64),
                                   (128, 128), (32, 192), (48, 80), (16, 16), (256, 64)])
def test_bf16_other_head_sizes(dk, dv):
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=1, T=260, H=2, dk=dk, dv=dv, h0_std=0.1)
    check_prefill(w, chunk=128, seed=3)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (32, 192)])
def test_bf16_direct_decay_form_head_sizes(dk, dv):
    """The direct decay form (lambda < e^-0.3: Q and K rows decayed in place after MMA1, per-element decay
    in the mask) with other tile sizes, a ragged tail and an initial state."""
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=390, H=2, dk=dk, dv=dv, h0_std=0.1)
    d = with_dev_cu(I.make_prefill(w, device="cuda", seed=14))
    d["log_decay"] = torch.tensor([-0.45, -1.7], device="cuda")
    out, hT = run_prefill(d, 128)
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"])
    assert oracle.rel_err(out.float().cpu().numpy(), o_ref) <= 1e-2
    assert oracle.rel_err(hT.cpu().numpy(), h_ref) <= 1e-2


def test_chunk_kernel_query_and_chunk64_on_tensor_cores():
    """gla_chunk_kernel names the kernel a call runs; chunk 64 runs on the tensor cores (two chunks per
    128-row tile) and gives exactly the chunk-128 result, forward and backward."""
    TC, SIMT = gla.KERNEL_TENSOR_CORE, gla.KERNEL_SIMT
    for op in (gla.OP_FORWARD, gla.OP_FORWARD_GATED, gla.OP_BACKWARD):
        assert gla.gla_chunk_kernel(op, gla.BF16, 96, 192, 128) == TC
        assert gla.gla_chunk_kernel(op, gla.BF16, 96, 192, 64) == TC
        assert gla.gla_chunk_kernel(op, gla.BF16, 96, 192, 32) == SIMT
        assert gla.gla_chunk_kernel(op, gla.F32, 96, 192, 128) == SIMT
        assert gla.gla_chunk_kernel(op, gla.BF16, 48, 80, 128) == SIMT
        assert gla.gla_chunk_kernel(op, gla.BF16, 128, 192, 128) == SIMT  # 240 KB of tiles
        assert gla.gla_chunk_kernel(op, gla.BF16, 96, 192, 100) == -2
    assert gla.gla_chunk_kernel(gla.OP_BACKWARD, gla.BF16, 32, 256, 128) == SIMT
    assert gla.gla_chunk_kernel(7, gla.BF16, 96, 192, 128) == -1
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=300, H=3, h0_std=0.02)
    d = with_dev_cu(I.make_backward(w, device="cuda", seed=17))
    o64, h64 = run_prefill(d, 64)
    o128, h128 = run_prefill(d, 128)
    assert torch.equal(o64, o128) and torch.equal(h64, h128)
    g64 = gla.chunk_bwd(d["q"], d["k"], d["v"], d["dout"], d["log_decay"], d["h0"], d["dhT"], chunk=64)
    g128 = gla.chunk_bwd(d["q"], d["k"], d["v"], d["dout"], d["log_decay"], d["h0"], d["dhT"], chunk=128)
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(g64, g128))
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"])
    assert oracle.rel_err(o64.float().cpu().numpy(), o_ref) <= 1e-2
    assert oracle.rel_err(h64.cpu().numpy(), h_ref) <= 1e-2


@pytest.mark.parametrize("T", [1, 2, 127, 128, 129, 256, 385])
def test_bf16_lengths(T):
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=T, H=2, h0_std=0.05)
    check_prefill(w, chunk=128, seed=4)


def test_ragged_small_with_empty_and_unit_sequences():
    w = I.scaled(I.WORKLOADS["ragged"], H=3)
    lengths = [0, 1, 127, 128, 129, 300, 5, 0, 257]
    check_prefill(w, lengths=lengths, seed=5)


def test_ragged_equal_lengths_take_distinct_sequences():
    """Packed batches are walked longest first; equal lengths are ranked by index, so every sequence is
    still taken by exactly one group of CTAs (ties, empty sequences and one long outlier)."""
    w = I.scaled(I.WORKLOADS["ragged"], H=2)
    lengths = [5, 5, 0, 200, 5, 200, 0, 5, 1, 1, 700, 5]
    check_prefill(w, lengths=lengths, seed=12)


def test_ragged_many_sequences_launch_order():
    """More packed sequences than the longest-first ranking takes on: the launch keeps blockIdx order."""
    w = I.scaled(I.WORKLOADS["ragged"], H=2, dk=32, dv=64)
    lengths = [(7 * i) % 41 for i in range(300)]
    check_prefill(w, lengths=lengths, seed=13)


def test_decay_extremes():
    """lambda = 1 (log_decay 0) and a vanishing decay in the same launch."""
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=1, T=300, H=2, h0_std=0.0)
    d = with_dev_cu(I.make_prefill(w, device="cuda", seed=6))
    d["log_decay"] = torch.tensor([0.0, -30.0], device="cuda")
    out, hT = run_prefill(d, 128)
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], None)
    assert oracle.rel_err(out.float().cpu().numpy(), o_ref) <= 1e-2
    assert oracle.rel_err(hT.cpu().numpy(), h_ref) <= 1e-2


@pytest.mark.parametrize("lds", [[-0.29, -0.31, -0.5, -2.0], [-1e-4, -0.05, -0.2999, -5.0]])
def test_bf16_mild_and_strong_decays(lds):
    """Both decay forms of the tensor-core kernel (factored for lambda >= e^-0.3, direct below)."""
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=400, H=4, h0_std=0.1)
    d = with_dev_cu(I.make_prefill(w, device="cuda", seed=11))
    d["log_decay"] = torch.tensor(lds, device="cuda")
    out, hT = run_prefill(d, 128)
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"])
    assert oracle.rel_err(out.float().cpu().numpy(), o_ref) <= 1e-2
    assert oracle.rel_err(hT.cpu().numpy(), h_ref) <= 1e-2


@pytest.mark.parametrize("B,H,T,h0_std,lds", [
    (1, 2, 2048, 0.0, None),             # 4 segments of 4 chunks
    (1, 3, 1000, 0.1, None),             # 2 segments, ragged last chunk
    (2, 4, 1536, 0.05, None),            # 3 segments per chain, 8 chains
    (1, 4, 2048, 0.1, [-0.01, -0.2, -0.5, -3.0]),  # direct decay form in both passes
])
def test_segmented_long_sequences(B, H, T, h0_std, lds):
    """Few chains and many chunks: the chains are split into segments (state-only pass, scan of
    the segment states, full pass from every segment's start state)."""
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=B, T=T, H=H, h0_std=h0_std)
    d = with_dev_cu(I.make_prefill(w, device="cuda", seed=12))
    if lds is not None:
        d["log_decay"] = torch.tensor(lds, device="cuda")
    launches = gla.gla_kernel_launches()
    out, hT = run_prefill(d, 128)
    assert gla.gla_kernel_launches() - launches == 3  # pass 1, scan, pass 2
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"])
    assert oracle.rel_err(out.float().cpu().numpy(), o_ref) <= 1e-2
    assert oracle.rel_err(hT.cpu().numpy(), h_ref) <= 1e-2


# ---- invariants on the GPU path ----
def test_deterministic_and_causal():
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=400, H=4, h0_std=0.02)
    d = with_dev_cu(I.make_prefill(w, device="cuda", seed=7))
    o1, h1 = run_prefill(d, 128)
    o2, h2 = run_prefill(d, 128)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    d["q"][:, -1] += 1
    d["k"][:, -1] -= 1
    d["v"][:, -1] *= -1
    o3, _ = run_prefill(d, 128)
    assert torch.equal(o1[:, :-1], o3[:, :-1])


@pytest.mark.parametrize("name", ["layer_bf16", "long_bf16"])
def test_repeated_launches_are_identical_and_never_time_out(name):
    """Back-to-back launches of a full-size workload: every result bit-identical, no wait timed out
    (a pipeline hand-off that could run a barrier two phases ahead would show up here)."""
    w = I.WORKLOADS[name]
    d = I.make_prefill(w, device="cuda", seed=13)
    nseq = d["q"].shape[0]
    outs = []
    for it in range(40 if name == "layer_bf16" else 12):
        out = torch.empty(d["q"].shape[:3] + (w.dv,), dtype=torch.bfloat16, device="cuda")
        hT = torch.empty(nseq, w.H, w.dk, w.dv, dtype=torch.float32, device="cuda")
        gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], out, hT, 128)
        if it < 2:
            outs.append((out, hT))
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[0][0], out) and torch.equal(outs[0][1], hT)


def test_resume_from_final_state():
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=512, H=2, h0_std=0.02)
    d = with_dev_cu(I.make_prefill(w, device="cuda", seed=8))
    o, hT = run_prefill(d, 128)
    T1 = 256
    oa, ha = gla.chunk_fwd(d["q"][:, :T1].contiguous(), d["k"][:, :T1].contiguous(), d["v"][:, :T1].contiguous(),
                           d["log_decay"], d["h0"], chunk=128)
    ob, hb = gla.chunk_fwd(d["q"][:, T1:].contiguous(), d["k"][:, T1:].contiguous(), d["v"][:, T1:].contiguous(),
                           d["log_decay"], ha, chunk=128)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"])
    assert oracle.rel_err(torch.cat([oa, ob], 1).float().cpu().numpy(), o_ref) <= 1e-2
    assert oracle.rel_err(hb.cpu().numpy(), h_ref) <= 1e-2


def test_single_token_prefill_equals_decode_step():
    w = I.scaled(I.WORKLOADS["decode"], B=6)
    d = I.make_decode(w, device="cuda", seed=9)
    s = d["state"].clone()
    o_dec = gla.decode_step(d["q"], d["k"], d["v"], d["log_decay"], s)
    o_pre, h_pre = gla.chunk_fwd(d["q"][:, None].contiguous(), d["k"][:, None].contiguous(),
                                 d["v"][:, None].contiguous(), d["log_decay"], d["state"], chunk=128)
    torch.cuda.synchronize()
    assert oracle.rel_err(o_pre[:, 0].float().cpu().numpy(), o_dec.float().cpu().numpy()) <= 1e-2
    assert oracle.rel_err(h_pre.cpu().numpy(), s.cpu().numpy()) <= 1e-2



@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_steps_follow_the_prefill_token_by_token(dtype):
    """Serving continuity: T recurrent decode steps from h0 reproduce the chunked prefill over the same
    T tokens, output by output and in the final state (T = 200 crosses a chunk boundary and ends in a
    partial chunk; the bf16 prefill runs on the tensor-core kernel).  Both sides are also held to the
    fp64 recurrence."""
    w = I.scaled(I.WORKLOADS["layer_bf16"] if dtype == "bf16" else I.WORKLOADS["tiny_f32"], B=2, T=200, H=4,
                 dk=96, dv=192, h0_std=0.02, dtype=dtype)
    d = I.make_prefill(w, device="cuda", seed=31)
    o_pre, h_pre = gla.chunk_fwd(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], chunk=128 if dtype == "bf16" else 64)
    state = d["h0"].clone()
    o_dec = torch.empty_like(o_pre)
    for t in range(w.T):
        o_dec[:, t] = gla.decode_step(d["q"][:, t].contiguous(), d["k"][:, t].contiguous(), d["v"][:, t].contiguous(),
                                      d["log_decay"], state)
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    o_ref, h_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["log_decay"], d["h0"])
    tol = TOL[dtype]
    pre, dec = o_pre.float().cpu().numpy(), o_dec.float().cpu().numpy()
    assert oracle.rel_err(pre, o_ref) <= tol and oracle.rel_err(dec, o_ref) <= tol
    assert oracle.rel_err(dec, pre) <= 2 * tol
    for t in (0, 127, 128, 199):  # token by token at the chunk edges as well
        assert oracle.rel_err(dec[:, t], pre[:, t]) <= 2 * tol, t
    assert oracle.rel_err(state.cpu().numpy(), h_ref) <= tol
    assert oracle.rel_err(state.cpu().numpy(), h_pre.cpu().numpy()) <= 2 * tol


# ---- decode ----
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv", [(96, 192), (64, 64), (100, 36), (8, 1024)])
def test_decode_step(dtype, dk, dv):
    w = I.scaled(I.WORKLOADS["decode"], B=37, H=3, dk=dk, dv=dv, dtype=dtype)
    d = I.make_decode(w, device="cuda", seed=10)
    s0 = d["state"].clone()
    o = gla.decode_step(d["q"], d["k"], d["v"], d["log_decay"], d["state"])
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.decode_step(d["q"], d["k"], d["v"], d["log_decay"], s0)
    tol = TOL[dtype]
    assert oracle.rel_err(o.float().cpu().numpy(), o_ref) <= tol
    assert oracle.rel_err(d["state"].cpu().numpy(), s_ref) <= tol


def test_decode_workload_full_size():
    """N = 1280 sequences x 16 heads, the launch the benchmark times."""
    w = I.WORKLOADS["decode"]
    d = I.make_decode(w, device="cuda", seed=0)
    s0 = d["state"].clone()
    o = gla.decode_step(d["q"], d["k"], d["v"], d["log_decay"], d["state"])
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.decode_step(d["q"], d["k"], d["v"], d["log_decay"], s0)
    assert oracle.rel_err(o.float().cpu().numpy(), o_ref) <= 1e-2
    assert oracle.rel_err(d["state"].cpu().numpy(), s_ref) <= 1e-2


# ---- full-size workloads: every chain of the workload against the reference ----
def test_layer_workload_full_size():
    """B8 T2048 H16 dk96 dv192, the launch the benchmark times: all 128 chains."""
    check_prefill(I.WORKLOADS["layer_bf16"])


def test_long_workload_full_size():
    """B1 T32768 H16 with h0 ~ N(0, 0.02^2) (segmented schedule): all 16 heads, every token."""
    check_prefill(I.WORKLOADS["long_bf16"])


def test_ragged_workload_full_size():
    """64 packed sequences of U[1, 8192] tokens with per-sequence h0, walked longest first: every
    (sequence, head) chain, every token and every final state."""
    check_prefill(I.WORKLOADS["ragged"])


# ---- errors recorded on the device ----
def test_bad_cu_seqlens_is_reported_not_trapped():
    w = I.scaled(I.WORKLOADS["ragged"], H=2)
    d = I.make_prefill(w, device="cuda", lengths=[10, 20, 30])
    bad = torch.tensor([0, 25, 20, 60], dtype=torch.int32, device="cuda")  # decreasing offsets
    out = torch.zeros_like(d["v"])
    gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], out, None, 128, bad)
    assert gla.gla_last_device_status() == -7
    assert gla.gla_last_device_status() == 0  # cleared
