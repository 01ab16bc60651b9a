"""The library inside CUDA graphs and on concurrent streams.

A serving or training loop captures its steps once and replays them.  These tests capture the
chunked forward (whole-chain and segmented schedules), the backward and a decode step in one graph,
replay it with new inputs copied into the captured buffers, and require results bit-identical to
eager calls on the same inputs (the kernels are deterministic).  A second test runs two forwards on
two streams at once and checks each against its eager result.
"""
import pytest
import torch

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


def eager(d, w, dd):
    out, hT = gla.chunk_fwd(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], chunk=128)
    grads = gla.chunk_bwd(d["q"], d["k"], d["v"], d["dout"], d["log_decay"], d["h0"], d["dhT"], chunk=128)
    st = dd["state"].clone()
    o = gla.decode_step(dd["q"], dd["k"], dd["v"], dd["log_decay"], st)
    torch.cuda.synchronize()
    return [out, hT, *grads, o, st]


@pytest.mark.parametrize("B_,T", [(2, 640), (1, 4096)])  # whole-chain schedule; segmented (few long chains)
def test_graph_replay_matches_eager(B_, T):
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=B_, T=T, H=4, h0_std=0.02)
    wd = I.scaled(I.WORKLOADS["decode"], B=16)
    bufs = I.make_backward(w, device="cuda", seed=1)
    dbufs = I.make_decode(wd, device="cuda", seed=1)
    state = dbufs["state"].clone()
    out = torch.empty(bufs["q"].shape[:3] + (w.dv,), dtype=torch.bfloat16, device="cuda")
    hT = torch.empty(B_, w.H, w.dk, w.dv, device="cuda")
    dq, dk, dv = (torch.empty_like(bufs[k]) for k in ("q", "k", "v"))
    dh0 = torch.empty_like(hT)
    dout_dec = torch.empty(16, wd.H, wd.dv, dtype=torch.bfloat16, device="cuda")

    def step(stream=None):
        gla.gla_chunk_fwd(bufs["q"], bufs["k"], bufs["v"], bufs["log_decay"], bufs["h0"], out, hT, 128, None, stream)
        gla.gla_chunk_bwd(bufs["q"], bufs["k"], bufs["v"], bufs["dout"], bufs["log_decay"], bufs["h0"], bufs["dhT"],
                          dq, dk, dv, dh0, 128, None, stream)
        gla.gla_decode_step(dbufs["q"], dbufs["k"], dbufs["v"], dbufs["log_decay"], state, dout_dec, stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s)  # warm-up outside the capture (first-call lookups)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (5, 6):
        d = I.make_backward(w, device="cuda", seed=seed)
        dd = I.make_decode(wd, device="cuda", seed=seed)
        for k in ("q", "k", "v", "dout", "h0", "dhT"):
            bufs[k].copy_(d[k])
        for k in ("q", "k", "v"):
            dbufs[k].copy_(dd[k])
        state.copy_(dd["state"])
        graph.replay()
        torch.cuda.synchronize()
        assert gla.gla_last_device_status() == 0
        ref = eager(d, w, dd)
        got = [out, hT, dq, dk, dv, dh0, dout_dec, state]
        for name, g, r in zip(("out", "hT", "dq", "dk", "dv", "dh0", "decode out", "decode state"), got, ref):
            assert torch.equal(g, r), f"{name} differs after replay (seed {seed})"


def test_two_streams_at_once():
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=4, T=1024, H=8, h0_std=0.02)
    ds = [I.make_prefill(w, device="cuda", seed=s) for s in (11, 12)]
    refs = [gla.chunk_fwd(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], chunk=128) for d in ds]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for d, st in zip(ds, streams):
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            outs.append(gla.chunk_fwd(d["q"], d["k"], d["v"], d["log_decay"], d["h0"], chunk=128, stream=st))
    torch.cuda.synchronize()
    for (o, h), (ro, rh) in zip(outs, refs):
        assert torch.equal(o, ro) and torch.equal(h, rh)


def test_saved_states_training_step_in_a_graph():
    """gla_chunk_fwd_save + gla_chunk_bwd_saved captured once and replayed with new inputs: bit-identical
    to eager calls (the backward's stream-ordered scratch becomes a graph memory node)."""
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=2, T=640, H=4, h0_std=0.02)
    bufs = I.make_backward(w, device="cuda", seed=3)
    out = torch.empty(bufs["q"].shape[:3] + (w.dv,), dtype=torch.bfloat16, device="cuda")
    hT = torch.empty(2, w.H, w.dk, w.dv, device="cuda")
    img = gla.state_images(bufs["q"], bufs["v"])
    dq, dk, dv = (torch.empty_like(bufs[k]) for k in ("q", "k", "v"))
    dh0 = torch.empty_like(hT)

    def step(b, o, h, im, gq, gk, gv, g0):
        gla.gla_chunk_fwd_save(b["q"], b["k"], b["v"], b["log_decay"], b["h0"], o, h, im, 128)
        gla.gla_chunk_bwd_saved(b["q"], b["k"], b["v"], b["dout"], b["log_decay"], b["h0"], b["dhT"], im,
                                gq, gk, gv, g0, 128)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(bufs, out, hT, img, dq, dk, dv, dh0)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(bufs, out, hT, img, dq, dk, dv, dh0)
    for seed in (8, 9):
        d = I.make_backward(w, device="cuda", seed=seed)
        for k in ("q", "k", "v", "dout", "h0", "dhT"):
            bufs[k].copy_(d[k])
        graph.replay()
        torch.cuda.synchronize()
        assert gla.gla_last_device_status() == 0
        ref = [torch.empty_like(t) for t in (out, hT, dq, dk, dv, dh0)]
        img2 = gla.state_images(d["q"], d["v"])
        step(d, ref[0], ref[1], img2, ref[2], ref[3], ref[4], ref[5])
        torch.cuda.synchronize()
        for name, g, r in zip(("out", "hT", "dq", "dk", "dv", "dh0"), (out, hT, dq, dk, dv, dh0), ref):
            assert torch.equal(g, r), f"{name} differs after replay (seed {seed})"


@pytest.mark.parametrize("T", [640, 4096])  # whole chains; segmented (one long sequence per head)
def test_gated_forward_and_layer_decode_in_a_graph(T):
    """The gated forward and a multi-layer decode step captured in one graph replay bit-identically to
    eager calls, also after new inputs are copied into the captured buffers."""
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=1 if T == 4096 else 2, T=T, H=4, h0_std=0.02)
    L, N, nslots = 3, 8, 16

    def inputs(seed):
        d = I.make_prefill(w, device="cuda", seed=seed)
        gen = torch.Generator().manual_seed(seed)
        dec = {"q": (torch.randn(L, N, 4, 96, generator=gen) / 96 ** 0.5).to(torch.bfloat16).cuda(),
               "k": (torch.randn(L, N, 4, 96, generator=gen) / 96 ** 0.5).to(torch.bfloat16).cuda(),
               "v": torch.randn(L, N, 4, 192, generator=gen).to(torch.bfloat16).cuda(),
               "pool": (torch.randn(nslots, L, 4, 96, 192, generator=gen) * 0.02).cuda(),
               "slots": torch.randperm(nslots, generator=gen)[:N].to(torch.int32).cuda()}
        g = I.make_gate(d["q"].shape[:3] + (192,), device="cuda", seed=seed)
        return d, dec, g

    ld_dec = torch.stack([I.log_decays(4)] * L).cuda()
    d, dec, g = inputs(41)
    out = torch.empty(d["q"].shape[:3] + (192,), dtype=torch.bfloat16, device="cuda")
    hT = torch.empty(d["q"].shape[0], 4, 96, 192, device="cuda")
    dout = torch.empty(L, N, 4, 192, dtype=torch.bfloat16, device="cuda")
    pool = dec["pool"].clone()

    def step(s=None):
        gla.gla_chunk_fwd_gated(d["q"], d["k"], d["v"], g, d["log_decay"], d["h0"], out, hT, 128, stream=s)
        gla.gla_decode_step_layers(dec["q"], dec["k"], dec["v"], ld_dec, pool, dec["slots"], dout, stream=s)

    def eager_results():
        pool.copy_(dec["pool"])
        step()
        torch.cuda.synchronize()
        return out.clone(), hT.clone(), dout.clone(), pool.clone()

    want = eager_results()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    pool.copy_(dec["pool"])
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=s):
        step(s)
    for round_ in range(2):
        if round_ == 1:  # new inputs into the captured buffers
            d2, dec2, g2 = inputs(42)
            for key in ("q", "k", "v"):
                d[key].copy_(d2[key])
                dec[key].copy_(dec2[key])
            g.copy_(g2)
            dec["pool"].copy_(dec2["pool"])
            dec["slots"].copy_(dec2["slots"])
            if d["h0"] is not None:
                d["h0"].copy_(d2["h0"])
            want = eager_results()
        pool.copy_(dec["pool"])
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        got = (out, hT, dout, pool)
        for a, b in zip(got, want):
            assert torch.equal(a, b)
    assert gla.gla_last_device_status() == 0
