"""GPU parity of the multi-layer decode step (gla_decode_step_layers) against the fp64 reference.

Pages hold every layer of a sequence ([nslots, page_layers, H, dk, dv]); one launch updates layers
layer0 .. layer0 + L - 1 of the pages the batch rows name (page "线性注意力模型如何实现固定推理状态",
section "Trainium2 上的推理优化": one fixed state page per sequence).  Each (layer, row) must match one
reference decode step of that layer of that page with that layer's decays; the other layers of every
page and the pages not named stay bit-identical; padding rows write zeros.
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


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build_library()
    gla.load()
    torch.cuda.set_device(0)
    yield
    assert gla.gla_last_device_status() == 0


def make_case(L, N, nslots, page_layers, seed, pad_rows=(), H=4, dk=96, dv=192):
    gen = torch.Generator().manual_seed(seed)
    s = 1.0 / np.sqrt(dk)
    q = (torch.randn(L, N, H, dk, generator=gen) * s).to(torch.bfloat16).cuda()
    k = (torch.randn(L, N, H, dk, generator=gen) * s).to(torch.bfloat16).cuda()
    v = torch.randn(L, N, H, dv, generator=gen).to(torch.bfloat16).cuda()
    ld = torch.stack([I.log_decays(H) * (1.0 + 0.5 * l) for l in range(L)]).cuda()
    pool = (torch.randn(nslots, page_layers, H, dk, dv, generator=gen) * 0.02).cuda()
    slots = torch.randperm(nslots, generator=gen)[:N].to(torch.int32)
    for r in pad_rows:
        slots[r] = -1
    return q, k, v, ld, pool, slots.cuda()


def reference(q, k, v, ld, pool0, slots, layer0, g=None, kind=0):
    """Per layer and live row: one oracle decode step of that page's layer (and the oracle's gate)."""
    sl = slots.cpu().numpy()
    live = np.nonzero(sl >= 0)[0]
    outs, states = [], []
    for l in range(q.shape[0]):
        pages = pool0[torch.as_tensor(sl[live]).long().cuda(), layer0 + l]
        o, s = oracle.decode_step(q[l, live], k[l, live], v[l, live], ld[l], pages)
        if g is not None:
            o = oracle.output_gate(o, g[l, live], kind)
        outs.append(o)
        states.append(s)
    return live, np.stack(outs), np.stack(states)


@pytest.mark.parametrize("gated", [False, True])
def test_layers_of_pages(gated):
    L, N, nslots, page_layers, layer0 = 4, 20, 48, 6, 1
    q, k, v, ld, pool, slots = make_case(L, N, nslots, page_layers, seed=31, pad_rows=(2, 11))
    g = I.make_gate((L, N, 4, 192), device="cuda", seed=31) if gated else None
    pool0 = pool.clone()
    out = torch.empty(L, N, 4, 192, dtype=torch.bfloat16, device="cuda")
    gla.gla_decode_step_layers(q, k, v, ld, pool, slots, out, layer0=layer0, g=g, gate_kind=gla.GATE_SILU)
    torch.cuda.synchronize()
    live, o_ref, s_ref = reference(q, k, v, ld, pool0, slots, layer0, g, gla.GATE_SILU)
    assert oracle.rel_err(out[:, live].float().cpu().numpy(), o_ref) <= TOL
    sl = torch.as_tensor(slots.cpu().numpy()[live]).long().cuda()
    got = torch.stack([pool[sl, layer0 + l] for l in range(L)])
    assert oracle.rel_err(got.cpu().numpy(), s_ref) <= 1e-5
    # layers outside [layer0, layer0 + L) of every page, and pages no row names, are untouched
    untouched = torch.ones(nslots, page_layers, dtype=torch.bool)
    for p in slots.cpu().tolist():
        if p >= 0:
            untouched[p, layer0:layer0 + L] = False
    assert torch.equal(pool[untouched.cuda()], pool0[untouched.cuda()])
    assert torch.count_nonzero(out[:, [2, 11]]).item() == 0


def test_one_launch_equals_one_call_per_layer():
    """L layers in one launch give bit-for-bit what L single-layer calls (L = 1, layer0 = l) give."""
    L, N, nslots, page_layers = 3, 16, 32, 3
    q, k, v, ld, pool, slots = make_case(L, N, nslots, page_layers, seed=32, pad_rows=(5,))
    pool_a, pool_b = pool.clone(), pool.clone()
    out_a = torch.empty(L, N, 4, 192, dtype=torch.bfloat16, device="cuda")
    out_b = torch.empty_like(out_a)
    gla.gla_decode_step_layers(q, k, v, ld, pool_a, slots, out_a)
    for l in range(L):
        gla.gla_decode_step_layers(q[l:l + 1].contiguous(), k[l:l + 1].contiguous(), v[l:l + 1].contiguous(),
                                   ld[l:l + 1].contiguous(), pool_b, slots, out_b[l:l + 1], layer0=l)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    assert torch.equal(pool_a, pool_b)


def test_single_layer_pages_match_the_paged_step():
    """page_layers = 1, L = 1 is the paged decode step."""
    N, nslots = 24, 40
    q, k, v, ld, pool, slots = make_case(1, N, nslots, 1, seed=33, pad_rows=(0,))
    pool_b = pool[:, 0].clone()
    out_a = torch.empty(1, N, 4, 192, dtype=torch.bfloat16, device="cuda")
    out_b = torch.empty(N, 4, 192, dtype=torch.bfloat16, device="cuda")
    gla.gla_decode_step_layers(q, k, v, ld, pool, slots, out_a)
    gla.gla_decode_step_paged(q[0], k[0], v[0], ld[0].contiguous(), pool_b, slots, out_b)
    torch.cuda.synchronize()
    assert torch.equal(out_a[0], out_b)
    assert torch.equal(pool[:, 0], pool_b)


def test_layer_range_is_checked():
    q, k, v, ld, pool, slots = make_case(2, 4, 8, 2, seed=34)
    out = torch.empty(2, 4, 4, 192, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gla.GLAError):
        gla.gla_decode_step_layers(q, k, v, ld, pool, slots, out, layer0=1)  # layers 1, 2 of 2-layer pages


def test_layers_bench_configuration_sampled_layers():
    """The bench's multi-layer leg: 128 sequences whose pages hold all 24 layers (H16, 96 x 192), one launch
    for every layer; three layers of every sequence are checked against the reference step, and the whole
    pool against one call per layer (bit for bit)."""
    L, N, H = 24, 128, 16
    gen = torch.Generator().manual_seed(13)
    s = 1.0 / np.sqrt(96)
    q = (torch.randn(L, N, H, 96, generator=gen) * s).to(torch.bfloat16).cuda()
    k = (torch.randn(L, N, H, 96, generator=gen) * s).to(torch.bfloat16).cuda()
    v = torch.randn(L, N, H, 192, generator=gen).to(torch.bfloat16).cuda()
    ld = torch.stack([I.log_decays(H)] * L).cuda()
    pool = (torch.randn(N, L, H, 96, 192, generator=gen) * 0.02).cuda()
    slots = torch.randperm(N, generator=gen).to(torch.int32).cuda()
    pool_b = pool.clone()
    out = torch.empty(L, N, H, 192, dtype=torch.bfloat16, device="cuda")
    out_b = torch.empty_like(out)
    sampled = (0, 11, 23)
    pages0 = {l: pool[slots.long(), l].cpu() for l in sampled}
    gla.gla_decode_step_layers(q, k, v, ld, pool, slots, out)
    for l in range(L):
        gla.gla_decode_step_layers(q[l:l + 1].contiguous(), k[l:l + 1].contiguous(), v[l:l + 1].contiguous(),
                                   ld[l:l + 1].contiguous(), pool_b, slots, out_b[l:l + 1], layer0=l)
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    assert torch.equal(out, out_b) and torch.equal(pool, pool_b)
    for l in sampled:
        o_ref, s_ref = oracle.decode_step(q[l], k[l], v[l], ld[l], pages0[l])
        assert oracle.rel_err(out[l].float().cpu().numpy(), o_ref) <= TOL
        assert oracle.rel_err(pool[slots.long(), l].cpu().numpy(), s_ref) <= 1e-5
