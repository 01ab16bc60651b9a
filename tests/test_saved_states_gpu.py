"""Training with saved states: gla_chunk_fwd_save writes the state before every chunk, and
gla_chunk_bwd_saved consumes it instead of walking the chains forwards again.

Checks: the save variant's out and hT are bit-identical to gla_chunk_fwd's (the images add stores,
not arithmetic); every image is the fp64 recurrence's state at its chunk start (h0 for the first
chunk) within the bf16 bar; the saved backward matches gla_chunk_bwd and the fp64 reference.
Dense with a partial chunk, packed with an empty sequence, and a long sequence that takes the
segmented schedule.
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


CASES = {
    "dense_partial_chunk": dict(B=2, T=300, H=4),
    "packed_with_empty": dict(lengths=[129, 0, 300, 1, 256]),
    "long_segmented": dict(B=1, T=4096, H=3),
}


def setup(name):
    kw = dict(CASES[name])
    lengths = kw.pop("lengths", None)
    w = I.scaled(I.WORKLOADS["ragged" if lengths else "layer_bf16"], h0_std=0.02, **({"H": 3} if lengths else kw))
    d = I.make_backward(w, device="cuda", seed=41, dhT_std=0.02, **({"lengths": lengths} if lengths else {}))
    d["cu_dev"] = None if d["cu_seqlens"] is None else d["cu_seqlens"].cuda()
    return w, d


def unswizzle(raw, dk, dv):
    """[slots, H, dk*dv] image tiles in the kernels' layout -> [slots, H, dk, dv]: dv in 64-column atoms
    of dk rows x 128 bytes; the 16-byte piece p (8 values) of row r sits at position p ^ (r mod 8)."""
    r = np.arange(dk)[:, None]
    j = np.arange(dv)[None, :]
    a, jj = j // 64, j % 64
    idx = a * dk * 64 + r * 64 + (((jj // 8) ^ (r % 8)) * 8) + jj % 8
    return raw[..., idx]


def starts(d):
    cu = d["cu_seqlens"]
    if cu is None:
        B, T = d["q"].shape[:2]
        return [(s, s * T, T) for s in range(B)]
    cu = cu.numpy()
    return [(s, int(cu[s]), int(cu[s + 1] - cu[s])) for s in range(len(cu) - 1)]


@pytest.mark.parametrize("name", list(CASES))
def test_forward_save_and_saved_backward(name):
    w, d = setup(name)
    q, k, v, ld, h0, cu = d["q"], d["k"], d["v"], d["log_decay"], d["h0"], d["cu_dev"]
    nseq = len(starts(d))
    out_a, hT_a = gla.chunk_fwd(q, k, v, ld, h0, chunk=128, cu_seqlens=cu)
    out_b = torch.empty_like(out_a)
    hT_b = torch.empty_like(hT_a)
    img = gla.state_images(q, v, cu)
    img.fill_(float("nan"))
    gla.gla_chunk_fwd_save(q, k, v, ld, h0, out_b, hT_b, img, 128, cu)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(hT_a, hT_b)

    # each image = the state before its chunk: fp64 recurrence over the sequence's prefix
    H, dk, dv = w.H, w.dk, w.dv
    imgs = unswizzle(img.view(-1, H, dk * dv).float().cpu().numpy(), dk, dv)
    for s, start, L in starts(d):
        for c in sorted({0, 1, (L - 1) // 128}):
            if L == 0 or c < 0 or c * 128 >= L:  # an empty sequence has no chunk and no image
                continue
            slot = start // 128 + s + c
            if c == 0:
                ref = np.zeros((H, dk, dv)) if h0 is None else h0[s].double().cpu().numpy()
            else:
                rows = slice(start, start + c * 128)
                qq = q[:, rows] if cu is not None else q[s:s + 1, :c * 128]
                kk = k[:, rows] if cu is not None else k[s:s + 1, :c * 128]
                vv = v[:, rows] if cu is not None else v[s:s + 1, :c * 128]
                _, h_ref = oracle.recurrent(qq, kk, vv, ld, None if h0 is None else h0[s:s + 1])
                ref = h_ref[0]
            assert oracle.rel_err(imgs[slot], ref) <= TOL, (name, s, c)

    dq_a, dk_a, dv_a, dh0_a = gla.chunk_bwd(q, k, v, d["dout"], ld, h0, d["dhT"], chunk=128, cu_seqlens=cu)
    dq_b, dk_b, dv_b = torch.empty_like(dq_a), torch.empty_like(dk_a), torch.empty_like(dv_a)
    dh0_b = torch.empty_like(dh0_a)
    gla.gla_chunk_bwd_saved(q, k, v, d["dout"], ld, h0, d["dhT"], img, dq_b, dk_b, dv_b, dh0_b, 128, cu)
    torch.cuda.synchronize()
    assert gla.gla_last_device_status() == 0
    g_ref = oracle.backward(q, k, v, d["dout"], ld, h0, d["dhT"], cu_seqlens=d["cu_seqlens"])
    for nm, a, b_, r in zip(("dq", "dk", "dv", "dh0"), (dq_a, dk_a, dv_a, dh0_a), (dq_b, dk_b, dv_b, dh0_b), g_ref):
        ga, gb = a.float().cpu().numpy(), b_.float().cpu().numpy()
        assert oracle.rel_err(gb, r) <= TOL, (name, nm)
        assert oracle.rel_err(gb, ga) <= TOL, (name, nm)
    assert nseq >= 1


def test_shapes_outside_the_tensor_core_backward_are_refused():
    """Saved states exist only on the tensor-core kernels: chunk 32 (SIMT) is refused, chunk 64 runs as two
    chunks per 128-row tile and gives exactly the chunk-128 result."""
    w = I.scaled(I.WORKLOADS["layer_bf16"], B=1, T=64, H=2, dk=96, dv=192)
    d = I.make_prefill(w, device="cuda", seed=1)
    out = torch.empty(1, 64, 2, 192, dtype=torch.bfloat16, device="cuda")
    img = gla.state_images(d["q"], d["v"])
    with pytest.raises(gla.GLAError) as e:
        gla.gla_chunk_fwd_save(d["q"], d["k"], d["v"], d["log_decay"], None, out, None, img, 32)
    assert e.value.status == -2  # GLA_ERR_UNSUPPORTED: chunk 32 runs on the SIMT kernels
    out128 = torch.empty_like(out)
    img.zero_()  # slots no chunk starts at are left untouched by both calls
    img128 = torch.zeros_like(img)
    gla.gla_chunk_fwd_save(d["q"], d["k"], d["v"], d["log_decay"], None, out, None, img, 64)
    gla.gla_chunk_fwd_save(d["q"], d["k"], d["v"], d["log_decay"], None, out128, None, img128, 128)
    torch.cuda.synchronize()
    assert torch.equal(out, out128) and torch.equal(img, img128)
