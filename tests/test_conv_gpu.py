"""GPU parity of the causal depthwise Conv1d (width 4) + SiLU against the fp64 reference.

Bar: max|gpu - ref| / max|ref| <= 1e-2 for bf16 outputs, 1e-5 for f32; the conv states (exact copies
of inputs) must match exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_linear_rnn_gb300 import build as B
from gated_linear_rnn_gb300 import gla

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 1e-2, torch.float32: 1e-5}


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build_library()
    gla.load()
    torch.cuda.set_device(0)
    yield
    assert gla.gla_last_device_status() == 0


def make(shape, D, dtype, seed, nseq, bias=True, state=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape + (D,), generator=g).to(dtype)
    w = torch.randn(D, 4, generator=g) * 0.5
    b = torch.randn(D, generator=g) * 0.1 if bias else None
    st = torch.randn(nseq, D, 3, generator=g).to(dtype).float() if state else None  # representable like x
    return x, w, b, st


def run_conv(x, w, b, st, cu=None):
    nseq = x.shape[0] if cu is None else cu.numel() - 1
    y = torch.full_like(x, float("nan")).cuda()
    so = torch.full((nseq, x.shape[2], 3), float("nan"), device="cuda")
    fn = gla.gla_conv1d_silu_f32 if x.dtype == torch.float32 else gla.gla_conv1d_silu
    fn(x.cuda(), w.cuda(), None if b is None else b.cuda(), None if st is None else st.cuda(), so, y,
       None if cu is None else cu.cuda())
    torch.cuda.synchronize()
    return y, so


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T", [1, 2, 5, 16, 37, 100])
def test_conv_dense(dtype, T):
    x, w, b, st = make((3, T), 64, dtype, seed=T, nseq=3)
    y, so = run_conv(x, w, b, st)
    y_ref, so_ref = oracle.conv1d_silu(x, w, b, st)
    assert oracle.rel_err(y.float().cpu().numpy(), y_ref) <= TOL[dtype]
    assert np.array_equal(so.cpu().numpy(), so_ref)


def test_conv_no_bias_no_state():
    x, w, _, _ = make((2, 40), 128, torch.bfloat16, seed=3, nseq=2, bias=False, state=False)
    y, so = run_conv(x, w, None, None)
    y_ref, so_ref = oracle.conv1d_silu(x, w)
    assert oracle.rel_err(y.float().cpu().numpy(), y_ref) <= 1e-2
    assert np.array_equal(so.cpu().numpy(), so_ref)


def test_conv_ragged_with_empty_sequences_and_tail_rows():
    lens = [5, 0, 17, 1, 40, 0, 2, 33]
    total = sum(lens)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    x, w, b, st = make((1, total + 7), 256, torch.bfloat16, seed=4, nseq=len(lens))  # 7 rows past the last
    y, so = run_conv(x, w, b, st, cu)
    y_ref, so_ref = oracle.conv1d_silu(x[:, :total], w, b, st, cu_seqlens=cu.numpy())
    yc = y.float().cpu().numpy()
    assert oracle.rel_err(yc[:, :total], y_ref) <= 1e-2
    assert np.isnan(yc[:, total:]).all()  # rows past cu_seqlens[N] are not written
    assert np.array_equal(so.cpu().numpy(), so_ref)


@pytest.mark.parametrize("N,D", [(1, 3072), (7, 3072), (151, 264), (1280, 3072), (3001, 3072)])
def test_conv_step_batch_sizes(N, D):
    """The step over batches that the launch splits into different numbers of sequences per block (one
    block of one sequence up to many sequences a block): every sequence's output and state updated once."""
    x, w, b, st = make((N, 1), D, torch.bfloat16, seed=N, nseq=N)
    state = st.clone().cuda()
    y = torch.empty(N, D, dtype=torch.bfloat16, device="cuda")
    gla.gla_conv1d_silu_step(x[:, 0].contiguous().cuda(), w.cuda(), b.cuda(), state, y)
    torch.cuda.synchronize()
    y_ref, so_ref = oracle.conv1d_silu(x, w, b, st)
    assert oracle.rel_err(y.float().cpu().numpy(), y_ref[:, 0]) <= 1e-2
    assert np.array_equal(state.cpu().numpy(), so_ref)


def test_conv_step_equals_one_token():
    N, D = 50, 3072
    x, w, b, st = make((N, 1), D, torch.bfloat16, seed=5, nseq=N)
    state = st.clone().cuda()
    y = torch.empty(N, D, dtype=torch.bfloat16, device="cuda")
    gla.gla_conv1d_silu_step(x[:, 0].contiguous().cuda(), w.cuda(), b.cuda(), state, y)
    torch.cuda.synchronize()
    y_ref, so_ref = oracle.conv1d_silu(x, w, b, st)
    assert oracle.rel_err(y.float().cpu().numpy(), y_ref[:, 0]) <= 1e-2
    assert np.array_equal(state.cpu().numpy(), so_ref)


def test_conv_layer_shape():
    """The layer's residual-stream shape: B8 T2048 D3072 bf16, bias, no incoming state."""
    x, w, b, _ = make((8, 2048), 3072, torch.bfloat16, seed=6, nseq=8, state=False)
    y, so = run_conv(x, w, b, None)
    y_ref, so_ref = oracle.conv1d_silu(x, w, b)
    assert oracle.rel_err(y.float().cpu().numpy(), y_ref) <= 1e-2
    assert np.array_equal(so.cpu().numpy(), so_ref)


@pytest.mark.parametrize("D", [264, 520, 2056])
def test_conv_partial_channel_slab(D):
    """Channel counts that leave a partial last 256-channel slab (the TMA box reaches past D)."""
    x, w, b, st = make((2, 150), D, torch.bfloat16, seed=D, nseq=2)
    y, so = run_conv(x, w, b, st)
    y_ref, so_ref = oracle.conv1d_silu(x, w, b, st)
    assert oracle.rel_err(y.float().cpu().numpy(), y_ref) <= 1e-2
    assert np.array_equal(so.cpu().numpy(), so_ref)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_conv_ragged_across_tiles(dtype):
    """Sequences that start and end on either side of 64-row tile and 8-row run boundaries."""
    lens = [64, 1, 63, 130, 3, 8, 0, 200, 7, 61, 2]
    total = sum(lens)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    x, w, b, st = make((1, total), 512, dtype, seed=7, nseq=len(lens))
    y, so = run_conv(x, w, b, st, cu)
    y_ref, so_ref = oracle.conv1d_silu(x, w, b, st, cu_seqlens=cu.numpy())
    assert oracle.rel_err(y.float().cpu().numpy(), y_ref) <= TOL[dtype]
    assert np.array_equal(so.cpu().numpy(), so_ref)


@pytest.mark.parametrize("case", range(24))
def test_conv_seeded_sweep(case):
    """Seeded random shapes: D any multiple of 8 (partial 256-channel slabs), dense or packed with
    empty sequences and rows past the packed total, bf16 or f32, with or without bias and state."""
    rng = np.random.default_rng(5000 + case)
    D = 8 * int(rng.integers(1, 520))
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    cu = None
    if rng.random() < 0.5:
        lens = [int(x) for x in rng.integers(0, 200, int(rng.integers(1, 12)))]
        lens[0] = max(lens[0], 1)
        total = sum(lens)
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
        shape, nseq = (1, total + int(rng.integers(0, 9))), len(lens)
    else:
        shape = (int(rng.integers(1, 4)), int(rng.integers(1, 300)))
        nseq, total = shape[0], shape[1]
    x, w, b, st = make(shape, D, dtype, seed=case, nseq=nseq, bias=rng.random() < 0.7, state=rng.random() < 0.6)
    y, so = run_conv(x, w, b, st, cu)
    yc = y.float().cpu().numpy()
    if cu is None:
        y_ref, so_ref = oracle.conv1d_silu(x, w, b, st)
    else:
        y_ref, so_ref = oracle.conv1d_silu(x[:, :total], w, b, st, cu_seqlens=cu.numpy())
        assert np.isnan(yc[:, total:]).all()  # rows past cu_seqlens[N] are not written
        yc = yc[:, :total]
    assert oracle.rel_err(yc, y_ref) <= TOL[dtype]
    assert np.array_equal(so.cpu().numpy(), so_ref)
