"""fp64 CPU reference ("oracle") for Simple Gated Linear Attention.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
benchmark's CPU-baseline leg may import this package.  The CUDA library never
imports, links or falls back to it, and the two share no code: the arithmetic
lives in ``gla_oracle.c`` (plain C, fp64), compiled here with gcc.

Citation key: [L3B] is the page "线性注意力模型如何实现固定推理状态" (Beyond
the KV cache: training and serving i14's Laplace 3B linear attention model on
AWS Trainium2); its section "i14 与 Laplace 3B 架构" (GLA mixer) defines the
recurrence and read-out, and section "挑战 1" (Figure 3) the chunked form.

Every function takes numpy arrays shaped like the CUDA entry points:
  q, k: [B, T, H, dk]; v: [B, T, H, dv]; log_decay: [H]; h0/hT: [B, H, dk, dv]
or, for a packed ragged batch, q/k/v of shape [1, total, H, .] together with
``cu_seqlens`` ([N+1], int) and h0/hT of shape [N, H, dk, dv].  Inputs are
converted to float32 (exact for bf16 and fp32 data); log_decay to float64
(exact for an fp32 value); outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libgla_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gla_oracle.c into a shared library (gcc, portable flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            common = [P, P, P, P, P, P, P, P, P, I, I, I, I]
            for name in ("gla_oracle_recurrent", "gla_oracle_quadratic"):
                fn = getattr(lib, name)
                fn.argtypes = common + [P, I, I]
                fn.restype = I
            lib.gla_oracle_chunked.argtypes = common + [I, P, I, I]
            lib.gla_oracle_chunked.restype = I
            lib.gla_oracle_decode_step.argtypes = [P, P, P, P, P, P, I, I, I, I, I]
            lib.gla_oracle_decode_step.restype = I
            lib.gla_oracle_backward.argtypes = [P] * 13 + [I, I, I, I, P, I, I]
            lib.gla_oracle_backward.restype = I
            lib.gla_oracle_conv1d_silu.argtypes = [P] * 8 + [I, I]
            lib.gla_oracle_conv1d_silu.restype = I
            lib.gla_oracle_output_gate.argtypes = [P, P, I, P, ctypes.c_int64]
            lib.gla_oracle_output_gate.restype = I
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _f32(x):
    if hasattr(x, "detach"):  # torch tensor (any dtype): exact widening to float32
        x = x.detach().cpu().float().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _prepare(q, k, v, log_decay, h0, cu_seqlens):
    q, k, v = _f32(q), _f32(k), _f32(v)
    if q.ndim != 4 or k.shape != q.shape or v.shape[:3] != q.shape[:3]:
        raise ValueError("q, k must be [B, T, H, dk] and v [B, T, H, dv]")
    B, T, H, dk = q.shape
    dv = v.shape[3]
    ld = _f64(log_decay).reshape(-1)
    if ld.shape[0] != H:
        raise ValueError("log_decay must have H entries")
    if cu_seqlens is None:
        starts = np.arange(B, dtype=np.int64) * T
        lens = np.full(B, T, dtype=np.int64)
    else:
        if B != 1:
            raise ValueError("a packed batch has leading dimension 1")
        cu = np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64)
        if cu[0] != 0 or np.any(np.diff(cu) < 0) or cu[-1] > T:
            raise ValueError("cu_seqlens must start at 0, be non-decreasing and end within T")
        starts = cu[:-1].copy()
        lens = np.diff(cu)
    nseq = starts.shape[0]
    if h0 is not None:
        h0 = _f64(h0)
        if h0.shape != (nseq, H, dk, dv):
            raise ValueError(f"h0 must be {(nseq, H, dk, dv)}")
    return q, k, v, ld, h0, starts, lens, nseq, (B, T, H, dk, dv)


def _units_arr(units):
    if units is None:
        return None, 0
    u = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
    return u, u.shape[0]


def _run(form, q, k, v, log_decay, h0=None, cu_seqlens=None, units=None, chunk=0, nthreads=None):
    q, k, v, ld, h0, starts, lens, nseq, (B, T, H, dk, dv) = _prepare(q, k, v, log_decay, h0, cu_seqlens)
    o = np.zeros((B, T, H, dv), dtype=np.float64)
    hT = np.zeros((nseq, H, dk, dv), dtype=np.float64)
    u, nu = _units_arr(units)
    nt = default_threads() if nthreads is None else int(nthreads)
    lib = _load()
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(ld), _ptr(h0), _ptr(o), _ptr(hT), _ptr(starts), _ptr(lens),
            nseq, H, dk, dv]
    if form == "recurrent":
        rc = lib.gla_oracle_recurrent(*args, _ptr(u), nu, nt)
    elif form == "quadratic":
        rc = lib.gla_oracle_quadratic(*args, _ptr(u), nu, nt)
    else:
        rc = lib.gla_oracle_chunked(*args, int(chunk), _ptr(u), nu, nt)
    if rc != 0:
        raise ValueError(f"oracle ({form}) rejected its arguments")
    return o, hT


def recurrent(q, k, v, log_decay, h0=None, cu_seqlens=None, units=None, nthreads=None):
    """Token-by-token recurrence S_t = lam S_{t-1} + k_t^T v_t, o_t = q_t S_t ([L3B] GLA mixer).

    Returns (o [B,T,H,dv] float64, hT [nseq,H,dk,dv] float64)."""
    return _run("recurrent", q, k, v, log_decay, h0, cu_seqlens, units, nthreads=nthreads)


def quadratic(q, k, v, log_decay, h0=None, cu_seqlens=None, units=None, nthreads=None):
    """Unrolled attention form O = ((Q K^T) .* D) V + diag(lam^(t+1)) Q h0 (pins the recurrence)."""
    return _run("quadratic", q, k, v, log_decay, h0, cu_seqlens, units, nthreads=nthreads)


def chunked(q, k, v, log_decay, chunk, h0=None, cu_seqlens=None, units=None, nthreads=None):
    """Chunkwise form with chunk length ``chunk`` ([L3B] §挑战 1, Figure 3), fp64."""
    return _run("chunked", q, k, v, log_decay, h0, cu_seqlens, units, chunk=chunk, nthreads=nthreads)


def backward(q, k, v, dout, log_decay, h0=None, dhT=None, cu_seqlens=None, units=None, nthreads=None):
    """Gradients of L = sum(dout * o) + sum(dhT * hT) through the recurrence ([L3B] §挑战 3).

    Reverse-mode chain rule of S_t = lam S_{t-1} + k_t^T v_t, o_t = q_t S_t, one token at a
    time (see ``gla_oracle.c``).  dout has the shape of o; dhT (optional) that of hT.  Returns
    (dq, dk, dv, dh0) in float64 with the shapes of q, k, v and h0 ([nseq, H, dk, dv])."""
    q, k, v, ld, h0, starts, lens, nseq, (B, T, H, dk, dv) = _prepare(q, k, v, log_decay, h0, cu_seqlens)
    do = _f32(dout)
    if do.shape != (B, T, H, dv):
        raise ValueError("dout must have the shape of o")
    if dhT is not None:
        dhT = _f64(dhT)
        if dhT.shape != (nseq, H, dk, dv):
            raise ValueError(f"dhT must be {(nseq, H, dk, dv)}")
    dq = np.zeros((B, T, H, dk), dtype=np.float64)
    dkk = np.zeros((B, T, H, dk), dtype=np.float64)
    dvv = np.zeros((B, T, H, dv), dtype=np.float64)
    dh0 = np.zeros((nseq, H, dk, dv), dtype=np.float64)
    u, nu = _units_arr(units)
    nt = default_threads() if nthreads is None else int(nthreads)
    rc = _load().gla_oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(ld), _ptr(h0), _ptr(dhT),
                                     _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dh0), _ptr(starts), _ptr(lens),
                                     nseq, H, dk, dv, _ptr(u), nu, nt)
    if rc != 0:
        raise ValueError("oracle backward rejected its arguments")
    return dq, dkk, dvv, dh0


def conv1d_silu(x, weight, bias=None, state=None, cu_seqlens=None):
    """Causal depthwise Conv1d (width 4) + SiLU per channel ([L3B] "i14 与 Laplace 3B 架构").

    x: [B, T, D] (or packed [1, T, D] with ``cu_seqlens``); weight [D, 4] (weight[:, 3] meets the
    current token); bias [D] or None; state [nseq, D, 3] (the three inputs before each sequence,
    oldest first) or None.  Returns (y [B, T, D] float64, state_out [nseq, D, 3] float64)."""
    x = _f32(x)
    if x.ndim != 3:
        raise ValueError("x must be [B, T, D]")
    B, T, D = x.shape
    w = _f64(weight)
    if w.shape != (D, 4):
        raise ValueError("weight must be [D, 4]")
    b = None if bias is None else _f64(bias).reshape(D)
    if cu_seqlens is None:
        starts = np.arange(B, dtype=np.int64) * T
        lens = np.full(B, T, dtype=np.int64)
    else:
        if B != 1:
            raise ValueError("a packed batch has leading dimension 1")
        cu = np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64)
        starts, lens = cu[:-1].copy(), np.diff(cu)
    nseq = starts.shape[0]
    st = None if state is None else _f64(state)
    if st is not None and st.shape != (nseq, D, 3):
        raise ValueError(f"state must be {(nseq, D, 3)}")
    y = np.zeros((B, T, D), dtype=np.float64)
    so = np.zeros((nseq, D, 3), dtype=np.float64)
    rc = _load().gla_oracle_conv1d_silu(_ptr(x), _ptr(w), _ptr(b), _ptr(st), _ptr(so), _ptr(y), _ptr(starts),
                                        _ptr(lens), nseq, D)
    if rc != 0:
        raise ValueError("oracle conv1d rejected its arguments")
    return y, so


def decode_step(q, k, v, log_decay, state, nthreads=None):
    """One decode step for [N, H] chains: state <- lam state + k^T v; o = q state.

    q, k: [N, H, dk]; v: [N, H, dv]; state: [N, H, dk, dv].  Returns
    (o [N,H,dv] float64, new_state float64); the input ``state`` is not modified."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    N, H, dk = q.shape
    dv = v.shape[2]
    ld = _f64(log_decay).reshape(-1)
    st = _f64(state).copy()
    if st.shape != (N, H, dk, dv) or ld.shape[0] != H or k.shape != q.shape or v.shape[:2] != (N, H):
        raise ValueError("bad decode shapes")
    o = np.zeros((N, H, dv), dtype=np.float64)
    nt = default_threads() if nthreads is None else int(nthreads)
    rc = _load().gla_oracle_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(ld), _ptr(st), _ptr(o),
                                        N, H, dk, dv, nt)
    if rc != 0:
        raise ValueError("oracle decode rejected its arguments")
    return o, st


GATE_SILU, GATE_SIGMOID = 0, 1


def output_gate(o, g, kind=GATE_SILU):
    """The mixer output times a function of the gate g_t ([L3B] "i14 与 Laplace 3B 架构", QKVG
    projection: the gate acts after the mixer).  kind 0: o * g / (1 + exp(-g)) (SiLU), kind 1:
    o / (1 + exp(-g)) (sigmoid).  o and g have the same shape; returns float64."""
    o = _f64(o)
    g = _f32(g)
    if o.shape != g.shape:
        raise ValueError("o and g must have the same shape")
    out = np.empty_like(o)
    rc = _load().gla_oracle_output_gate(_ptr(o), _ptr(g), int(kind), _ptr(out), o.size)
    if rc != 0:
        raise ValueError("oracle output gate rejected its arguments")
    return out


def rel_err(got, ref) -> float:
    """max|got - ref| / max|ref| over the whole tensor (0 when both are zero)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    if den == 0.0:
        return num
    return num / den
