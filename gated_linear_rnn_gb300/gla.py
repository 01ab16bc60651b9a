"""Thin Python binding of libgla.so (argument marshalling only).

The functions named ``gla_*`` mirror the C entry points of include/gla.h one to
one: they take torch tensors that already live on the current CUDA device,
check dtype / shape / contiguity, pass raw pointers and the current stream, and
raise ``GLAError`` on a non-zero status.  ``chunk_fwd`` and ``decode_step`` are
conveniences that allocate the outputs with torch and call those entry points.
Every step of the computation runs in the library's CUDA kernels; when the
library is missing this module raises instead of computing anything itself.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgla.so")

STATUS = {0: "GLA_OK", -1: "GLA_ERR_ARG", -2: "GLA_ERR_UNSUPPORTED", -3: "GLA_ERR_ALIGN", -4: "GLA_ERR_LAUNCH",
          -5: "GLA_ERR_TIMEOUT", -6: "GLA_ERR_NOMEM", -7: "GLA_ERR_DEVICE_ARG", -8: "GLA_ERR_SCRATCH_LIMIT"}

# C signatures (argtypes, restype) of every exported entry point, as declared in include/gla.h
_P, _I = ctypes.c_void_p, ctypes.c_int
SIGNATURES = {
    "gla_chunk_fwd": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "gla_chunk_fwd_gated": ([_P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "gla_decode_step_gated": ([_P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "gla_decode_step_paged_gated": ([_P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _I, _I, _I, _I, _P], _I),
    "gla_decode_step_layers": ([_P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _I, _I, _I, _I, _P], _I),
    "gla_chunk_fwd_noalloc": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "gla_chunk_fwd_host": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P], _I),
    "gla_chunk_fwd_f32": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "gla_chunk_bwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "gla_chunk_bwd_f32": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "gla_state_images_bytes": ([_I, _I, _I, _I, _I, _I], ctypes.c_longlong),
    "gla_chunk_fwd_save": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "gla_chunk_bwd_saved": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "gla_decode_step": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "gla_decode_step_f32": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "gla_decode_step_paged": ([_P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _P], _I),
    "gla_conv1d_silu": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P], _I),
    "gla_conv1d_silu_f32": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P], _I),
    "gla_conv1d_silu_step": ([_P, _P, _P, _P, _P, _I, _I, _P], _I),
    "gla_last_device_status": ([_P], _I),
    "gla_status_str": ([_I], ctypes.c_char_p),
    "gla_chunk_kernel": ([_I, _I, _I, _I, _I], _I),
    "gla_kernel_launches": ([], ctypes.c_uint64),
    "gla_version": ([], _I),
}


class GLAError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({_status_text(status)})")


_lock = threading.Lock()
_lib = None


def load(path: Optional[str] = None):
    """Load libgla.so once (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is missing: build it with gated_linear_rnn_gb300.build.build_library()")
            lib = ctypes.CDLL(p)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _status_text(status: int) -> str:
    try:
        return load().gla_status_str(int(status)).decode()
    except Exception:  # library not loadable: plain name only
        return STATUS.get(status, "unknown")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(t: Optional[torch.Tensor], name: str, dtype, shape=None, allow_none=False):
    if t is None:
        if allow_none:
            return
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _raise(rc: int, what: str):
    if rc != 0:
        raise GLAError(rc, what)


# ---- entry points (same names as the C ABI) ---------------------------------------------------

def _chunk_args(q, k, v, log_decay, h0, out, hT, cu_seqlens, dtype):
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, dk] (packed: [1, T, H, dk])")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    _check(q, "q", dtype)
    _check(k, "k", dtype, (B, T, H, dk))
    _check(v, "v", dtype, (B, T, H, dv))
    _check(out, "out", dtype, (B, T, H, dv))
    _check(log_decay, "log_decay", torch.float32, (H,))
    nseq = B
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("a packed batch has leading dimension 1")
        _check(cu_seqlens, "cu_seqlens", torch.int32)
        nseq = cu_seqlens.numel() - 1
    _check(h0, "h0", torch.float32, (nseq, H, dk, dv), allow_none=True)
    _check(hT, "hT", torch.float32, (nseq, H, dk, dv), allow_none=True)
    return nseq, T, H, dk, dv


def gla_chunk_fwd(q, k, v, log_decay, h0, out, hT, chunk: int, cu_seqlens=None, stream=None) -> None:
    """bf16 chunked forward: writes ``out`` and (if given) ``hT``.  See include/gla.h."""
    nseq, T, H, dk, dv = _chunk_args(q, k, v, log_decay, h0, out, hT, cu_seqlens, torch.bfloat16)
    rc = load().gla_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_decay), _ptr(h0), _ptr(out), _ptr(hT),
                              nseq, T, H, dk, dv, int(chunk), _ptr(cu_seqlens), _stream(stream))
    _raise(rc, "gla_chunk_fwd")


GATE_SILU, GATE_SIGMOID = 0, 1  # gla_gate_kind


def gla_chunk_fwd_gated(q, k, v, g, log_decay, h0, out, hT, chunk: int, cu_seqlens=None, gate_kind: int = GATE_SILU,
                        stream=None) -> None:
    """bf16 chunked forward with the output gate fused into the write of ``out``: out = o * f(g), f = SiLU
    (gate_kind 0) or sigmoid (1); ``g`` has the shape of ``out``.  See include/gla.h."""
    nseq, T, H, dk, dv = _chunk_args(q, k, v, log_decay, h0, out, hT, cu_seqlens, torch.bfloat16)
    _check(g, "g", torch.bfloat16, tuple(out.shape))
    rc = load().gla_chunk_fwd_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g), int(gate_kind), _ptr(log_decay), _ptr(h0),
                                    _ptr(out), _ptr(hT), nseq, T, H, dk, dv, int(chunk), _ptr(cu_seqlens),
                                    _stream(stream))
    _raise(rc, "gla_chunk_fwd_gated")


def gla_chunk_fwd_noalloc(q, k, v, log_decay, h0, out, hT, chunk: int, cu_seqlens=None, stream=None) -> None:
    """As gla_chunk_fwd, but the library allocates nothing: segment states of long sequences go to a
    fixed scratch array in the library image (for callers that may not let a library allocate
    device memory).  Raises GLAError(GLA_ERR_SCRATCH_LIMIT) when a problem needs more than that array."""
    nseq, T, H, dk, dv = _chunk_args(q, k, v, log_decay, h0, out, hT, cu_seqlens, torch.bfloat16)
    rc = load().gla_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_decay), _ptr(h0), _ptr(out), _ptr(hT),
                                      nseq, T, H, dk, dv, int(chunk), _ptr(cu_seqlens), _stream(stream))
    _raise(rc, "gla_chunk_fwd_noalloc")


def gla_chunk_fwd_host(q, k, v, log_decay, h0, out, hT, chunk: int, stream=None) -> None:
    """bf16 chunked forward on HOST tensors (pinned for overlap): copies in, computes and copies out
    in groups of sequences on three streams.  Enqueues and returns; the results are in ``out`` / ``hT``
    once ``stream`` has reached the call.  See include/gla.h."""
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, dk]")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for t, name, dtype, shape in ((q, "q", torch.bfloat16, None), (k, "k", torch.bfloat16, (B, T, H, dk)),
                                  (v, "v", torch.bfloat16, (B, T, H, dv)), (out, "out", torch.bfloat16, (B, T, H, dv)),
                                  (log_decay, "log_decay", torch.float32, (H,)),
                                  (h0, "h0", torch.float32, (B, H, dk, dv)), (hT, "hT", torch.float32, (B, H, dk, dv))):
        if t is None:
            if name in ("h0", "hT"):
                continue
            raise ValueError(f"{name} is required")
        if t.is_cuda:
            raise ValueError(f"{name} must be a host tensor")
        if t.dtype != dtype or not t.is_contiguous() or (shape is not None and tuple(t.shape) != tuple(shape)):
            raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {shape or '[B, T, H, dk]'}")
    rc = load().gla_chunk_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(log_decay), _ptr(h0), _ptr(out), _ptr(hT),
                                   B, T, H, dk, dv, int(chunk), _stream(stream))
    _raise(rc, "gla_chunk_fwd_host")


def gla_chunk_fwd_f32(q, k, v, log_decay, h0, out, hT, chunk: int, cu_seqlens=None, stream=None) -> None:
    """f32 chunked forward (SIMT kernel).  See include/gla.h."""
    nseq, T, H, dk, dv = _chunk_args(q, k, v, log_decay, h0, out, hT, cu_seqlens, torch.float32)
    rc = load().gla_chunk_fwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(log_decay), _ptr(h0), _ptr(out), _ptr(hT),
                                  nseq, T, H, dk, dv, int(chunk), _ptr(cu_seqlens), _stream(stream))
    _raise(rc, "gla_chunk_fwd_f32")


def _bwd_args(q, k, v, dout, log_decay, h0, dhT, dq, dk, dv, dh0, cu_seqlens, dtype):
    nseq, T, H, dk_, dv_ = _chunk_args(q, k, v, log_decay, h0, dout, dhT, cu_seqlens, dtype)
    B = q.shape[0]
    _check(dq, "dq", dtype, (B, T, H, dk_))
    _check(dk, "dk", dtype, (B, T, H, dk_))
    _check(dv, "dv", dtype, (B, T, H, dv_))
    _check(dh0, "dh0", torch.float32, (nseq, H, dk_, dv_), allow_none=True)
    return nseq, T, H, dk_, dv_


def gla_chunk_bwd(q, k, v, dout, log_decay, h0, dhT, dq, dk, dv, dh0, chunk: int, cu_seqlens=None,
                  stream=None) -> None:
    """bf16 backward of the chunked forward: writes dq, dk, dv and (if given) dh0.  See include/gla.h."""
    nseq, T, H, dk_, dv_ = _bwd_args(q, k, v, dout, log_decay, h0, dhT, dq, dk, dv, dh0, cu_seqlens, torch.bfloat16)
    rc = load().gla_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(log_decay), _ptr(h0), _ptr(dhT),
                              _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dh0), nseq, T, H, dk_, dv_, int(chunk),
                              _ptr(cu_seqlens), _stream(stream))
    _raise(rc, "gla_chunk_bwd")


def gla_chunk_bwd_f32(q, k, v, dout, log_decay, h0, dhT, dq, dk, dv, dh0, chunk: int, cu_seqlens=None,
                      stream=None) -> None:
    """f32 backward of the chunked forward (SIMT kernel).  See include/gla.h."""
    nseq, T, H, dk_, dv_ = _bwd_args(q, k, v, dout, log_decay, h0, dhT, dq, dk, dv, dh0, cu_seqlens, torch.float32)
    rc = load().gla_chunk_bwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(log_decay), _ptr(h0), _ptr(dhT),
                                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dh0), nseq, T, H, dk_, dv_, int(chunk),
                                  _ptr(cu_seqlens), _stream(stream))
    _raise(rc, "gla_chunk_bwd_f32")


def gla_state_images_bytes(B: int, T: int, H: int, dk: int, dv: int, packed: bool) -> int:
    """Bytes of the state-image buffer of gla_chunk_fwd_save / gla_chunk_bwd_saved.  See include/gla.h."""
    return int(load().gla_state_images_bytes(int(B), int(T), int(H), int(dk), int(dv), int(bool(packed))))


def state_images(q, v, cu_seqlens=None) -> torch.Tensor:
    """An uninitialised device buffer for the state images of this batch (bf16, flat)."""
    B, T, H, dk = q.shape
    nseq = B if cu_seqlens is None else cu_seqlens.numel() - 1
    n = gla_state_images_bytes(nseq, T, H, dk, v.shape[-1], cu_seqlens is not None)
    return torch.empty(n // 2, dtype=torch.bfloat16, device=q.device)


def _check_images(images, q, v, cu_seqlens):
    B, T, H, dk = q.shape
    nseq = B if cu_seqlens is None else cu_seqlens.numel() - 1
    need = gla_state_images_bytes(nseq, T, H, dk, v.shape[-1], cu_seqlens is not None)
    _check(images, "state_images", torch.bfloat16)
    if images.numel() * 2 < need:
        raise ValueError(f"state_images holds {images.numel() * 2} bytes, needs {need}")


def gla_chunk_fwd_save(q, k, v, log_decay, h0, out, hT, state_images, chunk: int, cu_seqlens=None,
                       stream=None) -> None:
    """gla_chunk_fwd that also writes the state before every chunk to ``state_images`` (for
    gla_chunk_bwd_saved).  See include/gla.h."""
    nseq, T, H, dk, dv = _chunk_args(q, k, v, log_decay, h0, out, hT, cu_seqlens, torch.bfloat16)
    _check_images(state_images, q, v, cu_seqlens)
    rc = load().gla_chunk_fwd_save(_ptr(q), _ptr(k), _ptr(v), _ptr(log_decay), _ptr(h0), _ptr(out), _ptr(hT),
                                   _ptr(state_images), nseq, T, H, dk, dv, int(chunk), _ptr(cu_seqlens),
                                   _stream(stream))
    _raise(rc, "gla_chunk_fwd_save")


def gla_chunk_bwd_saved(q, k, v, dout, log_decay, h0, dhT, state_images, dq, dk, dv, dh0, chunk: int,
                        cu_seqlens=None, stream=None) -> None:
    """gla_chunk_bwd with the states saved by gla_chunk_fwd_save.  See include/gla.h."""
    nseq, T, H, dk_, dv_ = _bwd_args(q, k, v, dout, log_decay, h0, dhT, dq, dk, dv, dh0, cu_seqlens, torch.bfloat16)
    _check_images(state_images, q, v, cu_seqlens)
    rc = load().gla_chunk_bwd_saved(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(log_decay), _ptr(h0), _ptr(dhT),
                                    _ptr(state_images), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dh0), nseq, T, H, dk_, dv_,
                                    int(chunk), _ptr(cu_seqlens), _stream(stream))
    _raise(rc, "gla_chunk_bwd_saved")


def _decode_args(q, k, v, log_decay, state, out, dtype):
    if q.dim() != 3:
        raise ValueError("q must be [N, H, dk]")
    N, H, dk = q.shape
    dv = v.shape[-1]
    _check(q, "q", dtype)
    _check(k, "k", dtype, (N, H, dk))
    _check(v, "v", dtype, (N, H, dv))
    _check(out, "out", dtype, (N, H, dv))
    _check(log_decay, "log_decay", torch.float32, (H,))
    _check(state, "state_inout", torch.float32, (N, H, dk, dv))
    return N, H, dk, dv


def gla_decode_step(q, k, v, log_decay, state_inout, out, stream=None) -> None:
    """bf16 decode step: updates ``state_inout`` in place and writes ``out``."""
    N, H, dk, dv = _decode_args(q, k, v, log_decay, state_inout, out, torch.bfloat16)
    rc = load().gla_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(log_decay), _ptr(state_inout), _ptr(out),
                                N, H, dk, dv, _stream(stream))
    _raise(rc, "gla_decode_step")


def gla_decode_step_f32(q, k, v, log_decay, state_inout, out, stream=None) -> None:
    N, H, dk, dv = _decode_args(q, k, v, log_decay, state_inout, out, torch.float32)
    rc = load().gla_decode_step_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(log_decay), _ptr(state_inout), _ptr(out),
                                    N, H, dk, dv, _stream(stream))
    _raise(rc, "gla_decode_step_f32")


def gla_decode_step_paged(q, k, v, log_decay, state_pool, slots, out, stream=None) -> None:
    """bf16 decode step on a page pool: row n updates page slots[n] (negative: padding row, zero out)."""
    if q.dim() != 3 or state_pool.dim() != 4:
        raise ValueError("q must be [N, H, dk] and state_pool [nslots, H, dk, dv]")
    N, H, dk = q.shape
    dv = v.shape[-1]
    _check(q, "q", torch.bfloat16)
    _check(k, "k", torch.bfloat16, (N, H, dk))
    _check(v, "v", torch.bfloat16, (N, H, dv))
    _check(out, "out", torch.bfloat16, (N, H, dv))
    _check(log_decay, "log_decay", torch.float32, (H,))
    _check(state_pool, "state_pool", torch.float32, (state_pool.shape[0], H, dk, dv))
    _check(slots, "slots", torch.int32, (N,))
    rc = load().gla_decode_step_paged(_ptr(q), _ptr(k), _ptr(v), _ptr(log_decay), _ptr(state_pool), _ptr(slots),
                                      int(state_pool.shape[0]), _ptr(out), N, H, dk, dv, _stream(stream))
    _raise(rc, "gla_decode_step_paged")


def gla_decode_step_gated(q, k, v, g, log_decay, state_inout, out, gate_kind: int = GATE_SILU, stream=None) -> None:
    """bf16 decode step with the output gate fused into ``out`` (``g`` shaped like ``out``)."""
    N, H, dk, dv = _decode_args(q, k, v, log_decay, state_inout, out, torch.bfloat16)
    _check(g, "g", torch.bfloat16, (N, H, dv))
    rc = load().gla_decode_step_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g), int(gate_kind), _ptr(log_decay),
                                      _ptr(state_inout), _ptr(out), N, H, dk, dv, _stream(stream))
    _raise(rc, "gla_decode_step_gated")


def gla_decode_step_paged_gated(q, k, v, g, log_decay, state_pool, slots, out, gate_kind: int = GATE_SILU,
                                stream=None) -> None:
    """The paged decode step with the output gate fused into ``out``."""
    if q.dim() != 3 or state_pool.dim() != 4:
        raise ValueError("q must be [N, H, dk] and state_pool [nslots, H, dk, dv]")
    N, H, dk = q.shape
    dv = v.shape[-1]
    _check(q, "q", torch.bfloat16)
    _check(k, "k", torch.bfloat16, (N, H, dk))
    _check(v, "v", torch.bfloat16, (N, H, dv))
    _check(g, "g", torch.bfloat16, (N, H, dv))
    _check(out, "out", torch.bfloat16, (N, H, dv))
    _check(log_decay, "log_decay", torch.float32, (H,))
    _check(state_pool, "state_pool", torch.float32, (state_pool.shape[0], H, dk, dv))
    _check(slots, "slots", torch.int32, (N,))
    rc = load().gla_decode_step_paged_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g), int(gate_kind), _ptr(log_decay),
                                            _ptr(state_pool), _ptr(slots), int(state_pool.shape[0]), _ptr(out), N, H,
                                            dk, dv, _stream(stream))
    _raise(rc, "gla_decode_step_paged_gated")


def gla_decode_step_layers(q, k, v, log_decay, state_pool, slots, out, layer0: int = 0, g=None,
                           gate_kind: int = GATE_SILU, stream=None) -> None:
    """Decode steps of L layers in one launch over pages of ``page_layers`` layers: q, k [L, N, H, dk],
    v, out (and g) [L, N, H, dv], log_decay [L, H], state_pool [nslots, page_layers, H, dk, dv], slots [N].
    Layer l of the call uses layer ``layer0 + l`` of page slots[n]."""
    if q.dim() != 4 or state_pool.dim() != 5:
        raise ValueError("q must be [L, N, H, dk] and state_pool [nslots, page_layers, H, dk, dv]")
    L, N, H, dk = q.shape
    dv = v.shape[-1]
    _check(q, "q", torch.bfloat16)
    _check(k, "k", torch.bfloat16, (L, N, H, dk))
    _check(v, "v", torch.bfloat16, (L, N, H, dv))
    _check(out, "out", torch.bfloat16, (L, N, H, dv))
    _check(g, "g", torch.bfloat16, (L, N, H, dv), allow_none=True)
    _check(log_decay, "log_decay", torch.float32, (L, H))
    nslots, page_layers = int(state_pool.shape[0]), int(state_pool.shape[1])
    _check(state_pool, "state_pool", torch.float32, (nslots, page_layers, H, dk, dv))
    _check(slots, "slots", torch.int32, (N,))
    rc = load().gla_decode_step_layers(_ptr(q), _ptr(k), _ptr(v), _ptr(g), int(gate_kind), _ptr(log_decay),
                                       _ptr(state_pool), _ptr(slots), nslots, page_layers, int(layer0), L, _ptr(out),
                                       N, H, dk, dv, _stream(stream))
    _raise(rc, "gla_decode_step_layers")


def _conv_args(x, weight, bias, state_in, state_out, y, cu_seqlens, dtype):
    if x.dim() != 3:
        raise ValueError("x must be [B, T, D] (packed: [1, T, D])")
    B, T, D = x.shape
    _check(x, "x", dtype)
    _check(y, "y", dtype, (B, T, D))
    _check(weight, "weight", torch.float32, (D, 4))
    _check(bias, "bias", torch.float32, (D,), allow_none=True)
    nseq = B
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("a packed batch has leading dimension 1")
        _check(cu_seqlens, "cu_seqlens", torch.int32)
        nseq = cu_seqlens.numel() - 1
    _check(state_in, "state_in", torch.float32, (nseq, D, 3), allow_none=True)
    _check(state_out, "state_out", torch.float32, (nseq, D, 3), allow_none=True)
    return nseq, T, D  # the C ABI takes the number of sequences (N for a packed batch)


def gla_conv1d_silu(x, weight, bias, state_in, state_out, y, cu_seqlens=None, stream=None) -> None:
    """bf16 causal depthwise Conv1d (width 4) + SiLU; see include/gla.h."""
    nseq, T, D = _conv_args(x, weight, bias, state_in, state_out, y, cu_seqlens, torch.bfloat16)
    rc = load().gla_conv1d_silu(_ptr(x), _ptr(weight), _ptr(bias), _ptr(state_in), _ptr(state_out), _ptr(y),
                                nseq, T, D, _ptr(cu_seqlens), _stream(stream))
    _raise(rc, "gla_conv1d_silu")


def gla_conv1d_silu_f32(x, weight, bias, state_in, state_out, y, cu_seqlens=None, stream=None) -> None:
    nseq, T, D = _conv_args(x, weight, bias, state_in, state_out, y, cu_seqlens, torch.float32)
    rc = load().gla_conv1d_silu_f32(_ptr(x), _ptr(weight), _ptr(bias), _ptr(state_in), _ptr(state_out), _ptr(y),
                                    nseq, T, D, _ptr(cu_seqlens), _stream(stream))
    _raise(rc, "gla_conv1d_silu_f32")


def gla_conv1d_silu_step(x, weight, bias, state_inout, y, stream=None) -> None:
    """bf16 conv step for one token of N sequences, in place on state_inout [N, D, 3]."""
    if x.dim() != 2:
        raise ValueError("x must be [N, D]")
    N, D = x.shape
    _check(x, "x", torch.bfloat16)
    _check(y, "y", torch.bfloat16, (N, D))
    _check(weight, "weight", torch.float32, (D, 4))
    _check(bias, "bias", torch.float32, (D,), allow_none=True)
    _check(state_inout, "state_inout", torch.float32, (N, D, 3))
    rc = load().gla_conv1d_silu_step(_ptr(x), _ptr(weight), _ptr(bias), _ptr(state_inout), _ptr(y), N, D,
                                     _stream(stream))
    _raise(rc, "gla_conv1d_silu_step")


def gla_last_device_status(stream=None) -> int:
    """Synchronise the stream; return and clear the library's device status word."""
    return int(load().gla_last_device_status(_stream(stream)))


def gla_status_str(status: int) -> str:
    return load().gla_status_str(int(status)).decode()


OP_FORWARD, OP_FORWARD_GATED, OP_BACKWARD = 0, 1, 2   # gla_op
BF16, F32 = 0, 1                                      # gla_dtype
KERNEL_TENSOR_CORE, KERNEL_SIMT = 1, 2                # gla_kernel_kind


def gla_chunk_kernel(op: int, dtype: int, dk: int, dv: int, chunk: int) -> int:
    """Which kernel a chunked entry point runs for these sizes on the current device: KERNEL_TENSOR_CORE,
    KERNEL_SIMT, or a negative gla_status for sizes it rejects.  See include/gla.h."""
    return int(load().gla_chunk_kernel(int(op), int(dtype), int(dk), int(dv), int(chunk)))


def gla_kernel_launches() -> int:
    """Kernels launched by the library so far in this process."""
    return int(load().gla_kernel_launches())


def gla_version() -> int:
    return int(load().gla_version())


# ---- conveniences ---------------------------------------------------------------------------

def chunk_fwd(q, k, v, log_decay, h0=None, chunk: int = 128, cu_seqlens=None, final_state: bool = True,
              stream=None):
    """Allocate ``out`` (and ``hT``) and run the chunked forward; returns (out, hT or None)."""
    nseq = q.shape[0] if cu_seqlens is None else cu_seqlens.numel() - 1
    out = torch.empty(q.shape[:3] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    hT = torch.empty((nseq, q.shape[2], q.shape[3], v.shape[-1]), dtype=torch.float32, device=q.device) \
        if final_state else None
    if q.dtype == torch.float32:
        gla_chunk_fwd_f32(q, k, v, log_decay, h0, out, hT, chunk, cu_seqlens, stream)
    else:
        gla_chunk_fwd(q, k, v, log_decay, h0, out, hT, chunk, cu_seqlens, stream)
    return out, hT


def chunk_bwd(q, k, v, dout, log_decay, h0=None, dhT=None, chunk: int = 128, cu_seqlens=None, stream=None):
    """Allocate and return (dq, dk, dv, dh0) for the chunked forward's gradients."""
    nseq = q.shape[0] if cu_seqlens is None else cu_seqlens.numel() - 1
    dq, dk = torch.empty_like(q), torch.empty_like(k)
    dv = torch.empty_like(v)
    dh0 = torch.empty((nseq, q.shape[2], q.shape[3], v.shape[-1]), dtype=torch.float32, device=q.device)
    fn = gla_chunk_bwd_f32 if q.dtype == torch.float32 else gla_chunk_bwd
    fn(q, k, v, dout, log_decay, h0, dhT, dq, dk, dv, dh0, chunk, cu_seqlens, stream)
    return dq, dk, dv, dh0


def decode_step(q, k, v, log_decay, state, stream=None):
    """Run one decode step in place on ``state``; returns the new ``out`` tensor."""
    out = torch.empty(q.shape[:2] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    if q.dtype == torch.float32:
        gla_decode_step_f32(q, k, v, log_decay, state, out, stream)
    else:
        gla_decode_step(q, k, v, log_decay, state, out, stream)
    return out
