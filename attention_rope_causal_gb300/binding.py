"""Thin ctypes binding over libattnfuse's C ABI (include/attnfuse.h).

Argument marshalling only: every step of the computation runs in the library's CUDA kernels.
PyTorch supplies device memory and the current CUDA stream.  There is no CPU fallback: if the
library is missing or the device is not sm_103a, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

ATTNFUSE_FUSED, ATTNFUSE_PREROTATE, ATTNFUSE_AUTO, ATTNFUSE_SPLIT, ATTNFUSE_NONE = 0, 1, 2, 3, 4
ATTNFUSE_BF16, ATTNFUSE_FP16 = 0, 1
STATUS = {0: "OK", 1: "ERR_INVALID_ARG", 2: "ERR_UNSUPPORTED", 3: "ERR_CUDA", 4: "ERR_TIMEOUT", 5: "ERR_NO_MEMORY"}
MODES = {"fused": ATTNFUSE_FUSED, "prerotate": ATTNFUSE_PREROTATE, "auto": ATTNFUSE_AUTO, "split": ATTNFUSE_SPLIT,
         "none": ATTNFUSE_NONE}
MODE_NAMES = {v: k for k, v in MODES.items()}
DTYPES = {torch.bfloat16: ATTNFUSE_BF16, torch.float16: ATTNFUSE_FP16}

class RopeOpts(ctypes.Structure):
    """attnfuse_rope_opts_t: rotary_dim (0 = d), interleaved (0 = half-split pairs), kv_len (0 = N) and the
    device pointers of the int32 query / key position arrays (NULL = defaults)."""
    _fields_ = [("rotary_dim", ctypes.c_int), ("interleaved", ctypes.c_int), ("kv_len", ctypes.c_int),
                ("q_positions", ctypes.c_void_p), ("k_positions", ctypes.c_void_p)]


# Every function the header declares, with its ctypes signature.
_SIGNATURES = {
    "attnfuse_rope_causal_fwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "attnfuse_rope_causal_fwd_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                                   ctypes.POINTER(RopeOpts), ctypes.c_void_p]),
    "attnfuse_rope_apply_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.POINTER(RopeOpts),
                                              ctypes.c_void_p]),
    "attnfuse_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 7),
    "attnfuse_rope_causal_bwd": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_int] * 5 + [ctypes.c_double, ctypes.c_int,
                                                                                        ctypes.c_void_p, ctypes.c_size_t,
                                                                                        ctypes.c_void_p]),
    "attnfuse_rope_causal_bwd_ex": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_int] * 5 +
                                    [ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                     ctypes.POINTER(RopeOpts), ctypes.c_void_p]),
    "attnfuse_bwd_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 6),
    "attnfuse_bwd_workspace_bytes_ex": (ctypes.c_size_t, [ctypes.c_int] * 6 + [ctypes.POINTER(RopeOpts)]),
    "attnfuse_workspace_bytes_ex": (ctypes.c_size_t, [ctypes.c_int] * 7 + [ctypes.POINTER(RopeOpts)]),
    "attnfuse_select_mode": (ctypes.c_int, [ctypes.c_int] * 6),
    "attnfuse_rope_causal_fwd_prerotate_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                                                  ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                                  ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                                                  ctypes.c_void_p]),
    "attnfuse_rope_apply": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_void_p]),
    "attnfuse_device_status": (ctypes.c_int, [ctypes.c_void_p]),
    "attnfuse_diag_wait_timeout": (ctypes.c_int, [ctypes.c_uint64, ctypes.c_void_p]),
    "attnfuse_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "attnfuse_last_error": (ctypes.c_char_p, []),
    "attnfuse_version": (ctypes.c_char_p, []),
}


class AttnFuseError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load libattnfuse.so (built by ``attention_rope_causal_gb300.build.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with attention_rope_causal_gb300.build.build()")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(status: int):
    if status != 0:
        lib = load()
        raise AttnFuseError(status, lib.attnfuse_last_error().decode(errors="replace"))


def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def workspace_bytes(B, Hq, Hkv, N, d, mode="fused", dtype=torch.bfloat16, kv_len=None) -> int:
    if kv_len is None:
        return int(load().attnfuse_workspace_bytes(B, Hq, Hkv, N, d, MODES[mode], DTYPES[dtype]))
    opts = RopeOpts(0, 0, int(kv_len), None, None)
    return int(load().attnfuse_workspace_bytes_ex(B, Hq, Hkv, N, d, MODES[mode], DTYPES[dtype], ctypes.byref(opts)))


def select_mode(B, Hq, Hkv, N, d, dtype=torch.bfloat16) -> str:
    """The mode ``auto`` resolves to for this shape (``attnfuse_select_mode``)."""
    return MODE_NAMES[int(load().attnfuse_select_mode(B, Hq, Hkv, N, d, DTYPES[dtype]))]


def _positions(pos, n_tokens: int, name: str):
    if pos is None:
        return None
    if not (pos.is_cuda and pos.dtype == torch.int32 and pos.is_contiguous() and pos.numel() == n_tokens):
        raise ValueError(f"{name} must be a contiguous CUDA int32 tensor of {n_tokens} elements")
    return pos.data_ptr()


def _opts(rotary_dim, interleaved, kv_len=0, q_positions=None, k_positions=None):
    if rotary_dim is None and not interleaved and not kv_len and q_positions is None and k_positions is None:
        return None
    return RopeOpts(int(rotary_dim or 0), int(bool(interleaved)), int(kv_len), q_positions, k_positions)


def rope_causal_fwd(q, k, v, rope_base: float, mode: str = "fused", out=None, lse=None, want_lse: bool = True,
                    workspace=None, stream=None, rotary_dim=None, interleaved: bool = False, q_positions=None,
                    k_positions=None):
    """Causal RoPE attention forward through ``attnfuse_rope_causal_fwd`` (``_ex`` with any option).

    q: [B, N, Hq, d], k/v: [B, Nk, Hkv, d] CUDA tensors (bf16 or fp16, contiguous), Nk >= N: the
    queries are the last N of the Nk tokens (query i sees keys j <= Nk - N + i).
    rotary_dim / interleaved select a RoPE variant; q_positions [B, N] / k_positions [B, Nk] (CUDA
    int32) replace the default rotation positions Nk - N + i / j (attnfuse_rope_opts_t).
    Returns (out [B, N, Hq, d], lse [B, Hq, N] float32 or None).
    """
    B, N, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    opts = _opts(rotary_dim, interleaved, Nk if Nk != N else 0, _positions(q_positions, B * N, "q_positions"),
                 _positions(k_positions, B * Nk, "k_positions"))
    if opts is None:
        _check(load().attnfuse_rope_causal_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, N, d,
                                               float(rope_base), MODES[mode], DTYPES[q.dtype], ws_ptr, ws_bytes,
                                               _stream_ptr(stream)))
    else:
        _check(load().attnfuse_rope_causal_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, N, d,
                                                  float(rope_base), MODES[mode], DTYPES[q.dtype], ws_ptr, ws_bytes,
                                                  ctypes.byref(opts), _stream_ptr(stream)))
    return out, lse


def rope_apply(x, rope_base: float, out=None, stream=None, rotary_dim=None, interleaved: bool = False,
               positions=None):
    """y = RoPE(x) for x [B, N, H, d] through ``attnfuse_rope_apply`` (out may be x: in place);
    ``attnfuse_rope_apply_ex`` for a RoPE variant or explicit positions ([B, N] CUDA int32)."""
    B, N, H, d = x.shape
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty_like(x)
    opts = _opts(rotary_dim, interleaved, 0, _positions(positions, B * N, "positions"))
    if opts is None:
        _check(load().attnfuse_rope_apply(_ptr(x), _ptr(out), B, N, H, d, float(rope_base), DTYPES[x.dtype],
                                          _stream_ptr(stream)))
    else:
        _check(load().attnfuse_rope_apply_ex(_ptr(x), _ptr(out), B, N, H, d, float(rope_base), DTYPES[x.dtype],
                                             ctypes.byref(opts), _stream_ptr(stream)))
    return out


def bwd_workspace_bytes(B, Hq, Hkv, N, d, dtype=torch.bfloat16, kv_len=None) -> int:
    if kv_len is None:
        return int(load().attnfuse_bwd_workspace_bytes(B, Hq, Hkv, N, d, DTYPES[dtype]))
    opts = RopeOpts(0, 0, int(kv_len), None, None)
    return int(load().attnfuse_bwd_workspace_bytes_ex(B, Hq, Hkv, N, d, DTYPES[dtype], ctypes.byref(opts)))


def rope_causal_bwd(q, k, v, out, lse, dout, rope_base: float, dq=None, dk=None, dv=None, workspace=None,
                    stream=None, rotary_dim=None, interleaved: bool = False, q_positions=None, k_positions=None):
    """Backward pass through ``attnfuse_rope_causal_bwd`` (``_ex`` with a RoPE variant, positions or
    more keys than queries): (dq, dk, dv) for q [B, N, Hq, d], k/v [B, Nk, Hkv, d] with Nk >= N (the
    queries are the last N of the Nk tokens), the forward's out [B, N, Hq, d] and lse [B, Hq, N]
    (float32), and dout = dL/dout.  All CUDA tensors, contiguous, one 16-bit dtype (lse float32);
    q_positions [B, N] and k_positions [B, Nk] CUDA int32."""
    B, N, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("lse", lse), ("dout", dout)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    opts = _opts(rotary_dim, interleaved, Nk if Nk != N else 0, _positions(q_positions, B * N, "q_positions"),
                 _positions(k_positions, B * Nk, "k_positions"))
    if opts is None:
        _check(load().attnfuse_rope_causal_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                                               _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, float(rope_base), DTYPES[q.dtype],
                                               ws_ptr, ws_bytes, _stream_ptr(stream)))
    else:
        _check(load().attnfuse_rope_causal_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                                  _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, float(rope_base),
                                                  DTYPES[q.dtype], ws_ptr, ws_bytes, ctypes.byref(opts),
                                                  _stream_ptr(stream)))
    return dq, dk, dv


def device_status(stream=None) -> int:
    """Synchronise the stream and read (and clear) the kernels' device status word; returns the status code."""
    return int(load().attnfuse_device_status(_stream_ptr(stream)))


def diag_wait_timeout(timeout_ns: int, stream=None):
    _check(load().attnfuse_diag_wait_timeout(int(timeout_ns), _stream_ptr(stream)))


def last_error() -> str:
    return load().attnfuse_last_error().decode(errors="replace")


class RopeCausalAttention(torch.autograd.Function):
    """torch.autograd wrapper: forward through ``attnfuse_rope_causal_fwd``, backward through
    ``attnfuse_rope_causal_bwd`` (gradients for q, k, v; the lse output carries none)."""

    @staticmethod
    def forward(ctx, q, k, v, rope_base: float, mode: str = "auto", rotary_dim=None, interleaved: bool = False):
        out, lse = rope_causal_fwd(q, k, v, rope_base, mode=mode, rotary_dim=rotary_dim, interleaved=interleaved)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.rope = (rope_base, rotary_dim, interleaved)
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, dlse):
        q, k, v, out, lse = ctx.saved_tensors
        rope_base, rotary_dim, interleaved = ctx.rope
        dq, dk, dv = rope_causal_bwd(q, k, v, out, lse, dout.contiguous(), rope_base, rotary_dim=rotary_dim,
                                     interleaved=interleaved)  # k, v may hold more rows than q
        return dq, dk, dv, None, None, None, None


def rope_causal_attention(q, k, v, rope_base: float, mode: str = "auto", rotary_dim=None, interleaved: bool = False):
    """Differentiable causal RoPE attention: returns out [B, N, Hq, d] (lse is kept for the backward).
    k, v may hold Nk >= N tokens (the queries are the last N); their gradients cover all Nk."""
    out, _ = RopeCausalAttention.apply(q, k, v, rope_base, mode, rotary_dim, interleaved)
    return out
