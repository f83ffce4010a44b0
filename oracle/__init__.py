"""Reference oracle for RoPE + causal softmax attention (CPU, IEEE double).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline leg may use
this package; the library's product path never imports it.  It shares no code with the CUDA path.

The arithmetic lives in ``rope_causal_oracle.c`` (plain C loops, fp64, threaded over rows).  This
module compiles it with the host C compiler into ``oracle/_build/`` and marshals arrays through
ctypes.  What it computes, and the passages it follows, are stated in that file's header:

* RoPE as a pre-multiplication transform on Q and K ("AttnFuse Makes RoPE a First-Class Attention
  Compilation Operation", 2026-09-13 AI papers report, paragraph 1; AttnFuse abstract), half-split
  pairs (k, k+d/2), theta_k = base^(-2k/d), position = token index;
* causal softmax attention (same report, paragraph 2: causality and softmax building blocks),
  scale 1/sqrt(d), natural-log log-sum-exp per row, GQA head h -> kv head floor(h*Hkv/Hq);
* RoPE variants (``rotary_dim``, ``interleaved``): only the first r entries rotated with
  theta_k = base^(-2k/r), and adjacent pairs (2k, 2k+1) instead of (k, k+r/2);
* more keys than queries (k, v with Nk >= Nq tokens: the queries are the last Nq, so query i sees
  keys j <= Nk - Nq + i) and explicit rotation positions (``q_positions``, ``k_positions``), which
  change the angles only;
* the backward pass (``rope_causal_bwd``): gradients of sum(dout * out) through the softmax, the
  products and the rotation (dq = R^T dq', dk = R^T dk').
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rope_causal_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

ORC_F64, ORC_BF16, ORC_F16 = 0, 1, 2

_lock = threading.Lock()
_lib = None


# Load this shared library instead of building oracle/_build/liboracle.so (the planted-mistake test
# runs the pin suites against deliberately broken copies of the C source built this way).
LIB_ENV = "ATTNFUSE_ORACLE_LIB"


def compile_source(src: str, out: str) -> str:
    """Compile an oracle C source into a shared library (plain IEEE: no fast-math, no FMA contraction)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math",
           src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        compile_source(_SRC, tmp)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def source_path() -> str:
    return _SRC


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(os.environ.get(LIB_ENV) or build())
            lib.orc_rope_rotate.restype = ctypes.c_int
            lib.orc_rope_rotate.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_void_p, ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
            lib.orc_rope_causal.restype = ctypes.c_int
            lib.orc_rope_causal.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int]
            lib.orc_rope_rotate_ex.restype = ctypes.c_int
            lib.orc_rope_rotate_ex.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                               ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
            lib.orc_rope_causal_ex.restype = ctypes.c_int
            lib.orc_rope_causal_ex.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_void_p,
                                               ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.orc_rope_causal_kv.restype = ctypes.c_int
            lib.orc_rope_causal_kv.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.orc_rope_causal_bwd_kv.restype = ctypes.c_int
            lib.orc_rope_causal_bwd_kv.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.orc_rope_causal_bwd_ex.restype = ctypes.c_int
            lib.orc_rope_causal_bwd_ex.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_void_p, ctypes.c_int]
            lib.orc_rope_causal_bwd.restype = ctypes.c_int
            lib.orc_rope_causal_bwd.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _as_raw(x):
    """Return (contiguous numpy buffer, dtype code).  Accepts torch CPU tensors (bf16/fp16/fp64) or numpy."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), ORC_BF16
        if x.dtype == torch.float16:
            return x.view(torch.int16).numpy().view(np.uint16), ORC_F16
        if x.dtype == torch.float64:
            return x.numpy(), ORC_F64
        raise TypeError(f"oracle accepts bf16, fp16 or fp64 tensors, got {x.dtype}")
    x = np.ascontiguousarray(x)
    if x.dtype == np.float64:
        return x, ORC_F64
    if x.dtype == np.float16:
        return x.view(np.uint16), ORC_F16
    raise TypeError(f"oracle accepts float64/float16 arrays or torch bf16/fp16/fp64 tensors, got {x.dtype}")


def rope_rotate(x, base: float, positions=None, threads: int | None = None, rotary_dim: int | None = None,
                interleaved: bool = False) -> np.ndarray:
    """Rotate x of shape [..., R, H, d] (R rows of H heads); row r sits at positions[r] (default: r).

    rotary_dim (default d) rotates only the first rotary_dim entries; interleaved pairs (2k, 2k+1).

    Leading dimensions are flattened into rows, so for [B, N, H, d] the default position of (b, n) is
    n only when B == 1; pass ``positions`` explicitly (or use :func:`rope_rotate_bnhd`) otherwise.
    """
    raw, dt = _as_raw(x)
    shape = raw.shape
    if len(shape) < 2:
        raise ValueError("x must have at least 2 dims [..., H, d]")
    H, d = shape[-2], shape[-1]
    rows = int(np.prod(shape[:-2])) if len(shape) > 2 else 1
    if positions is None:
        pos = np.arange(rows, dtype=np.float64)
    else:
        pos = np.ascontiguousarray(np.asarray(positions, dtype=np.float64).reshape(-1))
        if pos.size != rows:
            raise ValueError(f"positions has {pos.size} entries for {rows} rows")
    out = np.empty(shape, dtype=np.float64)
    r = d if rotary_dim is None else int(rotary_dim)
    rc = _load().orc_rope_rotate_ex(raw.ctypes.data, dt, rows, H, d, r, int(bool(interleaved)), pos.ctypes.data,
                                    float(base), out.ctypes.data, int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError("orc_rope_rotate_ex failed")
    return out


def rope_rotate_bnhd(x, base: float, threads: int | None = None, rotary_dim: int | None = None,
                     interleaved: bool = False) -> np.ndarray:
    """Rotate x of shape [B, N, H, d] with position = token index n (the library's convention)."""
    B, N = x.shape[0], x.shape[1]
    pos = np.tile(np.arange(N, dtype=np.float64), B)
    return rope_rotate(x, base, positions=pos, threads=threads, rotary_dim=rotary_dim, interleaved=interleaved)


def _positions(pos, B: int, n: int, what: str):
    if pos is None:
        return None
    if hasattr(pos, "detach"):
        pos = pos.detach().cpu().numpy()
    a = np.ascontiguousarray(np.asarray(pos, dtype=np.float64).reshape(-1))
    if a.size != B * n:
        raise ValueError(f"{what} has {a.size} entries, expected B * {n} = {B * n}")
    return a


def rope_causal(q, k, v, base: float, rows=None, threads: int | None = None, rotary_dim: int | None = None,
                interleaved: bool = False, q_positions=None, k_positions=None):
    """Causal softmax attention with RoPE on q and k.

    rotary_dim (default d) and interleaved select the RoPE variant (see :func:`rope_rotate`).

    q: [B, Nq, Hq, d]; k, v: [B, Nk, Hkv, d] with Nk >= Nq (same dtype: bf16/fp16 torch tensors, fp16 or
    fp64 arrays).  The queries are the last Nq of the Nk tokens: query i sees keys j <= (Nk - Nq) + i.
    q_positions [B, Nq] / k_positions [B, Nk] (integers; default (Nk - Nq) + i and j) are the rotation
    positions; they change the angles only, never the mask.
    rows: optional 1-D sequence of query rows to evaluate (default: all Nq in order).
    Returns (out [B, R, Hq, d] float64, lse [B, Hq, R] float64) with R = len(rows) or Nq.
    """
    qr, dq = _as_raw(q)
    kr, dk = _as_raw(k)
    vr, dv = _as_raw(v)
    if not (dq == dk == dv):
        raise TypeError("q, k, v must share one dtype")
    if qr.ndim != 4 or kr.ndim != 4 or vr.ndim != 4:
        raise ValueError("q, k, v must be 4-D [B, N, H, d]")
    B, N, Hq, d = qr.shape
    Nk, Hkv = kr.shape[1], kr.shape[2]
    if kr.shape != (B, Nk, Hkv, d) or vr.shape != (B, Nk, Hkv, d):
        raise ValueError("k and v must be [B, Nk, Hkv, d] matching q")
    if Nk < N:
        raise ValueError("k and v must hold at least as many tokens as q")
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    qp = _positions(q_positions, B, N, "q_positions")
    kp = _positions(k_positions, B, Nk, "k_positions")
    if rows is None:
        sel_ptr, n_sel, sel = None, N, None
    else:
        sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        if sel.size and (sel.min() < 0 or sel.max() >= N):
            raise ValueError("rows out of range")
        sel_ptr, n_sel = sel.ctypes.data, int(sel.size)
    out = np.zeros((B, n_sel, Hq, d), dtype=np.float64)
    lse = np.zeros((B, Hq, n_sel), dtype=np.float64)
    if n_sel == 0:
        return out, lse
    r = d if rotary_dim is None else int(rotary_dim)
    rc = _load().orc_rope_causal_kv(qr.ctypes.data, kr.ctypes.data, vr.ctypes.data, dq, B, Hq, Hkv, N, Nk, d, r,
                                    int(bool(interleaved)), float(base), None if qp is None else qp.ctypes.data,
                                    None if kp is None else kp.ctypes.data, sel_ptr, n_sel, out.ctypes.data,
                                    lse.ctypes.data, int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError("orc_rope_causal_kv failed")
    return out, lse


def _rows(rows, N: int, what: str):
    if rows is None:
        return None, N, None
    sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    if sel.size and (sel.min() < 0 or sel.max() >= N):
        raise ValueError(f"{what} out of range")
    if np.unique(sel).size != sel.size:
        raise ValueError(f"{what} must be distinct")
    return sel.ctypes.data, int(sel.size), sel


def rope_causal_bwd(q, k, v, dout, base: float, q_rows=None, k_rows=None, threads: int | None = None,
                    rotary_dim: int | None = None, interleaved: bool = False, q_positions=None, k_positions=None):
    """Backward pass of :func:`rope_causal`: the gradients of L = sum(dout * out) with respect to q,
    k and v (no lse term).

    q, dout: [B, Nq, Hq, d]; k, v: [B, Nk, Hkv, d] with Nk >= Nq (the queries are the last Nq of the
    Nk tokens, as in :func:`rope_causal`), one dtype (bf16/fp16 torch tensors, fp16 or fp64 arrays).
    q_rows / k_rows select the query rows whose dq and the key rows whose dk, dv are returned
    (default: all, in order).  rotary_dim, interleaved, q_positions ([B, Nq]) and k_positions
    ([B, Nk]) select the RoPE form as for :func:`rope_causal`.  Returns (dq [B, Rq, Hq, d],
    dk [B, Rk, Hkv, d], dv [B, Rk, Hkv, d]) as float64.
    """
    qr, dq_ = _as_raw(q)
    kr, dk_ = _as_raw(k)
    vr, dv_ = _as_raw(v)
    gr, dg_ = _as_raw(dout)
    if not (dq_ == dk_ == dv_ == dg_):
        raise TypeError("q, k, v, dout must share one dtype")
    B, N, Hq, d = qr.shape
    Nk, Hkv = kr.shape[1], kr.shape[2]
    if kr.shape != (B, Nk, Hkv, d) or vr.shape != (B, Nk, Hkv, d) or gr.shape != qr.shape:
        raise ValueError("k, v must be [B, Nk, Hkv, d] and dout [B, N, Hq, d]")
    if Nk < N:
        raise ValueError("k and v must hold at least as many tokens as q")
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    qpos = _positions(q_positions, B, N, "q_positions")
    kpos = _positions(k_positions, B, Nk, "k_positions")
    qp, nq, _qs = _rows(q_rows, N, "q_rows")
    kp, nk, _ks = _rows(k_rows, Nk, "k_rows")
    dq = np.zeros((B, nq, Hq, d))
    dk = np.zeros((B, nk, Hkv, d))
    dv = np.zeros((B, nk, Hkv, d))
    r = d if rotary_dim is None else int(rotary_dim)
    rc = _load().orc_rope_causal_bwd_kv(qr.ctypes.data, kr.ctypes.data, vr.ctypes.data, gr.ctypes.data, dq_, B, Hq,
                                        Hkv, N, Nk, d, r, int(bool(interleaved)), float(base),
                                        None if qpos is None else qpos.ctypes.data,
                                        None if kpos is None else kpos.ctypes.data, qp, nq, kp, nk, dq.ctypes.data,
                                        dk.ctypes.data, dv.ctypes.data, int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError("orc_rope_causal_bwd_kv failed")
    return dq, dk, dv
