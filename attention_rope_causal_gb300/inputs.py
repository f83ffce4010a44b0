"""Seeded synthetic inputs for RoPE + causal attention.

This module holds no arithmetic of the method: it only names the workloads (shapes, dtype, rope base,
value scale, seed) and draws q, k, v from a seeded CPU generator.  Both the CUDA path's tests and the
oracle's tests take their inputs from here.

Recipe: ``torch.Generator('cpu').manual_seed(seed)``; draw fp32 standard normals in the order q, k, v
with shapes [B, N, Hq, d], [B, N, Hkv, d], [B, N, Hkv, d]; multiply by ``sigma`` (a standard
deviation); round to the workload's dtype.  No dataset is involved: the Llama-3-8B workload of the
AttnFuse report stands in only through its attention shape (32 query heads, 8 KV heads, head_dim 128,
rope base 500000).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    dtype: str  # "bf16" | "fp16"
    rope_base: float
    sigma: float
    seed: int

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"bf16": torch.bfloat16, "fp16": torch.float16}[self.dtype]

    @property
    def causal_flops(self) -> float:
        """The conventional causal count 2*B*Hq*N^2*d (QK^T and PV over the causal half)."""
        return 2.0 * self.B * self.Hq * float(self.N) ** 2 * self.d

    @property
    def tokens(self) -> int:
        return self.B * self.N

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


TINY = Workload("tiny", B=1, Hq=2, Hkv=2, N=128, d=64, dtype="bf16", rope_base=10000.0, sigma=1.0, seed=0)
MHA = Workload("mha", B=2, Hq=16, Hkv=16, N=2048, d=64, dtype="bf16", rope_base=10000.0, sigma=1.0, seed=1)
LLAMA = Workload("llama3_8b_gqa", B=1, Hq=32, Hkv=8, N=4096, d=128, dtype="bf16", rope_base=500000.0,
                 sigma=1.0, seed=2)
LONG = Workload("long_32k", B=1, Hq=32, Hkv=8, N=32768, d=128, dtype="fp16", rope_base=500000.0, sigma=0.5,
                seed=3)

SWEEP_NS = (2048, 4096, 5500, 8192, 16384)
SWEEP_EXTRA_NS = (1024, 1536)  # below the sweep's range, so that a crossover near 2048 is bracketed
SWEEP_TOKENS = 16384


def sweep_workloads(extra: bool = False):
    """Crossover sweep: GQA d=128 (32/8) and MHA d=64 (16/16), N in SWEEP_NS, B = round(16384 / N),
    fp16 and bf16, rope base 500000.  Seeds are 100 + the point's index in this list.  With extra,
    the points N in SWEEP_EXTRA_NS follow (same families and dtypes, seeds continuing)."""
    out = []
    idx = 0
    groups = [SWEEP_NS] + ([SWEEP_EXTRA_NS] if extra else [])
    for ns in groups:
        for family, (Hq, Hkv, d) in (("gqa", (32, 8, 128)), ("mha", (16, 16, 64))):
            for dtype in ("bf16", "fp16"):
                for N in ns:
                    B = max(1, round(SWEEP_TOKENS / N))
                    out.append(Workload(f"sweep_{family}_d{d}_{dtype}_N{N}", B=B, Hq=Hq, Hkv=Hkv, N=N, d=d,
                                        dtype=dtype, rope_base=500000.0, sigma=1.0, seed=100 + idx))
                    idx += 1
    return out


NAMED = {w.name: w for w in (TINY, MHA, LLAMA, LONG)}


def make_inputs(w: Workload, device=None):
    """Draw (q, k, v) for workload ``w`` on the CPU from its seed, then move them to ``device``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed))
    shapes = ((w.B, w.N, w.Hq, w.d), (w.B, w.N, w.Hkv, w.d), (w.B, w.N, w.Hkv, w.d))
    out = []
    for shape in shapes:
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if w.sigma != 1.0:
            x.mul_(w.sigma)
        x = x.to(w.torch_dtype)
        if device is not None:
            x = x.to(device)
        out.append(x)
    return tuple(out)


def make_kv_inputs(B: int, N: int, Nk: int, Hq: int, Hkv: int, d: int, dtype: str, seed: int, sigma: float = 1.0,
                   device=None):
    """(q, k, v) with more keys than queries: q [B, N, Hq, d], k and v [B, Nk, Hkv, d]; same recipe as
    :func:`make_inputs` (fp32 standard normals in the order q, k, v from ``seed``, times sigma, cast)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    t = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    out = []
    for shape in ((B, N, Hq, d), (B, Nk, Hkv, d), (B, Nk, Hkv, d)):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if sigma != 1.0:
            x.mul_(sigma)
        x = x.to(t)
        out.append(x if device is None else x.to(device))
    return tuple(out)


def make_positions(B: int, n: int, seed: int, low: int = -4096, high: int = 1 << 20) -> torch.Tensor:
    """Random int32 rotation positions [B, n] in [low, high) (any integers are valid positions)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randint(low, high, (B, n), generator=g, dtype=torch.int64).to(torch.int32)
