"""RoPE variants through the C ABI (attnfuse_rope_apply_ex, attnfuse_rope_causal_fwd_ex): a rotary
dimension r < d (only the first r entries rotated, theta_k = base^(-2k/r)) and interleaved pairs
(2k, 2k+1), in the pre-rotation pass and in every attention mode, against the oracle's fp64
definition of each variant.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_rope_causal_gb300 import binding, build, inputs
from parity import TOL, assert_close, errors

pytestmark = pytest.mark.gpu

MANT = {torch.bfloat16: 7, torch.float16: 10}

VARIANTS = [
    # d, rotary_dim, interleaved
    (128, 128, True),
    (128, 64, False),
    (128, 64, True),
    (128, 32, False),
    (64, 32, True),
    (64, 16, False),
    (64, 64, True),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def ulp(x: np.ndarray, dtype) -> np.ndarray:
    m = MANT[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    min_exp = -126 if dtype == torch.bfloat16 else -14
    return np.exp2(np.maximum(e, min_exp) - m)


def partner(x: np.ndarray, r: int, interleaved: bool) -> np.ndarray:
    """For each rotated entry, the other entry of its pair (the tail maps to itself)."""
    d = x.shape[-1]
    idx = np.arange(d)
    if interleaved:
        idx[:r] = np.arange(r) ^ 1
    else:
        idx[: r // 2] = np.arange(r // 2, r)
        idx[r // 2: r] = np.arange(r // 2)
    return x[..., idx]


@pytest.mark.parametrize("d,r,il", VARIANTS)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_rope_apply_variant_matches_oracle(d, r, il, dtype):
    # Same bound as the default form: one ulp at the exact value plus 2^-20 (|x_a| + |x_b|) for the
    # pair's fp32 arithmetic; entries past the rotary dimension are copied exactly.
    B, N, H = 2, 777, 5
    g = torch.Generator().manual_seed(d + r + int(il))
    x = torch.randn((B, N, H, d), generator=g).to(dtype)
    y = binding.rope_apply(x.cuda(), 5e5, rotary_dim=r, interleaved=il).cpu()
    assert binding.device_status() == 0
    ref = oracle.rope_rotate_bnhd(x, 5e5, rotary_dim=r, interleaved=il)
    xd = x.double().numpy()
    err = np.abs(y.double().numpy() - ref)
    bound = ulp(ref, dtype) + 2.0 ** -20 * (np.abs(xd) + np.abs(partner(xd, r, il)))
    assert float((err / bound).max()) <= 1.0
    assert torch.equal(y[..., r:], x[..., r:])


@pytest.mark.parametrize("d,r,il", [(128, 64, True), (64, 16, False)])
def test_rope_apply_variant_in_place(d, r, il):
    g = torch.Generator().manual_seed(3)
    x = torch.randn((1, 300, 3, d), generator=g).to(torch.bfloat16).cuda()
    y = binding.rope_apply(x, 1e4, rotary_dim=r, interleaved=il)
    x2 = x.clone()
    binding.rope_apply(x2, 1e4, out=x2, rotary_dim=r, interleaved=il)
    torch.cuda.synchronize()
    assert torch.equal(x2, y)


def draw(B, N, Hq, Hkv, d, dtype, seed):
    w = inputs.Workload("case", B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, dtype=dtype, rope_base=1e4, sigma=1.0, seed=seed)
    return inputs.make_inputs(w)


ATTN = [
    # B, N, Hq, Hkv, d, dtype, rotary_dim, interleaved
    (1, 300, 4, 2, 128, "bf16", 64, True),    # head-pair units, ragged last tile
    (1, 257, 3, 3, 128, "fp16", 32, False),   # row-pair units
    (2, 200, 8, 2, 128, "bf16", 128, True),
    (1, 385, 2, 1, 64, "fp16", 32, True),
    (1, 640, 4, 4, 64, "bf16", 16, False),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,d,dt,r,il", ATTN)
def test_attention_variant_matches_oracle(B, N, Hq, Hkv, d, dt, r, il):
    q, k, v = draw(B, N, Hq, Hkv, d, dt, seed=N + r)
    o_ref, l_ref = oracle.rope_causal(q, k, v, 1e4, rotary_dim=r, interleaved=il)
    outs = {}
    for mode in ("fused", "prerotate", "split"):
        o, l = binding.rope_causal_fwd(q.cuda(), k.cuda(), v.cuda(), 1e4, mode=mode, rotary_dim=r, interleaved=il)
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        outs[mode] = (o.cpu(), l.cpu())
        assert_close(o.double().cpu().numpy(), l.double().cpu().numpy(), o_ref, l_ref, dt,
                     f"{mode} r={r} interleaved={il} {B}x{N}x{Hq}/{Hkv}x{d} {dt}")
    # the two modes agree to well within the oracle tolerance (as for the default form)
    t = TOL[dt]
    for m in ("fused", "split"):
        e = errors(outs[m][0].double().numpy(), outs[m][1].double().numpy(),
                   outs["prerotate"][0].double().numpy(), outs["prerotate"][1].double().numpy())
        assert e["max_abs"] <= t["max_abs"] / 4 and e["rel_l2"] <= t["rel_l2"] / 4, (m, e)


def test_full_half_split_options_equal_the_default_call():
    q, k, v = draw(1, 256, 4, 2, 128, "bf16", seed=5)
    a, la = binding.rope_causal_fwd(q.cuda(), k.cuda(), v.cuda(), 1e4)
    b, lb = binding.rope_causal_fwd(q.cuda(), k.cuda(), v.cuda(), 1e4, rotary_dim=128, interleaved=False)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(la, lb)
