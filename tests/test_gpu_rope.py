"""Pre-rotation kernel (attnfuse_rope_apply) against the oracle's fp64 rotation.

Bound per element: one unit in the last place of the output dtype at the exact value, plus
2^-20 (|x_k| + |x_{k+d/2}|) for the pair's fp32 arithmetic and its cos/sin (angle error below
4e-7 rad).  The second term matters only where x cos and y sin nearly cancel, where no fp32
evaluation can promise one ulp of the (tiny) result."""
import numpy as np
import pytest
import torch

import oracle
from attention_rope_causal_gb300 import binding, build

pytestmark = pytest.mark.gpu

MANT = {torch.bfloat16: 7, torch.float16: 10}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def ulp(x: np.ndarray, dtype) -> np.ndarray:
    m = MANT[dtype]
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 1e-30)))
    min_exp = -126 if dtype == torch.bfloat16 else -14
    return np.exp2(np.maximum(e, min_exp) - m)


@pytest.mark.parametrize("B,N,H,d,dtype,base,sigma", [
    (1, 128, 2, 64, torch.bfloat16, 1e4, 1.0),
    (2, 2048, 16, 64, torch.bfloat16, 1e4, 1.0),
    (1, 4096, 32, 128, torch.bfloat16, 5e5, 1.0),
    (1, 4096, 8, 128, torch.float16, 5e5, 1.0),
    (3, 5500, 3, 64, torch.float16, 5e5, 1.0),
    (1, 32768, 2, 128, torch.float16, 5e5, 0.5),
    (2, 33, 9, 128, torch.bfloat16, 10.0, 3.0),
])
def test_rope_apply_matches_oracle(B, N, H, d, dtype, base, sigma):
    g = torch.Generator().manual_seed(B * 1000 + N + H)
    x = (torch.randn((B, N, H, d), generator=g) * sigma).to(dtype)
    y = binding.rope_apply(x.cuda(), base).cpu()
    assert binding.device_status() == 0
    ref = oracle.rope_rotate(x, base, positions=np.tile(np.arange(N, dtype=np.float64), B).reshape(B * N))
    ref = ref.reshape(B, N, H, d)
    err = np.abs(y.double().numpy() - ref)
    xd = x.double().numpy()
    half = d // 2
    pair = np.abs(xd) + np.abs(np.concatenate([xd[..., half:], xd[..., :half]], axis=-1))
    bound = ulp(ref, dtype) + 2.0 ** -20 * pair
    worst = float((err / bound).max())
    assert worst <= 1.0, f"max error {worst:.3f} of the bound"
    # and most elements are correctly rounded or one ulp off
    assert float((err <= ulp(ref, dtype)).mean()) > 0.999


def test_rope_apply_in_place():
    g = torch.Generator().manual_seed(7)
    x = torch.randn((2, 300, 5, 128), generator=g).to(torch.bfloat16).cuda()
    y = binding.rope_apply(x, 5e5)
    x2 = x.clone()
    binding.rope_apply(x2, 5e5, out=x2)
    torch.cuda.synchronize()
    assert torch.equal(x2, y)
