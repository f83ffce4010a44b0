"""The torch.autograd wrapper over the C ABI: a training-style step (loss.backward()) gives the
oracle's gradients, in every forward mode."""
import pytest
import torch

import oracle
from attention_rope_causal_gb300 import binding, build, inputs

pytestmark = pytest.mark.gpu

BTOL = {"bf16": 1e-2, "fp16": 2e-3}  # relative L2, as in the backward parity tests


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


@pytest.mark.parametrize("mode", ["fused", "prerotate", "split", "auto"])
@pytest.mark.parametrize("B,N,Hq,Hkv,d,dt,r,il", [(1, 300, 4, 2, 128, "bf16", None, False),
                                                  (2, 200, 4, 4, 64, "fp16", 32, True)])
def test_loss_backward_matches_oracle(mode, B, N, Hq, Hkv, d, dt, r, il):
    w = inputs.Workload("case", B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, dtype=dt, rope_base=1e4, sigma=1.0, seed=N)
    q, k, v = inputs.make_inputs(w)
    dout = torch.randn(q.shape, generator=torch.Generator().manual_seed(3)).to(q.dtype)
    qc, kc, vc = (t.cuda().requires_grad_(True) for t in (q, k, v))
    out = binding.rope_causal_attention(qc, kc, vc, 1e4, mode=mode, rotary_dim=r, interleaved=il)
    (out.float() * dout.cuda().float()).sum().backward()
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    ref = oracle.rope_causal_bwd(q, k, v, dout, 1e4, rotary_dim=r, interleaved=il)
    for name, g, rr in zip(("dq", "dk", "dv"), (qc.grad, kc.grad, vc.grad), ref):
        x = g.double().cpu().numpy()
        rel = ((x - rr) ** 2).sum() ** 0.5 / ((rr ** 2).sum() ** 0.5)
        assert rel <= BTOL[dt], (mode, name, rel)


@pytest.mark.parametrize("mode", ["fused", "auto"])
def test_loss_backward_with_a_cache_matches_oracle(mode):
    # k, v hold more tokens than q (a prefill that extends a cache: the queries are the last N of the
    # Nk tokens); the wrapper passes them through unchanged and the backward returns dk, dv over Nk.
    B, N, Nk, Hq, Hkv, d = 1, 150, 410, 8, 2, 128
    q, k, v = inputs.make_kv_inputs(B, N, Nk, Hq, Hkv, d, "bf16", seed=41)
    dout = torch.randn(q.shape, generator=torch.Generator().manual_seed(42)).to(q.dtype)
    qc, kc, vc = (t.cuda().requires_grad_(True) for t in (q, k, v))
    out = binding.rope_causal_attention(qc, kc, vc, 1e4, mode=mode)
    (out.float() * dout.cuda().float()).sum().backward()
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert kc.grad.shape == k.shape and vc.grad.shape == v.shape
    ref = oracle.rope_causal_bwd(q, k, v, dout, 1e4)
    for name, g, rr in zip(("dq", "dk", "dv"), (qc.grad, kc.grad, vc.grad), ref):
        x = g.double().cpu().numpy()
        rel = ((x - rr) ** 2).sum() ** 0.5 / ((rr ** 2).sum() ** 0.5)
        assert rel <= BTOL["bf16"], (mode, name, rel)
