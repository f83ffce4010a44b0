"""Backward pass through the C ABI (attnfuse_rope_causal_bwd) against the oracle's fp64 gradients.

The GPU backward takes the GPU forward's out and lse (as a training step would) and rounds P and
dS to the input dtype for the products, like the forward rounds P.  Tolerance (per gradient
tensor): relative L2 <= 1e-2 (bf16) / 2e-3 (fp16) and max abs <= 2e-2 (bf16) / 5e-3 (fp16) times
max(1, max |reference|) -- the forward's bounds, carried over: the measured errors are about one
unit roundoff of the dtype in relative L2 (3.6e-3 bf16, 4.6e-4 fp16).
"""
import numpy as np
import pytest
import torch

import oracle
from attention_rope_causal_gb300 import binding, build, inputs

pytestmark = pytest.mark.gpu

BTOL = {"bf16": {"rel_l2": 1e-2, "max_abs": 2e-2}, "fp16": {"rel_l2": 2e-3, "max_abs": 5e-3}}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def _case(B, N, Hq, Hkv, d, dt, seed):
    w = inputs.Workload("case", B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, dtype=dt, rope_base=1e4, sigma=1.0, seed=seed)
    q, k, v = inputs.make_inputs(w)
    g = torch.Generator().manual_seed(seed + 1)
    dout = torch.randn(q.shape, generator=g).to(q.dtype)
    return q, k, v, dout


def _gpu_bwd(q, k, v, dout, base=1e4, mode="fused"):
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    o, l = binding.rope_causal_fwd(qc, kc, vc, base, mode=mode)
    dq, dk, dv = binding.rope_causal_bwd(qc, kc, vc, o, l, dc, base)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    return dq.cpu(), dk.cpu(), dv.cpu()


def assert_grad_close(x, ref, dt, label):
    x = x.double().numpy()
    err = x - ref
    assert not np.isnan(x).any(), label
    nref = np.linalg.norm(ref)
    if nref > 0:
        rel = np.linalg.norm(err) / nref
        assert rel <= BTOL[dt]["rel_l2"], f"{label}: rel_l2 {rel:.3e}"
    bound = BTOL[dt]["max_abs"] * max(1.0, float(np.abs(ref).max()))
    assert float(np.abs(err).max()) <= bound, f"{label}: max_abs {np.abs(err).max():.3e} > {bound:.3e}"


CASES = [
    # B, N, Hq, Hkv, d, dtype
    (1, 128, 2, 2, 64, "bf16"),
    (1, 300, 4, 2, 128, "bf16"),    # ragged last tile, GQA 2:1
    (1, 257, 2, 2, 64, "fp16"),     # ragged by one row
    (2, 128, 8, 2, 128, "bf16"),    # GQA 4:1, two batch entries
    (1, 1, 2, 1, 64, "bf16"),       # one token: dq = dk = 0, dv = dout summed over the group
    (1, 640, 4, 4, 128, "fp16"),    # several key and query tiles
    (1, 385, 6, 3, 64, "bf16"),     # odd group size
]


@pytest.mark.parametrize("B,N,Hq,Hkv,d,dt", CASES)
def test_backward_matches_oracle(B, N, Hq, Hkv, d, dt):
    q, k, v, dout = _case(B, N, Hq, Hkv, d, dt, seed=N + d + Hq)
    dq, dk, dv = _gpu_bwd(q, k, v, dout)
    rq, rk, rv = oracle.rope_causal_bwd(q, k, v, dout, 1e4)
    label = f"{B}x{N}x{Hq}/{Hkv}x{d} {dt}"
    assert_grad_close(dq, rq, dt, "dq " + label)
    assert_grad_close(dk, rk, dt, "dk " + label)
    assert_grad_close(dv, rv, dt, "dv " + label)


def test_backward_after_either_forward_mode():
    # The backward reads out and lse only; both forward modes give it the same function.
    q, k, v, dout = _case(1, 200, 4, 2, 128, "bf16", seed=3)
    a = _gpu_bwd(q, k, v, dout, mode="fused")
    b = _gpu_bwd(q, k, v, dout, mode="prerotate")
    for x, y in zip(a, b):
        err = (x.double() - y.double()).norm() / y.double().norm()
        assert float(err) <= BTOL["bf16"]["rel_l2"] / 4


def test_backward_llama_shape_sampled_rows():
    # B=1, Hq=32, Hkv=8, N=4096, d=128, bf16 (the forward benchmark's shape), checked on sampled
    # query rows (dq) and key rows (dk, dv) that include tile boundaries and the ends.
    w = inputs.LLAMA
    q, k, v = inputs.make_inputs(w)
    g = torch.Generator().manual_seed(11)
    dout = torch.randn(q.shape, generator=g).to(q.dtype)
    dq, dk, dv = _gpu_bwd(q, k, v, dout, base=w.rope_base)
    rng = np.random.default_rng(12)
    rows = sorted(set([0, 1, 127, 128, 129, 2047, 2048, 4095] + rng.integers(0, w.N, 24).tolist()))
    rq, rk, rv = oracle.rope_causal_bwd(q, k, v, dout, w.rope_base, q_rows=rows, k_rows=rows)
    assert_grad_close(dq[:, rows], rq, "bf16", "dq llama")
    assert_grad_close(dk[:, rows], rk, "bf16", "dk llama")
    assert_grad_close(dv[:, rows], rv, "bf16", "dv llama")


def test_backward_workspace_and_no_workspace_agree():
    q, k, v, dout = _case(1, 256, 4, 2, 64, "fp16", seed=21)
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    o, l = binding.rope_causal_fwd(qc, kc, vc, 1e4)
    a = binding.rope_causal_bwd(qc, kc, vc, o, l, dc, 1e4)
    ws = torch.empty(binding.bwd_workspace_bytes(1, 4, 2, 256, 64, torch.float16), dtype=torch.uint8, device="cuda")
    b = binding.rope_causal_bwd(qc, kc, vc, o, l, dc, 1e4, workspace=ws)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


VARIANTS = [
    # B, N, Hq, Hkv, d, dtype, rotary_dim, interleaved, explicit positions
    (1, 300, 4, 2, 128, "bf16", 64, False, False),
    (1, 257, 2, 2, 64, "fp16", None, True, False),
    (2, 200, 4, 1, 128, "bf16", None, False, True),
    (1, 390, 6, 3, 64, "fp16", 32, True, True),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,d,dt,r,il,pos", VARIANTS)
def test_backward_variants_and_positions_match_oracle(B, N, Hq, Hkv, d, dt, r, il, pos):
    # Other RoPE forms: the kernels return the gradients in the rotated frame and a pre-rotation
    # pass with the negated positions (R^T) rotates dq and dk back.
    q, k, v, dout = _case(B, N, Hq, Hkv, d, dt, seed=5 * N + d)
    qp = inputs.make_positions(B, N, seed=N) if pos else None
    kp = inputs.make_positions(B, N, seed=N + 1) if pos else None
    kw = dict(rotary_dim=r, interleaved=il)
    dev = dict(kw, q_positions=None if qp is None else qp.cuda(), k_positions=None if kp is None else kp.cuda())
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    o, l = binding.rope_causal_fwd(qc, kc, vc, 1e4, mode="prerotate", **dev)
    dq, dk, dv = binding.rope_causal_bwd(qc, kc, vc, o, l, dc, 1e4, **dev)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    rq, rk, rv = oracle.rope_causal_bwd(q, k, v, dout, 1e4, q_positions=None if qp is None else qp.numpy(),
                                        k_positions=None if kp is None else kp.numpy(), **kw)
    label = f"{B}x{N}x{Hq}/{Hkv}x{d} {dt} r={r} il={il} pos={pos}"
    assert_grad_close(dq.cpu(), rq, dt, "dq " + label)
    assert_grad_close(dk.cpu(), rk, dt, "dk " + label)
    assert_grad_close(dv.cpu(), rv, dt, "dv " + label)


def test_backward_explicit_index_positions_agree_with_the_default():
    # Same function, two routes: epilogue rotation (default) and the negated-position pass.  The pass
    # route rounds the rotated-frame gradient to bf16 once more before rotating it back, so the two
    # differ by about one bf16 rounding: within 2^-7 (one bf16 ulp, relative) in relative L2.
    q, k, v, dout = _case(1, 256, 4, 2, 128, "bf16", seed=77)
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    pos = torch.arange(256, dtype=torch.int32).reshape(1, 256).cuda()
    o, l = binding.rope_causal_fwd(qc, kc, vc, 1e4)
    a = binding.rope_causal_bwd(qc, kc, vc, o, l, dc, 1e4)
    b = binding.rope_causal_bwd(qc, kc, vc, o, l, dc, 1e4, q_positions=pos, k_positions=pos)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        err = (x.double() - y.double()).norm() / y.double().norm()
        assert float(err) <= 2.0 ** -7, float(err)


PREFILL = [
    # B, N, Nk, Hq, Hkv, d, dtype, rotary_dim, interleaved, explicit positions
    (1, 128, 256, 2, 2, 64, "bf16", None, False, False),    # offset a whole tile
    (1, 200, 333, 4, 2, 128, "bf16", None, False, False),   # ragged offset (133) and tails
    (2, 130, 517, 8, 2, 128, "fp16", None, False, False),   # offset 387, GQA 4:1, two batch entries
    (1, 1, 300, 4, 1, 64, "bf16", None, False, False),      # one query after 299 cached keys
    (1, 64, 1000, 6, 3, 64, "fp16", None, False, False),    # many key tiles every query sees in full
    (1, 190, 321, 4, 2, 128, "bf16", 64, False, False),     # partial rotary: the pass rotates back
    (1, 150, 290, 2, 1, 64, "fp16", None, True, True),      # interleaved pairs, explicit positions
]


@pytest.mark.parametrize("B,N,Nk,Hq,Hkv,d,dt,r,il,pos", PREFILL)
def test_backward_with_more_keys_than_queries_matches_oracle(B, N, Nk, Hq, Hkv, d, dt, r, il, pos):
    # The queries are the last N of the Nk tokens (query i sees keys j <= Nk - N + i): the backward
    # of a prefill that extends a cache.  The kernels start each key tile's query loop at the first
    # query tile that sees it and mask where the offset diagonal crosses a tile.
    q, k, v = inputs.make_kv_inputs(B, N, Nk, Hq, Hkv, d, dt, seed=N + Nk + d)
    g = torch.Generator().manual_seed(N + Nk)
    dout = torch.randn(q.shape, generator=g).to(q.dtype)
    qp = inputs.make_positions(B, N, seed=N) if pos else None
    kp = inputs.make_positions(B, Nk, seed=Nk) if pos else None
    kw = dict(rotary_dim=r, interleaved=il)
    dev = dict(kw, q_positions=None if qp is None else qp.cuda(), k_positions=None if kp is None else kp.cuda())
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    o, l = binding.rope_causal_fwd(qc, kc, vc, 1e4, mode="prerotate", **dev)
    dq, dk, dv = binding.rope_causal_bwd(qc, kc, vc, o, l, dc, 1e4, **dev)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert dk.shape == k.shape and dv.shape == v.shape
    rq, rk, rv = oracle.rope_causal_bwd(q, k, v, dout, 1e4, q_positions=None if qp is None else qp.numpy(),
                                        k_positions=None if kp is None else kp.numpy(), **kw)
    label = f"{B}x{N}/{Nk}x{Hq}/{Hkv}x{d} {dt} r={r} il={il} pos={pos}"
    assert_grad_close(dq.cpu(), rq, dt, "dq " + label)
    assert_grad_close(dk.cpu(), rk, dt, "dk " + label)
    assert_grad_close(dv.cpu(), rv, dt, "dv " + label)


def test_backward_prefill_is_the_full_backward_restricted_to_the_last_queries():
    # Nk tokens with zero dout on the first Nk - N queries: the full (N = Nk) backward gives the same
    # dk, dv as the prefill backward over the last N queries, and its dq rows there are the
    # prefill's dq.  Both routes on the GPU; the match is up to the two forwards' rounding of out.
    B, N, Nk, Hq, Hkv, d = 1, 170, 420, 4, 2, 128
    q_all, k, v = inputs.make_kv_inputs(B, Nk, Nk, Hq, Hkv, d, "bf16", seed=5)
    g = torch.Generator().manual_seed(6)
    dout_all = torch.randn(q_all.shape, generator=g).to(q_all.dtype)
    dout_all[:, : Nk - N] = 0
    qc, kc, vc = q_all.cuda(), k.cuda(), v.cuda()
    o, l = binding.rope_causal_fwd(qc, kc, vc, 1e4)
    fq, fk, fv = binding.rope_causal_bwd(qc, kc, vc, o, l, dout_all.cuda(), 1e4)
    qs, ds = qc[:, Nk - N:].contiguous(), dout_all[:, Nk - N:].contiguous().cuda()
    o2, l2 = binding.rope_causal_fwd(qs, kc, vc, 1e4)
    pq, pk, pv = binding.rope_causal_bwd(qs, kc, vc, o2, l2, ds, 1e4)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    for x, y, name in ((pq, fq[:, Nk - N:], "dq"), (pk, fk, "dk"), (pv, fv, "dv")):
        err = (x.double() - y.double()).norm() / y.double().norm()
        assert float(err) <= BTOL["bf16"]["rel_l2"] / 2, (name, float(err))

