"""Pins for the oracle's backward pass (gradients of L = sum(dout * out) with respect to q, k, v
through the causal softmax attention and the RoPE rotation).  Checked against central finite
differences of the oracle's *forward* pass (a different code path: the forward never forms a
derivative), against torch autograd in fp64 over RoPE written as complex multiplication and
torch's scaled_dot_product_attention, and against closed forms -- never against the backward's own
code path.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _loss(q, k, v, dout, base, **kw):
    out, _ = oracle.rope_causal(q, k, v, base, **kw)
    return float((out * dout).sum())


@pytest.mark.parametrize("Hq,Hkv,d,r,il,pos", [(2, 1, 8, None, False, False), (4, 2, 16, None, False, False),
                                               (2, 2, 16, 8, True, False), (2, 1, 8, None, False, True),
                                               (2, 2, 16, 8, False, True)])
def test_gradients_match_finite_differences_of_the_forward(Hq, Hkv, d, r, il, pos):
    B, N, base = 2, 7, 100.0
    q, k, v = _rand((B, N, Hq, d), 1), _rand((B, N, Hkv, d), 2), _rand((B, N, Hkv, d), 3)
    dout = _rand((B, N, Hq, d), 4)
    kw = dict(rotary_dim=r, interleaved=il)
    if pos:  # explicit rotation positions (any integers), different per batch entry
        rng0 = np.random.default_rng(30)
        kw.update(q_positions=rng0.integers(-50, 300, size=(B, N)), k_positions=rng0.integers(-50, 300, size=(B, N)))
    dq, dk, dv = oracle.rope_causal_bwd(q, k, v, dout, base, **kw)
    eps = 1e-6
    rng = np.random.default_rng(5)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            lp = _loss(**{**args, name: xp}, dout=dout, base=base, **kw)
            lm = _loss(**{**args, name: xm}, dout=dout, base=base, **kw)
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - g[idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


def _rope_torch(x, base):
    """RoPE (half-split pairs) as complex multiplication, differentiable.  x: [B, N, H, d]."""
    B, N, H, d = x.shape
    h = d // 2
    theta = base ** (-2.0 * torch.arange(h, dtype=torch.float64) / d)
    ang = torch.arange(N, dtype=torch.float64)[:, None] * theta[None, :]  # [N, h]
    z = torch.complex(x[..., :h], x[..., h:]) * torch.polar(torch.ones_like(ang), ang)[None, :, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


def test_gradients_match_torch_autograd():
    B, N, Hq, Hkv, d, base = 2, 33, 4, 2, 16, 1e4
    q = torch.tensor(_rand((B, N, Hq, d), 6), requires_grad=True)
    k = torch.tensor(_rand((B, N, Hkv, d), 7), requires_grad=True)
    v = torch.tensor(_rand((B, N, Hkv, d), 8), requires_grad=True)
    dout = torch.tensor(_rand((B, N, Hq, d), 9))
    g = Hq // Hkv
    qr = _rope_torch(q, base).transpose(1, 2)
    kr = _rope_torch(k, base).repeat_interleave(g, dim=2).transpose(1, 2)
    vr = v.repeat_interleave(g, dim=2).transpose(1, 2)
    out = torch.nn.functional.scaled_dot_product_attention(qr, kr, vr, is_causal=True).transpose(1, 2)
    (out * dout).sum().backward()
    dq, dk, dv = oracle.rope_causal_bwd(q.detach().numpy(), k.detach().numpy(), v.detach().numpy(), dout.numpy(), base)
    np.testing.assert_allclose(dq, q.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, k.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, v.grad.numpy(), rtol=0, atol=1e-11)


def test_constant_values_give_zero_query_and_key_gradients():
    # v_j = c for every key: out_i = c whatever the scores, so dq = dk = 0; dv_j = sum_i P_ij dout_i
    # with sum_j dv_j = sum_i dout_i (each row of P sums to 1).
    B, N, d = 1, 12, 8
    q, k = _rand((B, N, 2, d), 10), _rand((B, N, 1, d), 11)
    v = np.broadcast_to(_rand((1, 1, 1, d), 12), (B, N, 1, d)).copy()
    dout = _rand((B, N, 2, d), 13)
    dq, dk, dv = oracle.rope_causal_bwd(q, k, v, dout, 1e4)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    np.testing.assert_allclose(dv.sum(axis=1)[:, 0], dout.sum(axis=(1, 2)), rtol=0, atol=1e-12)


def test_zero_queries_give_uniform_weights():
    # q = 0: P_ij = 1/(i+1) for j <= i, so dv_j = sum_{i >= j} dout_i / (i + 1) (summed over the heads)
    B, N, d = 1, 10, 8
    q = np.zeros((B, N, 2, d))
    k, v, dout = _rand((B, N, 1, d), 14), _rand((B, N, 1, d), 15), _rand((B, N, 2, d), 16)
    _, _, dv = oracle.rope_causal_bwd(q, k, v, dout, 1e4)
    for j in range(N):
        want = sum(dout[0, i].sum(axis=0) / (i + 1) for i in range(j, N))
        np.testing.assert_allclose(dv[0, j, 0], want, rtol=0, atol=1e-13)


def test_row_selection_equals_the_full_run():
    B, N, d = 2, 20, 16
    q, k, v, dout = _rand((B, N, 4, d), 17), _rand((B, N, 2, d), 18), _rand((B, N, 2, d), 19), _rand((B, N, 4, d), 20)
    dq, dk, dv = oracle.rope_causal_bwd(q, k, v, dout, 1e4)
    qs, ks = [0, 7, 19, 3], [19, 0, 11]
    sq, sk, sv = oracle.rope_causal_bwd(q, k, v, dout, 1e4, q_rows=qs, k_rows=ks)
    assert np.array_equal(sq, dq[:, qs]) and np.array_equal(sk, dk[:, ks]) and np.array_equal(sv, dv[:, ks])


def test_gqa_key_gradients_sum_the_group():
    # A KV head shared by g query heads receives the sum of the gradients the g heads would give it
    # with their own copy of the KV head (MHA with repeated K, V).
    B, N, d, g = 1, 9, 8, 3
    q, dout = _rand((B, N, g, d), 21), _rand((B, N, g, d), 22)
    k, v = _rand((B, N, 1, d), 23), _rand((B, N, 1, d), 24)
    _, dk, dv = oracle.rope_causal_bwd(q, k, v, dout, 1e4)
    _, dk_m, dv_m = oracle.rope_causal_bwd(q, np.repeat(k, g, axis=2), np.repeat(v, g, axis=2), dout, 1e4)
    np.testing.assert_allclose(dk[:, :, 0], dk_m.sum(axis=2), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv[:, :, 0], dv_m.sum(axis=2), rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# More keys than queries (a prefill against a cache): the Nq queries are the last Nq of Nk tokens.


@pytest.mark.parametrize("Nq,Nk,Hq,Hkv,d,r,il,pos", [(5, 9, 2, 1, 8, None, False, False), (1, 6, 4, 2, 16, None, False, False),
                                                     (3, 11, 2, 2, 16, 8, True, False), (4, 7, 2, 1, 8, None, False, True)])
def test_prefill_gradients_match_finite_differences(Nq, Nk, Hq, Hkv, d, r, il, pos):
    B, base = 2, 100.0
    q, k, v = _rand((B, Nq, Hq, d), 11), _rand((B, Nk, Hkv, d), 12), _rand((B, Nk, Hkv, d), 13)
    dout = _rand((B, Nq, Hq, d), 14)
    kw = dict(rotary_dim=r, interleaved=il)
    if pos:
        rng0 = np.random.default_rng(31)
        kw.update(q_positions=rng0.integers(-50, 300, size=(B, Nq)), k_positions=rng0.integers(-50, 300, size=(B, Nk)))
    dq, dk, dv = oracle.rope_causal_bwd(q, k, v, dout, base, **kw)
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape
    eps = 1e-6
    rng = np.random.default_rng(15)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            lp = _loss(**{**args, name: xp}, dout=dout, base=base, **kw)
            lm = _loss(**{**args, name: xm}, dout=dout, base=base, **kw)
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - g[idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


def _rope_torch_at(x, pos, base):
    """RoPE (half-split pairs) at the given token positions, as complex multiplication.  x: [B, N, H, d]."""
    B, N, H, d = x.shape
    h = d // 2
    theta = base ** (-2.0 * torch.arange(h, dtype=torch.float64) / d)
    ang = torch.as_tensor(pos, dtype=torch.float64)[:, None] * theta[None, :]
    z = torch.complex(x[..., :h], x[..., h:]) * torch.polar(torch.ones_like(ang), ang)[None, :, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


def test_prefill_gradients_match_torch_autograd():
    # queries at positions Nk - Nq + i, keys at j, query i sees keys j <= Nk - Nq + i (bottom-right)
    B, Nq, Nk, Hq, Hkv, d, base = 2, 13, 40, 4, 2, 16, 1e4
    q = torch.tensor(_rand((B, Nq, Hq, d), 16), requires_grad=True)
    k = torch.tensor(_rand((B, Nk, Hkv, d), 17), requires_grad=True)
    v = torch.tensor(_rand((B, Nk, Hkv, d), 18), requires_grad=True)
    dout = torch.tensor(_rand((B, Nq, Hq, d), 19))
    g, off = Hq // Hkv, Nk - Nq
    qr = _rope_torch_at(q, np.arange(off, Nk), base).transpose(1, 2)
    kr = _rope_torch_at(k, np.arange(Nk), base).repeat_interleave(g, dim=2).transpose(1, 2)
    vr = v.repeat_interleave(g, dim=2).transpose(1, 2)
    mask = torch.arange(Nk)[None, :] <= (off + torch.arange(Nq))[:, None]
    out = torch.nn.functional.scaled_dot_product_attention(qr, kr, vr, attn_mask=mask).transpose(1, 2)
    (out * dout).sum().backward()
    dq, dk, dv = oracle.rope_causal_bwd(q.detach().numpy(), k.detach().numpy(), v.detach().numpy(), dout.numpy(), base)
    np.testing.assert_allclose(dq, q.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, k.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, v.grad.numpy(), rtol=0, atol=1e-11)


def test_prefill_is_the_full_backward_with_zero_gradient_on_the_cached_rows():
    # With dout = 0 on the first Nk - Nq query rows of a full causal problem over Nk tokens, those
    # rows add nothing to any gradient, and the last Nq rows are the prefill's queries.
    B, Nq, Nk, Hq, Hkv, d, base = 1, 6, 20, 2, 1, 16, 1e4
    q, k, v = _rand((B, Nk, Hq, d), 20), _rand((B, Nk, Hkv, d), 21), _rand((B, Nk, Hkv, d), 22)
    dout = _rand((B, Nk, Hq, d), 23)
    dout[:, : Nk - Nq] = 0.0
    dq_full, dk_full, dv_full = oracle.rope_causal_bwd(q, k, v, dout, base)
    dq, dk, dv = oracle.rope_causal_bwd(q[:, Nk - Nq:], k, v, dout[:, Nk - Nq:], base)
    np.testing.assert_allclose(dq, dq_full[:, Nk - Nq:], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, dk_full, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dv_full, rtol=0, atol=1e-13)
    assert np.all(dq_full[:, : Nk - Nq] == 0.0)
