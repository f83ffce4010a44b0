"""Pins for the oracle's general form: more keys than queries (Nk >= Nq, the queries being the last
Nq tokens, so query i sees keys j <= Nk - Nq + i) and explicit rotation positions for queries and
keys.  Checked against a brute-force evaluation built here from different primitives (RoPE as
multiplication of complex numbers by e^{i m theta}, attention through torch's fp64
scaled_dot_product_attention with an explicit boolean mask), against the plain causal case (a
prefill of Nq tokens equals the last Nq rows of causal attention over all Nk tokens), against
closed forms (q = 0 gives the mean of the visible values and lse = ln(count)), and against the
fact that RoPE scores depend on position differences only -- never against the oracle's own code
path.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _rope_complex(x, pos, base, r, interleaved):
    """RoPE by complex multiplication: plane (a, b) holds the complex number x_a + i x_b and is
    multiplied by exp(i * pos * theta_k), theta_k = base^(-2k/r).  x: [T, H, d], pos: [T]."""
    y = x.copy()
    for k in range(r // 2):
        a, b = (2 * k, 2 * k + 1) if interleaved else (k, k + r // 2)
        z = (x[:, :, a] + 1j * x[:, :, b]) * np.exp(1j * pos[:, None] * base ** (-2.0 * k / r))
        y[:, :, a], y[:, :, b] = z.real, z.imag
    return y


def _brute(q, k, v, base, qpos, kpos, r=None, interleaved=False):
    """q [B, Nq, Hq, d], k, v [B, Nk, Hkv, d] fp64; qpos [B, Nq], kpos [B, Nk]."""
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    r = d if r is None else r
    g = Hq // Hkv
    off = Nk - Nq
    out = np.zeros((B, Nq, Hq, d))
    lse = np.zeros((B, Hq, Nq))
    mask = torch.tensor(np.arange(Nk)[None, :] <= off + np.arange(Nq)[:, None])  # [Nq, Nk]
    for b in range(B):
        qr = torch.tensor(_rope_complex(q[b], qpos[b].astype(np.float64), base, r, interleaved))
        kr = torch.tensor(_rope_complex(k[b], kpos[b].astype(np.float64), base, r, interleaved))
        vb = torch.tensor(v[b])
        for h in range(Hq):
            qh, kh, vh = qr[:, h], kr[:, h // g], vb[:, h // g]
            o = torch.nn.functional.scaled_dot_product_attention(qh[None, None], kh[None, None], vh[None, None],
                                                                 attn_mask=mask)
            out[b, :, h] = o[0, 0].numpy()
            s = (qh @ kh.T) / math.sqrt(d)
            lse[b, h] = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1).numpy()
    return out, lse


@pytest.mark.parametrize("Nq,Nk,Hq,Hkv,d,r,il", [(5, 9, 4, 2, 8, None, False), (1, 7, 2, 1, 8, None, False),
                                                 (6, 6, 2, 2, 16, 8, True), (3, 11, 3, 1, 16, None, True)])
def test_positions_and_key_offset_match_brute_force(Nq, Nk, Hq, Hkv, d, r, il):
    B, base = 2, 10000.0
    q, k, v = _rand((B, Nq, Hq, d), 1), _rand((B, Nk, Hkv, d), 2), _rand((B, Nk, Hkv, d), 3)
    rng = np.random.default_rng(4)
    qpos = rng.integers(-5000, 40000, size=(B, Nq))
    kpos = rng.integers(-5000, 40000, size=(B, Nk))
    out, lse = oracle.rope_causal(q, k, v, base, rotary_dim=r, interleaved=il, q_positions=qpos, k_positions=kpos)
    bo, bl = _brute(q, k, v, base, qpos, kpos, r, il)
    np.testing.assert_allclose(out, bo, rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-11)


def test_default_positions_match_brute_force():
    B, Nq, Nk, d, base = 2, 4, 10, 8, 500000.0
    q, k, v = _rand((B, Nq, 2, d), 5), _rand((B, Nk, 1, d), 6), _rand((B, Nk, 1, d), 7)
    out, lse = oracle.rope_causal(q, k, v, base)
    qpos = np.tile(np.arange(Nk - Nq, Nk), (B, 1))
    kpos = np.tile(np.arange(Nk), (B, 1))
    bo, bl = _brute(q, k, v, base, qpos, kpos)
    np.testing.assert_allclose(out, bo, rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-11)


def test_prefill_is_the_tail_of_full_causal_attention():
    B, Nq, Nk, Hq, Hkv, d = 2, 37, 300, 4, 2, 16
    k, v = _rand((B, Nk, Hkv, d), 8), _rand((B, Nk, Hkv, d), 9)
    q_full = _rand((B, Nk, Hq, d), 10)
    full_o, full_l = oracle.rope_causal(q_full, k, v, 1e4)
    pre_o, pre_l = oracle.rope_causal(np.ascontiguousarray(q_full[:, Nk - Nq:]), k, v, 1e4)
    assert np.array_equal(pre_o, full_o[:, Nk - Nq:])
    assert np.array_equal(pre_l, full_l[:, :, Nk - Nq:])


def test_explicit_default_positions_are_the_defaults():
    B, Nq, Nk, d = 2, 20, 50, 32
    q, k, v = _rand((B, Nq, 2, d), 11), _rand((B, Nk, 2, d), 12), _rand((B, Nk, 2, d), 13)
    a = oracle.rope_causal(q, k, v, 1e4)
    b = oracle.rope_causal(q, k, v, 1e4, q_positions=np.tile(np.arange(Nk - Nq, Nk), (B, 1)),
                           k_positions=np.tile(np.arange(Nk), (B, 1)))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_scores_depend_on_position_differences_only():
    B, Nq, Nk, d = 1, 16, 40, 32
    q, k, v = _rand((B, Nq, 2, d), 14), _rand((B, Nk, 1, d), 15), _rand((B, Nk, 1, d), 16)
    rng = np.random.default_rng(17)
    qpos, kpos = rng.integers(0, 3000, size=(B, Nq)), rng.integers(0, 3000, size=(B, Nk))
    a = oracle.rope_causal(q, k, v, 1e4, q_positions=qpos, k_positions=kpos)
    b = oracle.rope_causal(q, k, v, 1e4, q_positions=qpos + 12345, k_positions=kpos + 12345)
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-9)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-9)
    # and a shift of the query positions alone does change them
    c = oracle.rope_causal(q, k, v, 1e4, q_positions=qpos + 7, k_positions=kpos)
    assert np.abs(a[0] - c[0]).max() > 1e-3


@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 33), (7, 7), (7, 20), (64, 200)])
def test_zero_queries_average_the_visible_values(Nq, Nk):
    # q = 0: every visible score is 0, so query i averages v_0 .. v_{Nk-Nq+i} and lse = ln(Nk-Nq+i+1)
    B, d = 2, 16
    q = np.zeros((B, Nq, 2, d))
    k, v = _rand((B, Nk, 1, d), 18), _rand((B, Nk, 1, d), 19)
    out, lse = oracle.rope_causal(q, k, v, 1e4)
    for i in range(Nq):
        last = Nk - Nq + i
        for h in range(2):
            np.testing.assert_allclose(out[:, i, h], v[:, :last + 1, 0].mean(axis=1), rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse[:, h, i], math.log(last + 1), rtol=0, atol=1e-13)


def test_rejects_fewer_keys_than_queries_and_bad_position_shapes():
    q, k, v = _rand((1, 8, 1, 8), 20), _rand((1, 4, 1, 8), 21), _rand((1, 4, 1, 8), 22)
    with pytest.raises(ValueError):
        oracle.rope_causal(q, k, v, 1e4)
    k, v = _rand((1, 8, 1, 8), 21), _rand((1, 8, 1, 8), 22)
    with pytest.raises(ValueError):
        oracle.rope_causal(q, k, v, 1e4, q_positions=np.arange(7))
    with pytest.raises(ValueError):
        oracle.rope_causal(q, k, v, 1e4, k_positions=np.arange(9))
