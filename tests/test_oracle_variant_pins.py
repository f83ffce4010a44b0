"""Pins for the oracle's RoPE variants: a rotary dimension r < d (only the first r entries
rotated, theta_k = base^(-2k/r)) and the interleaved pairing (2k, 2k+1).  Checked against explicit
rotation matrices built here, against the half-split form through a permutation of the head
dimensions (a permutation applied to q and k alike leaves every score, hence the attention output,
unchanged), and against identities that fix the untouched entries -- never against the oracle's
own code path.
"""
import math

import numpy as np
import pytest

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _rotation_matrix(m, d, r, interleaved, base):
    """Explicit d x d rotation at position m for the variant (r rotated entries, pairing)."""
    R = np.eye(d)
    for k in range(r // 2):
        th = m * base ** (-2.0 * k / r)
        c, s = math.cos(th), math.sin(th)
        a, b = (2 * k, 2 * k + 1) if interleaved else (k, k + r // 2)
        R[a, a], R[a, b] = c, -s
        R[b, a], R[b, b] = s, c
    return R


@pytest.mark.parametrize("d,r,interleaved", [(16, 16, True), (16, 8, False), (16, 8, True), (64, 32, False),
                                             (128, 64, True), (128, 32, False), (8, 2, True)])
def test_variant_rotation_matches_rotation_matrix(d, r, interleaved):
    base = 10000.0
    x = _rand((6, 2, d), 1)
    pos = np.array([0, 1, 7, 100, 4095, 32767], dtype=np.float64)
    got = oracle.rope_rotate(x, base, positions=pos, rotary_dim=r, interleaved=interleaved)
    for i, m in enumerate(pos):
        np.testing.assert_allclose(got[i], x[i] @ _rotation_matrix(m, d, r, interleaved, base).T, rtol=0, atol=1e-12)


def test_partial_rotation_leaves_the_tail_exactly():
    x = _rand((40, 3, 128), 2)
    got = oracle.rope_rotate(x, 500000.0, positions=np.arange(40) * 97.0, rotary_dim=32)
    assert np.array_equal(got[..., 32:], x[..., 32:])
    np.testing.assert_allclose(np.linalg.norm(got, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13, atol=0)


def test_full_rotary_dim_is_the_default_form():
    x = _rand((9, 2, 64), 3)
    pos = np.arange(9) * 13.0
    assert np.array_equal(oracle.rope_rotate(x, 1e4, positions=pos, rotary_dim=64),
                          oracle.rope_rotate(x, 1e4, positions=pos))


def _perm(d, r):
    """Index map taking the interleaved layout to the half-split layout on the first r entries:
    entry 2k -> k, 2k+1 -> k + r/2; entries >= r stay."""
    p = np.arange(d)
    p[: r // 2] = np.arange(0, r, 2)
    p[r // 2: r] = np.arange(1, r, 2)
    return p


@pytest.mark.parametrize("d,r", [(16, 16), (64, 32), (8, 4)])
def test_interleaved_equals_half_split_on_permuted_dims(d, r):
    # Rotation: interleaved(x)[perm] == half_split(x[perm]).
    x = _rand((5, 2, d), 4)
    pos = np.arange(5) * 31.0
    p = _perm(d, r)
    a = oracle.rope_rotate(x, 1e4, positions=pos, rotary_dim=r, interleaved=True)[..., p]
    b = oracle.rope_rotate(x[..., p], 1e4, positions=pos, rotary_dim=r, interleaved=False)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)
    # Attention: the same permutation of q's and k's head dimensions leaves the output unchanged.
    B, N, Hq, Hkv = 1, 11, 4, 2
    q, k, v = _rand((B, N, Hq, d), 5), _rand((B, N, Hkv, d), 6), _rand((B, N, Hkv, d), 7)
    oi, li = oracle.rope_causal(q, k, v, 1e4, rotary_dim=r, interleaved=True)
    oh, lh = oracle.rope_causal(q[..., p], k[..., p], v, 1e4, rotary_dim=r, interleaved=False)
    np.testing.assert_allclose(oi, oh, rtol=0, atol=1e-12)
    np.testing.assert_allclose(li, lh, rtol=0, atol=1e-12)


@pytest.mark.parametrize("r,interleaved", [(8, False), (8, True), (4, True)])
def test_variant_attention_matches_brute_force(r, interleaved):
    B, N, Hq, Hkv, d, base = 1, 13, 4, 2, 16, 10000.0
    q, k, v = _rand((B, N, Hq, d), 8), _rand((B, N, Hkv, d), 9), _rand((B, N, Hkv, d), 10)
    o, lse = oracle.rope_causal(q, k, v, base, rotary_dim=r, interleaved=interleaved)
    g = Hq // Hkv
    R = np.stack([_rotation_matrix(m, d, r, interleaved, base) for m in range(N)])
    mask = np.tril(np.ones((N, N), dtype=bool))
    for h in range(Hq):
        qr = np.einsum("mij,mj->mi", R, q[0, :, h])
        kr = np.einsum("mij,mj->mi", R, k[0, :, h // g])
        S = np.where(mask, qr @ kr.T / math.sqrt(d), -np.inf)
        mx = S.max(axis=1, keepdims=True)
        E = np.exp(S - mx)
        np.testing.assert_allclose(o[0, :, h], (E / E.sum(axis=1, keepdims=True)) @ v[0, :, h // g], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[0, h], mx[:, 0] + np.log(E.sum(axis=1)), rtol=0, atol=1e-12)


def test_rejects_bad_variants():
    x = _rand((2, 1, 16), 11)
    for r in (0, 3, 18, -2):
        with pytest.raises(RuntimeError):
            oracle.rope_rotate(x, 1e4, rotary_dim=r)
