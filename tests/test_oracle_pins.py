"""Pins for the CPU oracle: checks it against mathematics the pages and the RoPE definition fix,
never against itself.  Each test is chosen so that a plausible slip in the oracle (wrong pairing,
wrong frequency, wrong sign, missing scale, off-by-one in the causal mask, wrong GQA mapping, wrong
log-sum-exp units) fails at least one of them.

The RoPE definition pinned here is the one this library fixes (the pages name RoPE only, as a
pre-multiplication transform: "AttnFuse Makes RoPE a First-Class Attention Compilation Operation",
2026-09-13 AI papers report, paragraph 1): half-split pairs (k, k+d/2), theta_k = base^(-2k/d),
position = token index.  Causal masking and softmax: same report, paragraph 2.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed, dtype=np.float64):
    return np.random.default_rng(seed).standard_normal(shape).astype(dtype)


# ----------------------------------------------------------------------------------------------
# Decoding of 16-bit inputs (library cross-check against torch's own widening)


@pytest.mark.parametrize("tdtype", [torch.bfloat16, torch.float16])
def test_decode_and_position_zero_identity(tdtype):
    # Every finite 16-bit pattern, rotated at position 0, must come back as its exact fp64 value:
    # pins the decoder (normals, subnormals, signed zero) and that position 0 is the identity.
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    x = bits.view(tdtype)
    finite = torch.isfinite(x)
    x = x[finite]
    n = (x.numel() // 64) * 64
    x = x[:n].reshape(-1, 1, 64)
    got = oracle.rope_rotate(x, base=10000.0, positions=np.zeros(x.shape[0]))
    want = x.double().numpy()
    assert np.array_equal(got, want)


# ----------------------------------------------------------------------------------------------
# Rotation: closed forms


def test_rotation_d2_is_complex_multiplication():
    # d = 2: one pair, theta_0 = base^0 = 1, so RoPE at position m multiplies x0 + i x1 by e^{i m}.
    x = _rand((50, 1, 2), 1)
    pos = np.arange(50, dtype=np.float64) * 37.0 + 5.0
    got = oracle.rope_rotate(x, base=500000.0, positions=pos)
    z = (x[:, 0, 0] + 1j * x[:, 0, 1]) * np.exp(1j * pos)
    np.testing.assert_allclose(got[:, 0, 0], z.real, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got[:, 0, 1], z.imag, rtol=0, atol=1e-12)


@pytest.mark.parametrize("d,base,k,pos,angle", [
    (64, 10000.0, 16, 100.0, 1.0),      # theta_{d/4} = base^(-1/2) = 0.01 -> 100 * 0.01 = 1 rad
    (64, 10000.0, 0, 3.0, 3.0),         # theta_0 = 1
    (128, 500000.0, 32, 1414.0, 1414.0 / math.sqrt(500000.0)),   # theta_{d/4} = 1/sqrt(base)
    (128, 10000.0, 48, 1000.0, 1.0),    # theta_{3d/8} = base^(-3/4) = 1e-3
])
def test_rotation_unit_vector_closed_form(d, base, k, pos, angle):
    # e_k at position p goes to cos(p theta_k) e_k + sin(p theta_k) e_{k+d/2}; e_{k+d/2} goes to
    # -sin e_k + cos e_{k+d/2}.  Pins pairing (k, k+d/2), the frequency and the sign convention.
    x = np.zeros((2, 1, d))
    x[0, 0, k] = 1.0
    x[1, 0, k + d // 2] = 1.0
    got = oracle.rope_rotate(x, base=base, positions=[pos, pos])
    want = np.zeros((2, 1, d))
    want[0, 0, k], want[0, 0, k + d // 2] = math.cos(angle), math.sin(angle)
    want[1, 0, k], want[1, 0, k + d // 2] = -math.sin(angle), math.cos(angle)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_rotation_matches_block_rotation_matrix():
    # Brute force: R(m) as an explicit d x d matrix whose planes are (k, k+d/2).
    d, base = 16, 10000.0
    x = _rand((7, 3, d), 2)
    pos = np.array([0, 1, 2, 5, 100, 4095, 32767], dtype=np.float64)
    got = oracle.rope_rotate(x, base=base, positions=pos)
    for r, m in enumerate(pos):
        R = np.zeros((d, d))
        for k in range(d // 2):
            th = m * base ** (-2.0 * k / d)
            c, s = math.cos(th), math.sin(th)
            R[k, k], R[k, k + d // 2] = c, -s
            R[k + d // 2, k], R[k + d // 2, k + d // 2] = s, c
        np.testing.assert_allclose(got[r], x[r] @ R.T, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------------------------
# Rotation: invariants


def test_rotation_preserves_norm():
    x = _rand((64, 4, 128), 3)
    pos = np.arange(64, dtype=np.float64) * 517.0
    got = oracle.rope_rotate(x, base=500000.0, positions=pos)
    np.testing.assert_allclose(np.linalg.norm(got, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13, atol=0)


def test_rotation_composes():
    # R(a) R(b) = R(a + b)
    x = _rand((9, 2, 64), 4)
    a = np.arange(9, dtype=np.float64) * 11.0
    b = np.arange(9, dtype=np.float64) * 7.0 + 3.0
    two_step = oracle.rope_rotate(oracle.rope_rotate(x, 10000.0, positions=b), 10000.0, positions=a)
    one_step = oracle.rope_rotate(x, 10000.0, positions=a + b)
    np.testing.assert_allclose(two_step, one_step, rtol=0, atol=1e-11)


def test_rotated_dot_depends_only_on_offset():
    # q'_m . k'_n = q'_{m+s} . k'_{n+s}: shifting both positions leaves the score unchanged.
    d = 128
    q = _rand((1, 1, d), 5)
    k = _rand((1, 1, d), 6)
    for (m, n) in [(0, 0), (10, 3), (3, 10), (4095, 17)]:
        ref = None
        for s in (0, 1, 1000, 20000):
            qm = oracle.rope_rotate(q, 500000.0, positions=[m + s])[0, 0]
            kn = oracle.rope_rotate(k, 500000.0, positions=[n + s])[0, 0]
            dot = float(qm @ kn)
            if ref is None:
                ref = dot
            assert abs(dot - ref) < 1e-9 * max(1.0, abs(ref))


# ----------------------------------------------------------------------------------------------
# Attention


def _brute_force(q, k, v, base):
    """Independent brute force: explicit rotation matrices, full N x N scores, explicit mask."""
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    R = np.zeros((N, d, d))
    for m in range(N):
        for kk in range(d // 2):
            th = m * base ** (-2.0 * kk / d)
            c, s = math.cos(th), math.sin(th)
            R[m, kk, kk], R[m, kk, kk + d // 2] = c, -s
            R[m, kk + d // 2, kk], R[m, kk + d // 2, kk + d // 2] = s, c
    out = np.zeros((B, N, Hq, d))
    lse = np.zeros((B, Hq, N))
    mask = np.tril(np.ones((N, N), dtype=bool))
    for b in range(B):
        for h in range(Hq):
            qr = np.einsum("mij,mj->mi", R, q[b, :, h])
            kr = np.einsum("mij,mj->mi", R, k[b, :, h // g])
            S = qr @ kr.T / math.sqrt(d)
            S = np.where(mask, S, -np.inf)
            mx = S.max(axis=1, keepdims=True)
            E = np.exp(S - mx)
            P = E / E.sum(axis=1, keepdims=True)
            out[b, :, h] = P @ v[b, :, h // g]
            lse[b, h] = mx[:, 0] + np.log(E.sum(axis=1))
    return out, lse


@pytest.mark.parametrize("B,Hq,Hkv,N,d", [(1, 1, 1, 1, 2), (2, 4, 2, 16, 8), (1, 6, 3, 9, 4), (1, 2, 1, 13, 16)])
def test_attention_matches_brute_force(B, Hq, Hkv, N, d):
    q = _rand((B, N, Hq, d), 10)
    k = _rand((B, N, Hkv, d), 11)
    v = _rand((B, N, Hkv, d), 12)
    o, lse = oracle.rope_causal(q, k, v, base=10000.0)
    ob, lb = _brute_force(q, k, v, 10000.0)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-12)


def test_attention_matches_torch_sdpa_on_rotated_inputs():
    # Library cross-check: torch's scaled_dot_product_attention (fp64, is_causal) on q', k' rotated by
    # the oracle's rotation, GQA expanded with repeat_interleave (head h -> kv head floor(h/g)).
    B, N, Hq, Hkv, d, base = 2, 40, 8, 2, 32, 500000.0
    q = _rand((B, N, Hq, d), 20)
    k = _rand((B, N, Hkv, d), 21)
    v = _rand((B, N, Hkv, d), 22)
    o, lse = oracle.rope_causal(q, k, v, base=base)
    qr = torch.from_numpy(oracle.rope_rotate_bnhd(q, base)).transpose(1, 2)
    kr = torch.from_numpy(oracle.rope_rotate_bnhd(k, base)).transpose(1, 2)
    vt = torch.from_numpy(v).transpose(1, 2)
    g = Hq // Hkv
    kr, vt = kr.repeat_interleave(g, dim=1), vt.repeat_interleave(g, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(qr, kr, vt, is_causal=True)
    np.testing.assert_allclose(o, ref.transpose(1, 2).numpy(), rtol=0, atol=1e-12)
    S = (qr @ kr.transpose(-1, -2)) / math.sqrt(d)
    S = S.masked_fill(~torch.tril(torch.ones(N, N, dtype=torch.bool)), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(S, dim=-1).numpy(), rtol=0, atol=1e-12)


def test_zero_queries_give_uniform_causal_average():
    # q = 0: every visible score is 0, so o_i is the mean of v_0..v_i and lse_i = ln(i+1).
    B, N, Hq, Hkv, d = 1, 33, 4, 2, 16
    q = np.zeros((B, N, Hq, d))
    k = _rand((B, N, Hkv, d), 30)
    v = _rand((B, N, Hkv, d), 31)
    o, lse = oracle.rope_causal(q, k, v, base=10000.0)
    csum = np.cumsum(v, axis=1) / np.arange(1, N + 1)[None, :, None, None]
    np.testing.assert_allclose(o, np.repeat(csum, Hq // Hkv, axis=2), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, N + 1)), lse.shape), rtol=0, atol=1e-13)


def test_constant_values_give_constant_output():
    B, N, Hq, Hkv, d = 1, 20, 2, 1, 8
    q = _rand((B, N, Hq, d), 40) * 3
    k = _rand((B, N, Hkv, d), 41) * 3
    v = np.broadcast_to(np.linspace(-1, 1, d), (B, N, Hkv, d)).copy()
    o, _ = oracle.rope_causal(q, k, v, base=10000.0)
    np.testing.assert_allclose(o, np.broadcast_to(v[:, :, :1], o.shape[:2] + (1, d)).repeat(Hq, 2), atol=1e-14)


def test_one_hot_values_expose_probability_rows():
    # v_j = e_j turns o_i into the probability row P_i: rows sum to 1, and P_ij = 0 exactly for j > i
    # (the causal mask).  Row 0 attends to key 0 only: o_0 = v_0, and lse_0 = s_00 = q_0.k_0/sqrt(d)
    # because position 0 is the identity rotation.
    B, N, H, d = 1, 24, 1, 32
    q = _rand((B, N, H, d), 50) * 2
    k = _rand((B, N, H, d), 51) * 2
    v = np.zeros((B, N, H, d))
    for j in range(N):
        v[0, j, 0, j] = 1.0
    o, lse = oracle.rope_causal(q, k, v, base=10000.0)
    P = o[0, :, 0, :N]
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-13)
    assert np.all(P[np.triu_indices(N, 1)] == 0.0)
    assert np.all(P[np.tril_indices(N)] > 0.0)
    assert np.array_equal(o[0, 0, 0], v[0, 0, 0])
    assert abs(lse[0, 0, 0] - float(q[0, 0, 0] @ k[0, 0, 0]) / math.sqrt(d)) < 1e-14


def test_gqa_equals_mha_with_repeated_kv_heads():
    B, N, Hq, Hkv, d = 2, 17, 8, 2, 16
    q = _rand((B, N, Hq, d), 60)
    k = _rand((B, N, Hkv, d), 61)
    v = _rand((B, N, Hkv, d), 62)
    og, lg = oracle.rope_causal(q, k, v, base=10000.0)
    om, lm = oracle.rope_causal(q, np.repeat(k, Hq // Hkv, axis=2), np.repeat(v, Hq // Hkv, axis=2), base=10000.0)
    assert np.array_equal(og, om) and np.array_equal(lg, lm)
    # and the kv heads really differ, so a wrong mapping would show
    assert not np.allclose(og[:, :, 0], og[:, :, Hq - 1])


def test_row_subset_equals_full():
    B, N, Hq, Hkv, d = 2, 50, 4, 4, 16
    q, k, v = (_rand((B, N, h, d), 70 + i) for i, h in enumerate((Hq, Hkv, Hkv)))
    of, lf = oracle.rope_causal(q, k, v, base=10000.0)
    rows = [49, 0, 17, 17, 31]
    os_, ls = oracle.rope_causal(q, k, v, base=10000.0, rows=rows)
    assert np.array_equal(os_, of[:, rows]) and np.array_equal(ls, lf[:, :, rows])


@pytest.mark.parametrize("tdtype", [torch.bfloat16, torch.float16])
def test_16bit_inputs_equal_fp64_of_decoded_values(tdtype):
    g = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn(shape, generator=g).to(tdtype) for shape in ((1, 30, 4, 64), (1, 30, 2, 64), (1, 30, 2, 64)))
    o16, l16 = oracle.rope_causal(q, k, v, base=10000.0)
    o64, l64 = oracle.rope_causal(q.double(), k.double(), v.double(), base=10000.0)
    assert np.array_equal(o16, o64) and np.array_equal(l16, l64)


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.rope_causal(np.zeros((1, 4, 3, 8)), np.zeros((1, 4, 2, 8)), np.zeros((1, 4, 2, 8)), 10000.0)
    with pytest.raises(ValueError):
        oracle.rope_causal(np.zeros((1, 4, 2, 8)), np.zeros((1, 4, 2, 8)), np.zeros((1, 4, 2, 8)), 10000.0,
                           rows=[4])
