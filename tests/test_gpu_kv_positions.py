"""The general causal form through the C ABI: more keys than queries (k, v hold Nk >= N tokens and
the queries are the last N of them, so query i sees keys j <= Nk - N + i: a prefill that extends a
cache, and N = 1 a decode step) and explicit int32 rotation positions for queries and keys, in the
pre-rotation pass and every attention mode, against the oracle's fp64 definition.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_rope_causal_gb300 import binding, build, inputs
from parity import TOL, assert_close, decode_path, errors

pytestmark = pytest.mark.gpu

MANT = {torch.bfloat16: 7, torch.float16: 10}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def ulp(x: np.ndarray, dtype) -> np.ndarray:
    m = MANT[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    min_exp = -126 if dtype == torch.bfloat16 else -14
    return np.exp2(np.maximum(e, min_exp) - m)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("d", [64, 128])
def test_rope_apply_positions_match_oracle(d, dtype):
    # one ulp at the exact value plus 2^-20 (|x_a| + |x_b|) for the pair's fp32 arithmetic, as for the
    # default positions
    B, N, H = 2, 333, 3
    g = torch.Generator().manual_seed(d)
    x = torch.randn((B, N, H, d), generator=g).to(dtype)
    pos = inputs.make_positions(B, N, seed=d + 1)
    y = binding.rope_apply(x.cuda(), 5e5, positions=pos.cuda()).cpu()
    assert binding.device_status() == 0
    ref = oracle.rope_rotate(x, 5e5, positions=pos.reshape(-1).numpy())
    xd = x.double().numpy()
    partner = np.concatenate([xd[..., d // 2:], xd[..., : d // 2]], axis=-1)
    bound = ulp(ref, dtype) + 2.0 ** -20 * (np.abs(xd) + np.abs(partner))
    err = np.abs(y.double().numpy() - ref)
    assert float((err / bound).max()) <= 1.0


def test_rope_apply_explicit_index_positions_are_bitwise_the_default():
    B, N, H, d = 2, 200, 4, 128
    g = torch.Generator().manual_seed(7)
    x = torch.randn((B, N, H, d), generator=g).to(torch.bfloat16).cuda()
    pos = torch.arange(N, dtype=torch.int32).repeat(B, 1).cuda()
    a = binding.rope_apply(x, 1e4)
    b = binding.rope_apply(x, 1e4, positions=pos)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def _check_both_modes(q, k, v, dt, label, **kw):
    qp, kp = kw.get("q_positions"), kw.get("k_positions")
    o_ref, l_ref = oracle.rope_causal(q, k, v, 1e4, rotary_dim=kw.get("rotary_dim"),
                                      interleaved=kw.get("interleaved", False),
                                      q_positions=None if qp is None else qp.numpy(),
                                      k_positions=None if kp is None else kp.numpy())
    dev = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in kw.items()}
    outs = {}
    for mode in ("fused", "prerotate", "split"):
        o, l = binding.rope_causal_fwd(q.cuda(), k.cuda(), v.cuda(), 1e4, mode=mode, **dev)
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        outs[mode] = (o.cpu(), l.cpu())
        assert_close(o.double().cpu().numpy(), l.double().cpu().numpy(), o_ref, l_ref, dt, f"{mode} {label}")
    t = TOL[dt]
    N, Hq, Hkv = q.shape[1], q.shape[2], k.shape[2]
    for m in ("fused", "split"):
        e = errors(outs[m][0].double().numpy(), outs[m][1].double().numpy(),
                   outs["prerotate"][0].double().numpy(), outs["prerotate"][1].double().numpy())
        rel = t["rel_l2"] / 4
        if m == "fused" and decode_path(q.shape[0], Hq, Hkv, N):
            # the fused call runs the split-KV decode kernels: they keep P in fp32 and sum in another
            # order, so the outputs differ by about one rounding of the output type
            rel = max(rel, 2.0 ** -7 if dt == "bf16" else 2.0 ** -10)
        assert e["max_abs"] <= t["max_abs"] / 4 and e["rel_l2"] <= rel, (m, e)
    return outs


KV = [
    # B, N, Nk, Hq, Hkv, d, dtype
    (1, 300, 377, 4, 2, 128, "bf16"),   # offset 77: two masked key tiles per query tile, head pairs
    (2, 128, 512, 8, 2, 128, "fp16"),   # offset 384 (a multiple of 128)
    (1, 1, 1000, 8, 2, 128, "bf16"),    # one decode step over 1000 keys
    (2, 1, 129, 4, 4, 64, "fp16"),      # decode, MHA (row-pair units), ragged key tail
    (1, 5, 4096, 4, 4, 64, "bf16"),     # short prefill after a long cache
    (1, 257, 700, 3, 3, 64, "fp16"),    # row-pair units, ragged queries and keys
    (1, 640, 640, 4, 2, 128, "bf16"),   # Nk == N through the _ex entry
]


@pytest.mark.parametrize("B,N,Nk,Hq,Hkv,d,dt", KV)
def test_more_keys_than_queries_match_oracle(B, N, Nk, Hq, Hkv, d, dt):
    q, k, v = inputs.make_kv_inputs(B, N, Nk, Hq, Hkv, d, dt, seed=N + Nk)
    _check_both_modes(q, k, v, dt, f"{B}x{N}/{Nk}x{Hq}/{Hkv}x{d} {dt}")


POS = [
    # B, N, Nk, Hq, Hkv, d, dtype, rotary_dim, interleaved
    (2, 300, 300, 4, 2, 128, "bf16", None, False),
    (1, 200, 450, 4, 4, 64, "fp16", None, False),
    (1, 129, 390, 8, 2, 128, "bf16", 64, True),
    (2, 64, 64, 2, 1, 64, "fp16", 32, False),
]


@pytest.mark.parametrize("B,N,Nk,Hq,Hkv,d,dt,r,il", POS)
def test_explicit_positions_match_oracle(B, N, Nk, Hq, Hkv, d, dt, r, il):
    q, k, v = inputs.make_kv_inputs(B, N, Nk, Hq, Hkv, d, dt, seed=3 * N + Nk)
    qp = inputs.make_positions(B, N, seed=N)
    kp = inputs.make_positions(B, Nk, seed=Nk + 1)
    _check_both_modes(q, k, v, dt, f"positions {B}x{N}/{Nk}x{Hq}/{Hkv}x{d} {dt} r={r} il={il}",
                      q_positions=qp, k_positions=kp, rotary_dim=r, interleaved=il)


def test_query_positions_only_and_key_positions_only():
    q, k, v = inputs.make_kv_inputs(1, 150, 400, 4, 2, 128, "bf16", seed=11)
    _check_both_modes(q, k, v, "bf16", "q positions only", q_positions=inputs.make_positions(1, 150, seed=12))
    _check_both_modes(q, k, v, "bf16", "k positions only", k_positions=inputs.make_positions(1, 400, seed=13))


def test_explicit_default_positions_agree_with_the_defaults():
    B, N, Nk = 1, 256, 600
    q, k, v = inputs.make_kv_inputs(B, N, Nk, 4, 2, 128, "bf16", seed=21)
    qp = torch.arange(Nk - N, Nk, dtype=torch.int32).reshape(1, N).cuda()
    kp = torch.arange(Nk, dtype=torch.int32).reshape(1, Nk).cuda()
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    for mode in ("fused", "prerotate", "split"):
        a, la = binding.rope_causal_fwd(qc, kc, vc, 1e4, mode=mode)
        b, lb = binding.rope_causal_fwd(qc, kc, vc, 1e4, mode=mode, q_positions=qp, k_positions=kp)
        torch.cuda.synchronize()
        if mode == "prerotate":
            # the pre-rotation pass computes every row's angle exactly either way
            assert torch.equal(a, b) and torch.equal(la, lb)
        else:
            # exact per-row cos/sin against the carried walk: far inside the oracle tolerance
            e = errors(a.double().cpu().numpy(), la.double().cpu().numpy(), b.double().cpu().numpy(),
                       lb.double().cpu().numpy())
            assert e["max_abs"] <= TOL["bf16"]["max_abs"] / 4 and e["rel_l2"] <= TOL["bf16"]["rel_l2"] / 4, e


def test_prefill_rows_equal_the_tail_of_full_attention():
    # The last N rows of causal attention over Nk tokens, computed as a prefill of N queries.
    B, N, Nk, Hq, Hkv, d = 1, 200, 520, 4, 2, 128
    q_full, k, v = inputs.make_kv_inputs(B, Nk, Nk, Hq, Hkv, d, "bf16", seed=31)
    qc, kc, vc = q_full.cuda(), k.cuda(), v.cuda()
    for mode in ("fused", "prerotate", "split"):
        full_o, full_l = binding.rope_causal_fwd(qc, kc, vc, 1e4, mode=mode)
        pre_o, pre_l = binding.rope_causal_fwd(qc[:, Nk - N:].contiguous(), kc, vc, 1e4, mode=mode)
        torch.cuda.synchronize()
        e = errors(pre_o.double().cpu().numpy(), pre_l.double().cpu().numpy(),
                   full_o[:, Nk - N:].double().cpu().numpy(), full_l[:, :, Nk - N:].double().cpu().numpy())
        assert e["max_abs"] <= TOL["bf16"]["max_abs"] / 4 and e["rel_l2"] <= TOL["bf16"]["rel_l2"] / 4, (mode, e)


def test_fewer_keys_than_queries_is_rejected():
    q, k, v = inputs.make_kv_inputs(1, 64, 64, 2, 2, 64, "bf16", seed=41)
    with pytest.raises(binding.AttnFuseError):
        binding.rope_causal_fwd(q.cuda(), k[:, :32].contiguous().cuda(), v[:, :32].contiguous().cuda(), 1e4)
