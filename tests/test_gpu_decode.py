"""Few queries against many keys (decode, speculative decode): fused and auto calls with at most 16
query rows ((Hq / Hkv) N) per KV head run the split-KV decode kernels; every element is compared with
the oracle, and with the tile kernels (pre-rotate mode) on the same inputs."""
import pytest
import torch

import oracle
from attention_rope_causal_gb300 import binding, build, inputs
from parity import TOL, assert_close, decode_path, errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


CASES = [
    # B, N, Nk, Hq, Hkv, d, dtype, rotary_dim, interleaved, positions
    (1, 1, 4096, 32, 8, 128, "bf16", None, False, False),   # one decode step, Llama-3-8B heads
    (4, 1, 1000, 32, 8, 128, "fp16", None, False, False),   # ragged split tail, 32 KV heads
    (16, 1, 300, 8, 4, 128, "bf16", None, False, False),    # 64 KV heads, two slices, ragged last chunk
    (32, 1, 1024, 16, 4, 128, "bf16", None, False, False),  # 128 KV heads, one slice each
    (304, 1, 2304, 1, 1, 64, "bf16", None, False, False),   # one slice of 144 chunks, 18 per warp: the
                                                            # key cos/sin walk is exact again at chunk 16
    (2, 4, 777, 8, 2, 64, "bf16", None, False, False),      # speculative decode, 16 rows (the maximum)
    (1, 16, 2048, 16, 4, 128, "bf16", None, False, False),  # 64 rows per KV head: the tile kernels
    (1, 8, 300, 8, 8, 64, "fp16", None, False, False),      # MHA
    (1, 1, 1, 4, 1, 128, "bf16", None, False, False),       # a single key
    (1, 4, 770, 8, 2, 128, "bf16", None, False, False),     # last slice [768, 770): queries 0 and 1
                                                            # see none of its keys (empty partials)
    (2, 3, 500, 8, 2, 128, "bf16", 64, True, False),        # RoPE variant
    (2, 2, 640, 4, 2, 64, "fp16", None, False, True),       # explicit positions
    (2, 2, 500, 8, 4, 128, "bf16", 64, True, False),        # 4 rows, two queries (per-row masks), variant
    (1, 2, 1000, 16, 4, 128, "fp16", None, False, False),   # 8 rows: the most the 8-row form takes
    (3, 1, 2100, 8, 1, 128, "bf16", None, False, True),     # 8 heads per KV head, explicit positions
    # more than 16 (batch, KV head) pairs at d = 128 with at most 8 rows: the twelve-warp form
    (6, 2, 700, 16, 4, 128, "bf16", 96, True, True),        # per-row masks, variant, explicit positions
    (152, 1, 3300, 1, 1, 128, "bf16", None, False, False),  # one slice of 207 chunks, 17 or 18 per warp:
                                                            # the key cos/sin walk is exact again at 16
]


@pytest.mark.parametrize("B,N,Nk,Hq,Hkv,d,dt,r,il,pos", CASES)
def test_decode_matches_oracle(B, N, Nk, Hq, Hkv, d, dt, r, il, pos):
    q, k, v = inputs.make_kv_inputs(B, N, Nk, Hq, Hkv, d, dt, seed=N + Nk + d)
    qp = inputs.make_positions(B, N, seed=N) if pos else None
    kp = inputs.make_positions(B, Nk, seed=Nk) if pos else None
    kw = dict(rotary_dim=r, interleaved=il)
    dev = dict(kw, q_positions=None if qp is None else qp.cuda(), k_positions=None if kp is None else kp.cuda())
    o_ref, l_ref = oracle.rope_causal(q, k, v, 1e4, q_positions=None if qp is None else qp.numpy(),
                                      k_positions=None if kp is None else kp.numpy(), **kw)
    outs = {}
    for mode in ("fused", "auto", "prerotate"):
        o, l = binding.rope_causal_fwd(q.cuda(), k.cuda(), v.cuda(), 1e4, mode=mode, **dev)
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        outs[mode] = (o.cpu(), l.cpu())
        assert_close(o.double().cpu().numpy(), l.double().cpu().numpy(), o_ref, l_ref, dt,
                     f"{mode} {B}x{N}/{Nk}x{Hq}/{Hkv}x{d} {dt}")
    if decode_path(B, Hq, Hkv, N):  # both run the decode kernels
        assert torch.equal(outs["fused"][0], outs["auto"][0])
    # Against the tile kernels: those round P to the input type for P V and sum in another order,
    # so the two outputs differ by about one rounding of the output type (relative L2 within two
    # unit roundoffs: 2^-7 bf16, 2^-10 fp16), far inside the oracle tolerance.
    e = errors(outs["fused"][0].double().numpy(), outs["fused"][1].double().numpy(),
               outs["prerotate"][0].double().numpy(), outs["prerotate"][1].double().numpy())
    t = TOL[dt]
    assert e["max_abs"] <= t["max_abs"] / 4 and e["rel_l2"] <= max(t["rel_l2"] / 4, 2.0 ** -7 if dt == "bf16" else 2.0 ** -10), e


def test_decode_workspace_is_reported_and_used():
    B, N, Nk, Hq, Hkv, d = 2, 1, 3000, 32, 8, 128
    need = binding.workspace_bytes(B, Hq, Hkv, N, d, "fused", torch.bfloat16, kv_len=Nk)
    assert need > 0
    q, k, v = inputs.make_kv_inputs(B, N, Nk, Hq, Hkv, d, "bf16", seed=9)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    a, la = binding.rope_causal_fwd(q.cuda(), k.cuda(), v.cuda(), 1e4, mode="fused", workspace=ws)
    b, lb = binding.rope_causal_fwd(q.cuda(), k.cuda(), v.cuda(), 1e4, mode="fused")
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(la, lb)
