"""Attention forward (attnfuse_rope_causal_fwd, both modes) against the fp64 oracle.

Small problems, the MHA workload (2x16x2048 d64) and the Llama-3-8B GQA workload (1x32/8x4096 d128,
the benchmark's default) are compared on every output element; the crossover sweep and the 32k
context are compared on sampled query rows (first rows, every 128-row tile boundary +-1, the last
tile, random rows) computed by the oracle one by one, at the same launch configuration the
benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_rope_causal_gb300 import binding, build, inputs
from parity import TOL, assert_close, dtype_name, errors, sample_rows

pytestmark = pytest.mark.gpu

# fused: Q and K rotated on chip; prerotate: both rotated by a pass first; split: K by a pass, Q on chip
MODES = ["fused", "prerotate", "split"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def run_gpu(q, k, v, base, mode):
    out, lse = binding.rope_causal_fwd(q.cuda(), k.cuda(), v.cuda(), base, mode=mode)
    torch.cuda.synchronize()
    st = binding.device_status()
    assert st == 0, f"device status {st}: {binding.last_error()}"
    return out.cpu(), lse.cpu()


def draw(B, N, Hq, Hkv, d, dtype, seed, sigma=1.0):
    w = inputs.Workload("case", B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, dtype=dtype, rope_base=1e4, sigma=sigma, seed=seed)
    return inputs.make_inputs(w)


# ---------------------------------------------------------------------------------------------
# Full comparison on small and ragged problems


SMALL = [
    # B, N, Hq, Hkv, d, dtype
    (1, 128, 2, 2, 64, "bf16"),     # the tiny workload's shape
    (1, 1, 1, 1, 64, "bf16"),       # a single row
    (1, 2, 1, 1, 128, "fp16"),
    (2, 127, 4, 1, 128, "bf16"),    # ragged last tile
    (1, 129, 2, 2, 64, "fp16"),     # second query tile holds one row
    (1, 255, 2, 1, 128, "bf16"),
    (1, 256, 4, 2, 64, "bf16"),     # exactly one CTA block
    (2, 257, 2, 2, 128, "fp16"),    # next block holds one row
    (1, 300, 6, 2, 128, "bf16"),
    (1, 385, 3, 3, 64, "fp16"),
    (1, 640, 8, 1, 128, "bf16"),    # GQA 8:1, several key tiles
]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("B,N,Hq,Hkv,d,dt", SMALL)
def test_small_full(B, N, Hq, Hkv, d, dt, mode):
    q, k, v = draw(B, N, Hq, Hkv, d, dt, seed=N * 7 + Hq)
    base = 1e4 if d == 64 else 5e5
    o_ref, l_ref = oracle.rope_causal(q, k, v, base)
    out, lse = run_gpu(q, k, v, base, mode)
    assert_close(out.double().numpy(), lse.double().numpy(), o_ref, l_ref, dt, f"{mode} {B}x{N}x{Hq}/{Hkv}x{d} {dt}")


# d = 128 with query-head groups of 4, 8, 12 and 16 (the Llama-3-8B layout and its neighbours):
# head-pair units of the fused kernel, ragged lengths around 64 and 128 rows, one to several units
# per CTA.
GROUPED = [
    # B, N, Hq, Hkv, dtype
    (1, 1, 4, 1, "bf16"),
    (1, 63, 4, 1, "fp16"),
    (1, 64, 4, 1, "bf16"),
    (1, 65, 4, 1, "bf16"),
    (2, 129, 8, 2, "fp16"),
    (1, 191, 4, 1, "bf16"),
    (3, 257, 4, 1, "bf16"),
    (1, 384, 8, 1, "fp16"),
    (1, 1000, 16, 1, "bf16"),
    (2, 700, 12, 3, "bf16"),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,dt", GROUPED)
def test_grouped_heads_full(B, N, Hq, Hkv, dt):
    q, k, v = draw(B, N, Hq, Hkv, 128, dt, seed=N * 5 + Hq)
    o_ref, l_ref = oracle.rope_causal(q, k, v, 5e5)
    out, lse = run_gpu(q, k, v, 5e5, "fused")
    assert_close(out.double().numpy(), lse.double().numpy(), o_ref, l_ref, dt, f"grouped {B}x{N}x{Hq}/{Hkv} {dt}")


def test_tiny_workload_both_modes():
    w = inputs.TINY
    q, k, v = inputs.make_inputs(w)
    o_ref, l_ref = oracle.rope_causal(q, k, v, w.rope_base)
    for mode in MODES:
        out, lse = run_gpu(q, k, v, w.rope_base, mode)
        assert_close(out.double().numpy(), lse.double().numpy(), o_ref, l_ref, w.dtype, f"tiny {mode}")


def test_row_zero_is_v0():
    # Causal row 0 sees only key 0, so o_0 = v_0 (to the rounding of the output).
    q, k, v = draw(1, 512, 4, 2, 128, "bf16", seed=11)
    for mode in MODES:
        out, _ = run_gpu(q, k, v, 1e4, mode)
        torch.testing.assert_close(out[:, 0], v[:, 0].repeat_interleave(2, dim=1), rtol=0, atol=0)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("H", [2, 4])
def test_rescale_path_one_hot(mode, H):
    # Energy only in the slowest pair (k = 63 with k + 64 = 127; theta = 1e4^(-126/128) ~ 1.2e-4),
    # q_i = (a, 0), k_j = (j/8, 0): the score a (j/8) cos((i-j) theta) / sqrt(d) rises with j by
    # more than 22 per key, so the softmax of row i is one-hot on j = i and the running max jumps
    # by thousands (log2 units) at every key tile.  Each jump rescales O by 2^-huge = 0, so o_i = v_i
    # up to (a) the rounding of the max itself (p_ii = 2^r, |r| < 1e-3: one fp16 ulp) and (b) fp16
    # rounding of the rotated keys (j/8)(cos, sin)(j theta), which can shrink a neighbour's score gap
    # to ~11 and leak e^-11 ~ 2e-5 of its value (|v| < 5): atol 1e-4.  A missing or wrong rescale
    # would leave earlier tiles' values in O, errors of order one.
    B, N, d = 1, 640, 128  # H query heads on one KV head
    q = torch.zeros((B, N, H, d), dtype=torch.float16)
    k = torch.zeros((B, N, 1, d), dtype=torch.float16)
    q[..., 63] = 2048.0
    k[..., 0, 63] = torch.arange(N, dtype=torch.float32).div(8).to(torch.float16)
    v = torch.randn((B, N, 1, d), generator=torch.Generator().manual_seed(9)).to(torch.float16)
    out, _ = run_gpu(q, k, v, 1e4, mode)
    torch.testing.assert_close(out.float(), v.expand(B, N, H, d).float(), rtol=1e-3, atol=1e-4)
    o_ref, _ = oracle.rope_causal(q, k, v, 1e4, rows=[0, 1, 127, 128, 300, 639])
    assert np.abs(out[:, [0, 1, 127, 128, 300, 639]].double().numpy() - o_ref).max() <= TOL["fp16"]["max_abs"]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("Hq", [4, 8])
def test_running_max_jumps(mode, dt, Hq):
    # q_63 = 8 and k_63 = c_t on key tile t, in the pair with the slowest frequency (theta ~ 2.6e-6
    # at base 5e5, so cos((i-j) theta) ~ 1): every score of key tile t is shifted by about
    # 8 c_t / sqrt(128) nats, which is 1.02 c_t in log2 units, on top of the N(0,1) scores.  With
    # c = 0, 12, 30, 15, 36 a row's running max grows by ~12 at key tile 1 (kept: P reaches 2^12),
    # by ~18 at tile 2 (the tile is redone with its own max) and by ~6 at tile 4.  Every element is
    # compared with the oracle.
    B, N, Hkv, d = 1, 640, 2, 128  # Hq = 4 or 8: groups of two or four
    q, k, v = draw(B, N, Hq, Hkv, d, dt, seed=21)
    c = torch.tensor([0.0, 12.0, 30.0, 15.0, 36.0]).repeat_interleave(128)[:N]
    q[..., 63] = 8.0
    k[..., 63] = c.view(1, N, 1).to(k.dtype)
    o_ref, l_ref = oracle.rope_causal(q, k, v, 5e5)
    out, lse = run_gpu(q, k, v, 5e5, mode)
    assert_close(out.double().numpy(), lse.double().numpy(), o_ref, l_ref, dt, f"max jumps {mode} {dt}")


@pytest.mark.parametrize("shape", [(1, 2048, 4, 2, 64, "bf16"), (1, 300, 4, 4, 64, "fp16"),
                                   (1, 2048, 2, 2, 64, "fp16"), (1, 4096, 2, 2, 64, "bf16")])
def test_auto_mode_runs_the_selected_mode(shape):
    # mode "auto" resolves on the host to one of fused, pre-rotate and split (attnfuse_select_mode:
    # here split for GQA, then fused, pre-rotate and split for MHA as N grows) and then runs exactly
    # that path: bitwise the same result, and within the oracle tolerance.
    B, N, Hq, Hkv, d, dt = shape
    q, k, v = draw(B, N, Hq, Hkv, d, dt, seed=31)
    sel = binding.select_mode(B, Hq, Hkv, N, d, q.dtype)
    oa, la = run_gpu(q, k, v, 1e4, "auto")
    os_, ls = run_gpu(q, k, v, 1e4, sel)
    assert torch.equal(oa, os_) and torch.equal(la, ls)
    o_ref, l_ref = oracle.rope_causal(q, k, v, 1e4)
    assert_close(oa.double().numpy(), la.double().numpy(), o_ref, l_ref, dt, f"auto ({sel}) {shape}")


@pytest.mark.parametrize("shape", [(1, 300, 4, 2, 128, "bf16"), (2, 257, 2, 2, 64, "fp16"), (1, 4096, 32, 8, 128, "bf16")])
def test_none_mode_is_the_prerotate_paths_attention(shape):
    # mode "none" runs the pre-rotate path's attention kernel on q and k as given; fed the RoPE
    # pass's output it reproduces the pre-rotate mode bit for bit (same kernels, same operands).
    B, N, Hq, Hkv, d, dt = shape
    q, k, v = (t.cuda() for t in draw(B, N, Hq, Hkv, d, dt, seed=41))
    qr, kr = binding.rope_apply(q, 5e5), binding.rope_apply(k, 5e5)
    on, ln = binding.rope_causal_fwd(qr, kr, v, 5e5, mode="none")
    op, lp = binding.rope_causal_fwd(q, k, v, 5e5, mode="prerotate")
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert torch.equal(on, op) and torch.equal(ln, lp)


def test_lse_optional():
    q, k, v = draw(1, 200, 2, 1, 64, "bf16", seed=3)
    out_a, _ = binding.rope_causal_fwd(q.cuda(), k.cuda(), v.cuda(), 1e4, want_lse=False)
    out_b, _ = binding.rope_causal_fwd(q.cuda(), k.cuda(), v.cuda(), 1e4)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)


def test_explicit_workspace_and_stream():
    q, k, v = (t.cuda() for t in draw(2, 300, 4, 2, 128, "fp16", seed=5))
    need = binding.workspace_bytes(2, 4, 2, 300, 128, "prerotate", torch.float16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out_ws, lse_ws = binding.rope_causal_fwd(q, k, v, 5e5, mode="prerotate", workspace=ws, stream=s)
    s.synchronize()
    out, lse = binding.rope_causal_fwd(q, k, v, 5e5, mode="prerotate")
    torch.cuda.synchronize()
    assert torch.equal(out, out_ws) and torch.equal(lse, lse_ws)


# ---------------------------------------------------------------------------------------------
# Full-size workloads, sampled rows


def _sampled(w, mode, n_random=96):
    q, k, v = inputs.make_inputs(w)
    rows = sample_rows(w.N, n_random, seed=w.seed)
    o_ref, l_ref = oracle.rope_causal(q, k, v, w.rope_base, rows=rows)
    out, lse = run_gpu(q, k, v, w.rope_base, mode)
    return assert_close(out[:, rows].double().numpy(), lse[:, :, rows].double().numpy(), o_ref, l_ref, w.dtype,
                        f"{w.name} {mode}")


@pytest.mark.parametrize("mode", MODES)
def test_mha_workload_full(mode):
    w = inputs.MHA
    q, k, v = inputs.make_inputs(w)
    o_ref, l_ref = oracle.rope_causal(q, k, v, w.rope_base)
    out, lse = run_gpu(q, k, v, w.rope_base, mode)
    assert_close(out.double().numpy(), lse.double().numpy(), o_ref, l_ref, w.dtype, f"mha {mode}")


@pytest.fixture(scope="module")
def llama_ref():
    # The oracle over every row of the Llama-3-8B workload (a few seconds on the host cores),
    # computed once for the three modes.
    w = inputs.LLAMA
    q, k, v = inputs.make_inputs(w)
    o_ref, l_ref = oracle.rope_causal(q, k, v, w.rope_base)
    return q, k, v, o_ref, l_ref


@pytest.mark.parametrize("mode", MODES)
def test_llama_workload_full(mode, llama_ref):
    # Every element of the benchmark's default workload, in the launch configuration it times.
    w = inputs.LLAMA
    q, k, v, o_ref, l_ref = llama_ref
    out, lse = run_gpu(q, k, v, w.rope_base, mode)
    assert_close(out.double().numpy(), lse.double().numpy(), o_ref, l_ref, w.dtype, f"llama {mode}")


@pytest.mark.parametrize("mode", MODES)
def test_long_context_sampled(mode):
    _sampled(inputs.LONG, mode, n_random=32)


@pytest.mark.parametrize("w", inputs.sweep_workloads(), ids=lambda w: w.name)
def test_sweep_points_sampled(w):
    for mode in MODES:
        _sampled(w, mode, n_random=16)


# ---------------------------------------------------------------------------------------------
# Fused and pre-rotate modes agree


@pytest.mark.parametrize("w", [inputs.TINY, inputs.MHA, inputs.LLAMA], ids=lambda w: w.name)
def test_modes_agree(w):
    # Both modes rotate Q with identical arithmetic; K differs only in how cos/sin are produced
    # (exact per element vs. angle addition along the key tile), a relative difference below 3e-5,
    # so rotated keys differ by at most one rounding of the dtype on a few elements.  The outputs
    # then agree to well under the oracle tolerance: a quarter of it is required here.
    # The split mode rotates K exactly (the pass) and Q along the tile (on chip): the same bound holds.
    q, k, v = (t.cuda() for t in inputs.make_inputs(w))
    op, lp = binding.rope_causal_fwd(q, k, v, w.rope_base, mode="prerotate")
    t = TOL[w.dtype]
    for m in ("fused", "split"):
        of, lf = binding.rope_causal_fwd(q, k, v, w.rope_base, mode=m)
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        e = errors(of.double().cpu().numpy(), lf.double().cpu().numpy(), op.double().cpu().numpy(),
                   lp.double().cpu().numpy())
        assert e["max_abs"] <= t["max_abs"] / 4 and e["rel_l2"] <= t["rel_l2"] / 4, (m, e)
        assert e["lse_row"] <= t["lse_row"] / 4, (m, e)
