"""The no-allocation pre-rotate entry point (attnfuse_rope_causal_fwd_prerotate_noalloc).

It serves callers that cannot allocate device memory (their framework's allocator owns the GPU's
memory, or they must not risk an allocation failing or stalling mid-step) and cannot lend a
workspace either: the rotated Q and K go to a fixed 64 MiB buffer inside the library.  These tests
call it through the C ABI and compare it with the regular entry point, on two calls in a row (the
buffer keeps the previous call's contents, which must not leak into the next result).  The file is
named to be collected last.
"""
import ctypes

import pytest
import torch

from attention_rope_causal_gb300 import binding, build, inputs
from parity import TOL, errors

SCRATCH = 64 << 20


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def call_noalloc(lib, q, k, v, out, lse, base):
    B, N, Hq, d = q.shape
    return lib.attnfuse_rope_causal_fwd_prerotate_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq, k.shape[2], N, d,
        float(base), binding.DTYPES[q.dtype], torch.cuda.current_stream().cuda_stream)


def test_argument_errors_come_before_any_device_work(lib):
    # Null or misaligned pointers and unsupported sizes are refused by the same checks as the regular
    # entry point, before the device is touched (so these run without a GPU).
    assert lib.attnfuse_rope_causal_fwd_prerotate_noalloc(None, 0x10000, 0x10000, 0x10000, None, 1, 2, 2, 16, 64,
                                                          1e4, 0, None) == 1
    assert lib.attnfuse_rope_causal_fwd_prerotate_noalloc(0x10008, 0x10000, 0x10000, 0x10000, None, 1, 2, 2, 16, 64,
                                                          1e4, 0, None) == 1
    assert b"aligned" in lib.attnfuse_last_error()
    assert lib.attnfuse_rope_causal_fwd_prerotate_noalloc(0x10000, 0x10000, 0x10000, 0x10000, None, 1, 2, 2, 16,
                                                          96, 1e4, 0, None) == 2  # d = 96: unsupported


@pytest.mark.gpu
def test_rejects_problems_larger_than_the_buffer(lib):
    # 32k tokens of 32 + 8 heads at d = 128 need 335 MB of rotated Q and K: refused before any launch
    # (the size check follows the device check, so it needs the GPU to be an sm_103 part).
    st = lib.attnfuse_rope_causal_fwd_prerotate_noalloc(0x10000, 0x10000, 0x10000, 0x10000, None, 1, 32, 8, 32768,
                                                        128, 5e5, 0, None)
    assert st == 1 and b"fixed" in lib.attnfuse_last_error()


@pytest.mark.gpu
def test_matches_regular_entry_point_on_two_calls_in_a_row(lib):
    cases = [inputs.LLAMA,  # 42 MB of rotated Q and K: most of the buffer
             inputs.Workload("ragged_fp16", B=2, Hq=6, Hkv=2, N=300, d=128, dtype="fp16", rope_base=5e5, sigma=1.0,
                             seed=21)]
    for w in cases:
        assert binding.workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d, "prerotate", w.torch_dtype) <= SCRATCH
        q, k, v = (t.cuda() for t in inputs.make_inputs(w))
        ref_out, ref_lse = binding.rope_causal_fwd(q, k, v, w.rope_base, mode="prerotate")
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, w.Hq, w.N), float("nan"), device="cuda")
        assert call_noalloc(lib, q, k, v, out, lse, w.rope_base) == 0, binding.last_error()
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        e = errors(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out.double().cpu().numpy(),
                   ref_lse.double().cpu().numpy())
        t = TOL[w.dtype]
        assert e["max_abs"] <= t["max_abs"] and e["rel_l2"] <= t["rel_l2"], (w.name, e)
        assert e["lse_row"] <= t["lse_row"], (w.name, e)


@pytest.mark.gpu
def test_a_call_allocates_no_device_memory(lib):
    # After a first call (which looks up the buffer and loads the kernels), further calls change
    # neither the device's free memory nor what torch's allocator holds.
    w = inputs.Workload("small", B=1, Hq=4, Hkv=2, N=512, d=128, dtype="bf16", rope_base=5e5, sigma=1.0, seed=5)
    q, k, v = (t.cuda() for t in inputs.make_inputs(w))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.N), device="cuda")
    assert call_noalloc(lib, q, k, v, out, lse, w.rope_base) == 0, binding.last_error()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    held0 = torch.cuda.memory_allocated()
    for _ in range(3):
        assert call_noalloc(lib, q, k, v, out, lse, w.rope_base) == 0, binding.last_error()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_allocated() == held0
    assert binding.device_status() == 0
