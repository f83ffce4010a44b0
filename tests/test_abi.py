"""CPU-side checks of the C ABI: the library builds and loads without a GPU, exports every function
include/attnfuse.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from attention_rope_causal_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attnfuse.h")

FAKE = 0x10000  # a 16-byte-aligned non-null address; never dereferenced by argument checks


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attnfuse_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("attnfuse_rope_causal_fwd", "attnfuse_rope_apply", "attnfuse_workspace_bytes",
              "attnfuse_status_string", "attnfuse_last_error", "attnfuse_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(binding._SIGNATURES)


def test_status_strings(lib):
    for code in range(6):
        assert lib.attnfuse_status_string(code)
    assert lib.attnfuse_version().startswith(b"libattnfuse")


def fwd(lib, q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=None, B=1, Hq=4, Hkv=2, N=128, d=64, base=1e4, mode=0, dtype=0,
        ws=None, ws_bytes=0):
    return lib.attnfuse_rope_causal_fwd(q, k, v, out, lse, B, Hq, Hkv, N, d, base, mode, dtype, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(out=None), 1), (dict(B=0), 1), (dict(N=0), 1), (dict(Hq=3, Hkv=2), 1),
    (dict(d=96), 2), (dict(d=256), 2), (dict(dtype=7), 1), (dict(mode=5), 1), (dict(mode=-1), 1),
    (dict(base=0.5), 1), (dict(mode=2, B=0), 1),
    (dict(base=float("nan")), 1), (dict(q=FAKE + 8), 1), (dict(lse=FAKE + 2), 1), (dict(N=1 << 24), 1),
    (dict(mode=1, ws=FAKE, ws_bytes=16), 1), (dict(mode=1, ws=FAKE + 16, ws_bytes=1 << 40), 1),
])
def test_forward_rejects_bad_arguments(lib, kw, status):
    assert fwd(lib, **kw) == status
    assert lib.attnfuse_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), 1), (dict(d=80), 2), (dict(H=0), 1), (dict(x=FAKE, y=FAKE + 64), 1), (dict(y=FAKE + 4), 1),
])
def test_rope_apply_rejects_bad_arguments(lib, kw, status):
    a = dict(x=FAKE, y=FAKE, B=1, N=16, H=2, d=64, base=1e4, dtype=0)
    a.update(kw)
    assert lib.attnfuse_rope_apply(a["x"], a["y"], a["B"], a["N"], a["H"], a["d"], a["base"], a["dtype"], None) == status


def test_none_mode_needs_no_workspace_and_takes_no_rotation_option(lib):
    assert lib.attnfuse_workspace_bytes(1, 32, 8, 4096, 128, 4, 0) == 0
    opts = binding.RopeOpts(64, 0, 0, None, None)  # rotary_dim: meaningless without a rotation
    st = lib.attnfuse_rope_causal_fwd_ex(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 128, 128, 1e4, 4, 0, None, 0,
                                         ctypes.byref(opts), None)
    assert st == 1 and b"none" in lib.attnfuse_last_error()


def test_workspace_bytes(lib):
    assert lib.attnfuse_workspace_bytes(1, 32, 8, 4096, 128, 0, 0) == 0
    q = 1 * 4096 * 32 * 128 * 2
    k = 1 * 4096 * 8 * 128 * 2
    assert lib.attnfuse_workspace_bytes(1, 32, 8, 4096, 128, 1, 0) == q + k
    assert lib.attnfuse_workspace_bytes(1, 1, 1, 1, 64, 1, 1) == 256 + 256
    assert lib.attnfuse_workspace_bytes(1, 1, 1, 1, 96, 1, 1) == 0


@pytest.mark.parametrize("B,Hq,Hkv,N,mode", [
    (1, 32, 8, 4096, 3), (4, 32, 8, 2048, 3), (1, 32, 8, 16384, 3), (16, 32, 8, 1024, 3),  # GQA 4:1
    (8, 32, 8, 1023, 0), (1, 8, 4, 3000, 3), (1, 64, 8, 1023, 0),                          # other groups
    (2, 16, 16, 1536, 0), (1, 16, 16, 1891, 0), (1, 16, 16, 1892, 1), (1, 16, 16, 4095, 1),  # MHA
    (1, 16, 16, 4096, 3), (1, 16, 16, 32768, 3),
    (0, 16, 16, 4096, 0), (1, 6, 4, 4096, 0),                                          # not classified
])
def test_select_mode_follows_the_measured_crossover(lib, B, Hq, Hkv, N, mode):
    for d in (64, 128):
        for dtype in (0, 1):
            assert lib.attnfuse_select_mode(B, Hq, Hkv, N, d, dtype) == mode


def test_split_mode_workspace_is_the_rotated_keys(lib):
    assert lib.attnfuse_workspace_bytes(1, 32, 8, 4096, 128, 3, 0) == 1 * 4096 * 8 * 128 * 2
    assert lib.attnfuse_workspace_bytes(1, 1, 1, 1, 64, 3, 1) == 256
    assert fwd(lib, mode=3, ws=FAKE, ws_bytes=16) == 1       # workspace too small for K'
    assert fwd(lib, mode=5) == 1                              # no mode 5


def test_auto_mode_workspace_is_that_of_the_selected_mode(lib):
    for shape in ((1, 32, 8, 4096, 128), (2, 16, 16, 1536, 64), (1, 16, 16, 8192, 64)):
        sel = lib.attnfuse_select_mode(*shape, 0)
        assert lib.attnfuse_workspace_bytes(*shape, 2, 0) == lib.attnfuse_workspace_bytes(*shape, sel, 0)
    assert binding.select_mode(1, 32, 8, 4096, 128) == "split"
    assert binding.select_mode(2, 16, 16, 1536, 64) == "fused"
    assert binding.select_mode(1, 16, 16, 2048, 64) == "prerotate"
    assert binding.select_mode(1, 16, 16, 8192, 64) == "split"


@pytest.mark.parametrize("r,il,status", [(8, 0, 1), (24, 0, 1), (80, 1, 1), (-16, 0, 1), (64, 2, 1), (64, -1, 1)])
def test_variant_options_are_checked_before_the_device(lib, r, il, status):
    opts = binding.RopeOpts(r, il)
    assert lib.attnfuse_rope_causal_fwd_ex(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 128, 64, 1e4, 0, 0, None, 0,
                                           ctypes.byref(opts), None) == status
    assert lib.attnfuse_rope_apply_ex(FAKE, FAKE, 1, 16, 2, 64, 1e4, 0, ctypes.byref(opts), None) == status
    assert b"rotary_dim" in lib.attnfuse_last_error() or b"interleaved" in lib.attnfuse_last_error()


@pytest.mark.parametrize("kv_len,qpos,kpos,what", [(100, None, None, b"kv_len"), (1 << 24, None, None, b"kv_len"),
                                                  (-5, None, None, b"kv_len"), (0, FAKE + 2, None, b"positions"),
                                                  (200, None, FAKE + 1, b"positions")])
def test_key_length_and_position_options_are_checked_before_the_device(lib, kv_len, qpos, kpos, what):
    opts = binding.RopeOpts(0, 0, kv_len, qpos, kpos)
    assert lib.attnfuse_rope_causal_fwd_ex(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 128, 64, 1e4, 0, 0, None, 0,
                                           ctypes.byref(opts), None) == 1
    assert what in lib.attnfuse_last_error()


def test_rope_apply_takes_query_positions_only(lib):
    for opts in (binding.RopeOpts(0, 0, 32, None, None), binding.RopeOpts(0, 0, 0, None, FAKE)):
        assert lib.attnfuse_rope_apply_ex(FAKE, FAKE, 1, 16, 2, 64, 1e4, 0, ctypes.byref(opts), None) == 1
        assert b"q_positions only" in lib.attnfuse_last_error()


def test_workspace_bytes_with_more_keys(lib):
    opts = binding.RopeOpts(0, 0, 1000, None, None)
    q = 1 * 300 * 4 * 128 * 2
    k = 1 * 1000 * 2 * 128 * 2
    assert lib.attnfuse_workspace_bytes_ex(1, 4, 2, 300, 128, 1, 0, ctypes.byref(opts)) == q + k
    assert lib.attnfuse_workspace_bytes_ex(1, 4, 2, 300, 128, 0, 0, ctypes.byref(opts)) == 0
    assert lib.attnfuse_workspace_bytes_ex(1, 4, 2, 300, 128, 1, 0, None) == lib.attnfuse_workspace_bytes(
        1, 4, 2, 300, 128, 1, 0)
    short = binding.RopeOpts(0, 0, 100, None, None)
    assert lib.attnfuse_workspace_bytes_ex(1, 4, 2, 300, 128, 1, 0, ctypes.byref(short)) == 0
    # AUTO judges the shape by the key length
    long_kv = binding.RopeOpts(0, 0, 8192, None, None)
    assert lib.attnfuse_workspace_bytes_ex(1, 32, 8, 16, 128, 2, 0, ctypes.byref(long_kv)) > 0
    assert binding.workspace_bytes(1, 4, 2, 300, 128, "prerotate", kv_len=1000) == q + k


@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 32, 8, 1), (64, 32, 8, 1), (1, 32, 8, 4), (1, 32, 8, 5), (1, 16, 4, 16),
                                       (1, 8, 8, 8), (8, 8, 8, 16), (2, 8, 8, 17), (65535, 1, 1, 1), (65536, 1, 1, 1)])
def test_decode_routing_shows_in_the_fused_workspace(lib, B, Hq, Hkv, N):
    # The fused tile kernel needs no workspace, the decode kernels need room for their partials, so
    # the size a fused call asks for shows which path it takes.
    from parity import decode_path
    opts = binding.RopeOpts(0, 0, 4096, None, None)
    need = lib.attnfuse_workspace_bytes_ex(B, Hq, Hkv, N, 128, 0, 0, ctypes.byref(opts))
    # (past 65535 batch entries the grid cannot hold the decode kernels: the tile kernels run)
    assert (need > 0) == (decode_path(B, Hq, Hkv, N) and B <= 65535)


def bwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1, Hq=4, Hkv=2, N=128,
             d=64, base=1e4, dtype=0, ws=None, wsb=0)
    a.update(kw)
    return lib.attnfuse_rope_causal_bwd(a["q"], a["k"], a["v"], a["out"], a["lse"], a["dout"], a["dq"], a["dk"],
                                        a["dv"], a["B"], a["Hq"], a["Hkv"], a["N"], a["d"], a["base"], a["dtype"],
                                        a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,status", [({"lse": None}, 1), ({"dout": None}, 1), ({"dq": None}, 1), ({"dv": FAKE + 8}, 1),
                                        ({"d": 96}, 2), ({"Hq": 3}, 1), ({"N": 0}, 1), ({"dtype": 7}, 1),
                                        ({"ws": FAKE, "wsb": 64}, 1), ({"base": 0.5}, 1)])
def test_backward_arguments_are_checked_before_the_device(lib, kw, status):
    assert bwd(lib, **kw) == status


def test_backward_workspace_bytes(lib):
    q = 1 * 4096 * 32 * 128 * 2
    k = 1 * 4096 * 8 * 128 * 2
    dvec = 32 * 4096 * 4
    counter = 256  # the dQ kernel's work counter
    assert lib.attnfuse_bwd_workspace_bytes(1, 32, 8, 4096, 128, 0) == q + k + dvec + counter
    assert lib.attnfuse_bwd_workspace_bytes(1, 32, 8, 4096, 96, 0) == 0
    assert lib.attnfuse_bwd_workspace_bytes(0, 32, 8, 4096, 128, 0) == 0


def test_valid_call_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd(lib) == 3  # ERR_CUDA: no device; nothing was launched
    assert lib.attnfuse_device_status(None) == 3


def test_diag_rejects_bad_timeout(lib):
    assert lib.attnfuse_diag_wait_timeout(0, None) == 1
    assert lib.attnfuse_diag_wait_timeout(2_000_000_000, None) == 1


def test_binding_rejects_host_tensors_before_the_library():
    # The binding marshals device pointers only: host tensors are refused with ValueError (no CPU
    # path exists to fall back on).
    import torch
    q = torch.zeros((1, 8, 2, 64), dtype=torch.bfloat16)
    kv = torch.zeros((1, 8, 1, 64), dtype=torch.bfloat16)
    lse = torch.zeros((1, 2, 8), dtype=torch.float32)
    with pytest.raises(ValueError):
        binding.rope_causal_fwd(q, kv, kv, 1e4)
    with pytest.raises(ValueError):
        binding.rope_apply(q, 1e4)
    with pytest.raises(ValueError):
        binding.rope_causal_bwd(q, kv, kv, q, lse, q, 1e4)


def test_backward_workspace_with_more_keys_than_queries():
    # q' over N tokens, k' over Nk = kv_len, D over N (float), each rounded up to 256 bytes, and 256
    # bytes for the dQ kernel's work counter.
    import torch
    B, N, Nk, Hq, Hkv, d = 2, 130, 517, 8, 2, 128
    up = lambda x: (x + 255) // 256 * 256
    want = up(B * N * Hq * d * 2) + up(B * Nk * Hkv * d * 2) + up(B * Hq * N * 4) + 256
    assert binding.bwd_workspace_bytes(B, Hq, Hkv, N, d, torch.bfloat16, kv_len=Nk) == want
    assert binding.bwd_workspace_bytes(B, Hq, Hkv, N, d, torch.bfloat16, kv_len=N) == \
        binding.bwd_workspace_bytes(B, Hq, Hkv, N, d, torch.bfloat16)
    assert binding.bwd_workspace_bytes(B, Hq, Hkv, N, d, torch.bfloat16, kv_len=N - 1) == 0
