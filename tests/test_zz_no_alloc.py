"""pkv_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory (a plugin inside a runtime that owns the memory budget,
a loop that must never call cudaMalloc).  Its scratch is a device array built
into the library instead of a caller workspace.

Called through the C ABI (ctypes) and checked against pkv_decode_attention,
which gets a workspace of its own, on two calls in a row, within the decode
tolerance used everywhere else (|a - b| <= 2e-3 + 1e-2 |b|).  This file is
collected last so that a failure here comes after every other test has run.
"""

import ctypes

import numpy as np
import pytest

from paged_kv_cache_131_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_131_gb300 import _build
    _build.build()
    import paged_kv_cache_131_gb300 as pkv
    assert torch.cuda.is_available()
    pkv.pkv_get_device_error()
    return pkv


def _noalloc(pkv, dev, out):
    """One call of the allocation-free entry point, straight through ctypes."""
    wl = dev.wl
    stream = torch.cuda.current_stream().cuda_stream
    return pkv.load().pkv_decode_attention_noalloc(
        out.data_ptr(), dev.q.data_ptr(), dev.k_cache.data_ptr(), dev.v_cache.data_ptr(),
        dev.block_tables.data_ptr(), dev.seq_lens.data_ptr(), ctypes.c_float(wl.scale),
        wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, wl.num_seqs,
        wl.max_blocks_per_seq, wl.max_seq_len, wl.num_blocks, ctypes.c_void_p(stream))


def _close(a, b):
    a = a.cpu().numpy().astype(np.float64)
    b = b.cpu().numpy().astype(np.float64)
    assert np.isfinite(a).all()
    err = np.abs(a - b)
    assert (err <= ATOL + RTOL * np.abs(b)).all(), f"max |err| {err.max():.3e}"


@pytest.mark.parametrize("case", [
    dict(index=301, lens=[1, 17, 600, 1500, 2100, 33, 0, 900], H=32, Hk=8, D=128),
    dict(index=302, lens=[5, 700, 1300, 64], H=8, Hk=1, D=64),
])
def test_noalloc_matches_workspace_entry_point_twice(lib, case):
    from paged_kv_cache_131_gb300.harness import DeviceDecode
    wl = W.small_decode(case["index"], case["lens"], H=case["H"], Hk=case["Hk"], D=case["D"])
    dev = DeviceDecode(wl)  # owns the workspace the regular entry point uses
    dev.write()
    ref = dev.decode().clone()
    for _ in range(2):  # two calls in a row share the built-in scratch
        out = torch.full_like(dev.q, float("nan"))
        assert _noalloc(lib, dev, out) == 0
        torch.cuda.synchronize()
        _close(out, ref)
    assert lib.pkv_get_device_error() == (0, -1)


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    # 64 sequences of up to 32768 tokens with 16 KV heads: too many KV heads for
    # the balanced schedule and 64 partitions x 64 heads x 128 dims of fp32
    # partials for the grid schedule -- far beyond the built-in scratch
    S, H, Hk, D, L = 64, 64, 16, 128, 32768
    q = torch.zeros(S, H, D, dtype=torch.float16, device="cuda")
    cache = torch.zeros(4, 16, Hk, D, dtype=torch.float16, device="cuda")
    bt = torch.zeros(S, L // 16, dtype=torch.int32, device="cuda")
    sl = torch.zeros(S, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    st = lib.load().pkv_decode_attention_noalloc(
        out.data_ptr(), q.data_ptr(), cache.data_ptr(), cache.data_ptr(), bt.data_ptr(),
        sl.data_ptr(), ctypes.c_float(0.125), H, Hk, D, 16, S, L // 16, L, 4, None)
    assert st == -5
    assert "scratch" in lib.pkv_last_error_string()
