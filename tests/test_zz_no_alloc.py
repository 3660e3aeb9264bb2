"""pkv_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory (a plugin inside a runtime that owns the memory budget,
a loop that must never call cudaMalloc).  Its scratch is a device array built
into the library instead of a caller workspace.

Called through the C ABI (ctypes) and checked against pkv_decode_attention,
which gets a workspace of its own, and against the float64 oracle, on two
calls in a row, within the decode tolerance used everywhere else
(|a - b| <= 2e-3 + 1e-2 |b|).  This file is collected last so that a failure
here comes after every other test has run.
"""

import ctypes

import numpy as np
import pytest

import oracle
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


def _oracle(wl):
    """The oracle's decode after the write of the new rows."""
    k, v = wl.k_cache.copy(), wl.v_cache.copy()
    row = wl.num_kv_heads * wl.head_dim * 2
    for cache, new in ((k, wl.k_new), (v, wl.v_new)):
        oracle.cache_write(cache.view(np.uint8).reshape(-1), new.view(np.uint8), wl.slot_mapping,
                           offset=0, layer=0, layer_stride=0, block_stride=wl.block_size * row,
                           row_width=row, block_size=wl.block_size, num_blocks=wl.num_blocks)
    return oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale)


def _check_twice(lib, wl):
    from paged_kv_cache_131_gb300.harness import DeviceDecode
    dev = DeviceDecode(wl)  # owns the workspace the regular entry point uses
    dev.write()
    ref = dev.decode().clone()
    exact = _oracle(wl)
    for _ in range(2):  # two calls in a row share the built-in scratch
        out = torch.full_like(dev.q, float("nan"))
        assert _noalloc(lib, dev, out) == 0
        torch.cuda.synchronize()
        _close(out, ref)
        _close(out, torch.from_numpy(exact))
    assert lib.pkv_get_device_error() == (0, -1)


@pytest.mark.parametrize("case", [
    dict(index=301, lens=[1, 17, 600, 1500, 2100, 33, 0, 900], H=32, Hk=8, D=128),
    dict(index=302, lens=[5, 700, 1300, 64], H=8, Hk=1, D=64),
    dict(index=303, lens=[600, 1000, 70, 1500], H=128, Hk=16, D=128),  # 2 head groups
    # many blocks per CTA range, every sequence cut several times
    dict(index=307, lens=[3000 + 37 * i for i in range(16)], H=8, Hk=8, D=128),
])
def test_noalloc_matches_workspace_entry_point_twice(lib, case):
    wl = W.small_decode(case["index"], case["lens"], H=case["H"], Hk=case["Hk"], D=case["D"])
    _check_twice(lib, wl)


def test_noalloc_grid_schedule_twice(lib):
    # 28000 short sequences: the balanced schedule's per-sequence tables do
    # not fit its shared memory, so the grid schedule runs (one partition per
    # sequence; its own counter layout, per query head)
    lens = [1 + (7 * i) % 40 for i in range(28000)]
    wl = W.small_decode(306, lens, H=8, Hk=2, D=64)
    _check_twice(lib, wl)


def test_noalloc_clears_what_an_earlier_shape_left(lib):
    # A first call with one KV head and two long sequences cut into many
    # pieces writes partial states right behind its small counter region; a
    # second call with 64 sequences x 8 KV heads puts its counters on those
    # bytes.  The second call starts from cleared counters all the same.
    first = W.small_decode(304, [3000, 2800], H=8, Hk=1, D=64)
    _check_twice(lib, first)
    second = W.small_decode(305, [200 + 37 * i for i in range(64)], H=32, Hk=8, D=128)
    _check_twice(lib, second)


def test_noalloc_refused_calls_return_before_any_work(lib):
    # argument errors are reported as by pkv_decode_attention, before the
    # scratch is touched or anything is enqueued
    S, H, Hk, D = 2, 8, 2, 64
    q = torch.zeros(S, H, D, dtype=torch.float16, device="cuda")
    cache = torch.zeros(4, 16, Hk, D, dtype=torch.float16, device="cuda")
    bt = torch.zeros(S, 4, dtype=torch.int32, device="cuda")
    sl = torch.ones(S, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    f = lib.load().pkv_decode_attention_noalloc

    def call(out_ptr=out.data_ptr(), q_ptr=q.data_ptr(), H=H, D=D, bs=16):
        return f(out_ptr, q_ptr, cache.data_ptr(), cache.data_ptr(), bt.data_ptr(),
                 sl.data_ptr(), ctypes.c_float(0.125), H, Hk, D, bs, S, 4, 64, 4, None)

    assert call(out_ptr=None) == -1           # PKV_ERR_NULL
    assert call(bs=32) == -3                  # PKV_ERR_UNSUPPORTED: block size
    assert call(D=96) == -3                   # head_dim
    assert call(H=2 * 16) == -3               # group of 16 query heads
    assert call(q_ptr=q.data_ptr() + 2) == -4  # PKV_ERR_ALIGNMENT
    assert call() == 0
    torch.cuda.synchronize()
    assert lib.pkv_get_device_error() == (0, -1)


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    # 28000 sequences of up to 8192 tokens: too many sequences for the
    # balanced schedule's shared memory, and 16 partitions x 8 heads x 64 dims
    # of fp32 partials per sequence for the grid schedule -- far beyond the
    # built-in scratch
    S, H, Hk, D, L = 28000, 8, 2, 64, 8192
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
