"""Writes stay inside their buffers: the attention outputs, the caller's
workspace and a cache being written are placed inside larger device buffers
filled with a sentinel, and afterwards every sentinel byte before and after
them is unchanged (fp16 decode on both schedules, FP8 decode, the
multi-token call, the cache write at every vector width).  The attention
cases split sequences across CTAs, so partial states, tickets and merges all
run; every result is also checked against the oracle."""

import numpy as np
import pytest

import oracle
from paged_kv_cache_131_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2
PAD = 4096            # fp16 elements of sentinel on each side of an output
WS_PAD = 1 << 16      # sentinel bytes after the workspace
OUT_SENTINEL = 0x7BAD  # an fp16 bit pattern no attention output here has
WS_SENTINEL = 0xA5


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_131_gb300 import _build
    _build.build()
    import paged_kv_cache_131_gb300 as m
    assert torch.cuda.is_available()
    m.pkv_get_device_error()
    return m


def _guard_out(like):
    n = like.numel()
    buf = torch.full((PAD + n + PAD,), OUT_SENTINEL, dtype=torch.int16, device=like.device)
    return buf, buf[PAD:PAD + n].view(torch.float16).view(like.shape)


def _guard_ws(ws):
    nbytes = ws.numel()
    buf = torch.full((nbytes + WS_PAD,), WS_SENTINEL, dtype=torch.uint8, device=ws.device)
    buf[:nbytes].zero_()
    return buf, buf[:nbytes]


def _check_guards(obuf, n, wbuf, nbytes):
    o = obuf.cpu().numpy()
    assert (o[:PAD] == OUT_SENTINEL).all() and (o[PAD + n:] == OUT_SENTINEL).all()
    w = wbuf.cpu().numpy()
    assert (w[nbytes:] == WS_SENTINEL).all()


def _close(got, ref):
    got = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert (err <= ATOL + RTOL * np.abs(ref)).all(), f"max |err| {err.max():.3e}"


def _oracle_decode(wl):
    k, v = wl.k_cache.copy(), wl.v_cache.copy()
    row = wl.num_kv_heads * wl.head_dim * 2
    for cache, new in ((k, wl.k_new), (v, wl.v_new)):
        oracle.cache_write(cache.view(np.uint8).reshape(-1), new.view(np.uint8), wl.slot_mapping,
                           offset=0, layer=0, layer_stride=0, block_stride=wl.block_size * row,
                           row_width=row, block_size=wl.block_size, num_blocks=wl.num_blocks)
    return oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale,
                                   workers=oracle.default_workers())


@pytest.mark.parametrize("schedule", [1, 2], ids=["grid", "balanced"])
def test_decode_writes_stay_in_bounds(pkv, schedule):
    from paged_kv_cache_131_gb300.harness import DeviceDecode
    wl = W.small_decode(701, [3000 + 97 * i for i in range(12)], H=32, Hk=8, D=128)
    dev = DeviceDecode(wl, schedule=schedule)
    obuf, out = _guard_out(dev.out)
    wbuf, dev.workspace = _guard_ws(dev.workspace)
    dev.write()
    for _ in range(2):
        dev.decode(out=out)
    torch.cuda.synchronize()
    _check_guards(obuf, out.numel(), wbuf, dev.workspace.numel())
    _close(out, _oracle_decode(wl))
    assert pkv.pkv_get_device_error() == (0, -1)


def test_fp8_decode_writes_stay_in_bounds(pkv):
    from paged_kv_cache_131_gb300.harness import DeviceDecodeFp8
    wl = W.small_decode(702, [2500 + 131 * i for i in range(10)], H=32, Hk=8, D=128)
    dev = DeviceDecodeFp8(wl)
    obuf, dev.out = _guard_out(dev.out)
    wbuf, dev.workspace = _guard_ws(dev.workspace)
    dev.write()
    for _ in range(2):
        dev.decode()
    torch.cuda.synchronize()
    _check_guards(obuf, dev.out.numel(), wbuf, dev.workspace.numel())
    assert np.isfinite(dev.out.float().cpu().numpy()).all()
    assert pkv.pkv_get_device_error() == (0, -1)


def test_chunk_writes_stay_in_bounds(pkv):
    # a long chunk on the tile kernel over three KV partitions (partial
    # states and their merge) beside short ones on the balanced schedule
    from paged_kv_cache_131_gb300.harness import DeviceChunk
    wl = W.chunk_workload(703, [9000, 300, 4500, 700], [150, 3, 64, 1], H=32, Hk=8, D=128)
    dev = DeviceChunk(wl)
    obuf, dev.out = _guard_out(dev.out)
    wbuf, dev.workspace = _guard_ws(dev.workspace)
    for _ in range(2):
        dev.step()
    torch.cuda.synchronize()
    _check_guards(obuf, dev.out.numel(), wbuf, dev.workspace.numel())
    from test_oracle_chunk import written_caches
    k, v = written_caches(wl)
    ref = oracle.chunk_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.query_start,
                                 wl.scale, workers=oracle.default_workers())
    _close(dev.out, ref)
    assert pkv.pkv_get_device_error() == (0, -1)


@pytest.mark.parametrize("row_width,vec_align", [(2048, 16), (656, 16), (132, 4), (37, 1)])
def test_cache_write_stays_in_the_cache(pkv, row_width, vec_align):
    """The cache sits inside a sentinel-filled buffer; slots include the
    cache's first and last, plus a padding slot and one out of range (both
    skipped).  Every byte outside the cache keeps its sentinel, and the cache
    equals the oracle's write."""
    nb, bs = 8, 16
    rng = np.random.default_rng(row_width)
    cache_bytes = nb * bs * row_width
    buf = torch.full((WS_PAD + cache_bytes + WS_PAD,), WS_SENTINEL, dtype=torch.uint8,
                     device="cuda")
    init = rng.integers(0, 256, size=cache_bytes, dtype=np.uint8)
    cache = buf[WS_PAD:WS_PAD + cache_bytes]
    cache.copy_(torch.from_numpy(init))
    slots = np.array([0, nb * bs - 1, -1, 5, nb * bs, 77], dtype=np.int64)
    rows = rng.integers(0, 256, size=(slots.size, row_width), dtype=np.uint8)
    view = pkv.pkv_view(0, 0, bs * row_width, row_width, 0)
    st = pkv.pkv_cache_write(torch.from_numpy(rows).cuda(), None, torch.from_numpy(slots).cuda(),
                             cache, None, view, bs, nb, check=False)
    assert st == 0
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert (b[:WS_PAD] == WS_SENTINEL).all() and (b[WS_PAD + cache_bytes:] == WS_SENTINEL).all()
    ref = init.copy()
    ok = (slots >= 0) & (slots < nb * bs)
    oracle.cache_write(ref, rows[ok], slots[ok], offset=0, layer=0, layer_stride=0,
                       block_stride=bs * row_width, row_width=row_width, block_size=bs,
                       num_blocks=nb)
    assert np.array_equal(b[WS_PAD:WS_PAD + cache_bytes], ref)
    # the out-of-range slot (token 4) was recorded as a slot error, and skipped
    assert pkv.pkv_get_device_error() == (1, 4)
