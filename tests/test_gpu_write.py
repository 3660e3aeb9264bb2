"""GPU parity of the paged KV-cache write against the oracle: bit-exact bytes,
untouched bytes included."""

import numpy as np
import pytest

import oracle
from paged_kv_cache_131_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_131_gb300 import _build
    _build.build()
    import paged_kv_cache_131_gb300 as m
    assert torch.cuda.is_available()
    m.pkv_get_device_error()  # start from a clean device error record
    return m


def _oracle_decode_write(wl):
    """Oracle cache state after writing the workload's new rows."""
    k, v = wl.k_cache.copy(), wl.v_cache.copy()
    row = wl.num_kv_heads * wl.head_dim * 2
    for cache, new in ((k, wl.k_new), (v, wl.v_new)):
        oracle.cache_write(cache.view(np.uint8).reshape(-1), new.view(np.uint8), wl.slot_mapping,
                           offset=0, layer=0, layer_stride=0, block_stride=wl.block_size * row,
                           row_width=row, block_size=wl.block_size, num_blocks=wl.num_blocks)
    return k, v


def _bytes(t):
    return t.cpu().contiguous().view(torch.uint8).numpy().reshape(-1)


@pytest.mark.parametrize("cfg", [1, 2])
def test_decode_config_write_bit_exact(pkv, cfg):
    from paged_kv_cache_131_gb300.harness import DeviceDecode
    wl = W.config(cfg)
    dev = DeviceDecode(wl)
    dev.write()
    k_ref, v_ref = _oracle_decode_write(wl)
    assert np.array_equal(_bytes(dev.k_cache), k_ref.view(np.uint8).reshape(-1))
    assert np.array_equal(_bytes(dev.v_cache), v_ref.view(np.uint8).reshape(-1))
    assert pkv.pkv_get_device_error() == (0, -1)


@pytest.fixture(scope="module")
def dsa():
    return W.config5_dsa_write()


@pytest.mark.parametrize("layout", ["BLHNC", "LBNHC"])
def test_dsa_two_cache_write_bit_exact(pkv, dsa, layout):
    from paged_kv_cache_131_gb300.harness import DeviceWrite
    dev = DeviceWrite(dsa)
    n = dev.write_layout(layout)
    assert n == 4
    ref = dsa.init.copy()
    for c, v in dsa.views[layout].items():
        for layer in range(dsa.num_layers):
            oracle.cache_write(ref, dsa.rows[(c, layer)], dsa.slot_mapping, offset=v.offset,
                               layer=layer, layer_stride=v.layer_stride,
                               block_stride=v.block_stride, row_width=v.row_width,
                               block_size=dsa.block_size, num_blocks=dsa.num_blocks)
    got = dev.cache.cpu().numpy()
    assert np.array_equal(got, ref)
    assert pkv.pkv_get_device_error() == (0, -1)


@pytest.mark.parametrize("row_width,offset,block_stride", [
    (656, 0, 64 * 656),        # 16-byte rows
    (132, 16, 64 * 132 + 8),   # 4-byte rows
    (24, 8, 64 * 24 + 8),      # 8-byte rows
    (6, 2, 64 * 6 + 2),        # 2-byte rows
    (7, 3, 64 * 7 + 1),        # byte rows, odd offset
    (4096, 0, 64 * 4096),      # wide rows (4 rows per 16 KB batch)
    (20000, 0, 64 * 20000),    # a row wider than one batch: one token, two rounds
    (50000, 8, 64 * 50000 + 8),  # 8-byte vectors, seven rounds of one row
])
def test_write_alignment_paths(pkv, row_width, offset, block_stride):
    rng = np.random.default_rng(row_width)
    bs, nb, T, layers = 64, 12, 300 if row_width < 10000 else 40, 2
    layer_stride = nb * block_stride + 16
    total = offset + layers * layer_stride + nb * block_stride
    init = rng.integers(0, 256, size=total, dtype=np.uint8)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[::17] = -1  # padding tokens
    rows_k = rng.integers(0, 256, size=(T, row_width), dtype=np.uint8)
    rows_v = rng.integers(0, 256, size=(T, row_width), dtype=np.uint8)
    kc = torch.from_numpy(init.copy()).cuda()
    vc = torch.from_numpy(init[::-1].copy()).cuda()
    view = pkv.pkv_view(offset, layer_stride, block_stride, row_width, 1)
    pkv.pkv_cache_write(torch.from_numpy(rows_k).cuda(), torch.from_numpy(rows_v).cuda(),
                        torch.from_numpy(slots).cuda(), kc, vc, view, bs, nb)
    ref_k, ref_v = init.copy(), init[::-1].copy()
    for ref, rows in ((ref_k, rows_k), (ref_v, rows_v)):
        oracle.cache_write(ref, rows, slots, offset=offset, layer=1, layer_stride=layer_stride,
                           block_stride=block_stride, row_width=row_width, block_size=bs,
                           num_blocks=nb)
    assert np.array_equal(kc.cpu().numpy(), ref_k)
    assert np.array_equal(vc.cpu().numpy(), ref_v)
    assert pkv.pkv_get_device_error() == (0, -1)


def test_write_single_cache_and_empty(pkv):
    rng = np.random.default_rng(5)
    bs, nb, R = 16, 4, 64
    init = rng.integers(0, 256, size=nb * bs * R, dtype=np.uint8)
    cache = torch.from_numpy(init.copy()).cuda()
    rows = rng.integers(0, 256, size=(3, R), dtype=np.uint8)
    slots = np.array([5, 63, 0], dtype=np.int64)
    view = pkv.pkv_view(0, 0, bs * R, R, 0)
    pkv.pkv_cache_write(torch.from_numpy(rows).cuda(), None, torch.from_numpy(slots).cuda(),
                        cache, None, view, bs, nb)
    ref = init.copy()
    oracle.cache_write(ref, rows, slots, offset=0, layer=0, layer_stride=0, block_stride=bs * R,
                       row_width=R, block_size=bs, num_blocks=nb)
    assert np.array_equal(cache.cpu().numpy(), ref)
    # zero tokens: nothing changes
    empty = torch.empty(0, dtype=torch.int64, device="cuda")
    pkv.pkv_cache_write(torch.empty(0, R, dtype=torch.uint8, device="cuda"), None, empty, cache,
                        None, view, bs, nb)
    assert np.array_equal(cache.cpu().numpy(), ref)


def test_write_out_of_range_slot_recorded_and_skipped(pkv):
    bs, nb, R = 16, 4, 32
    cache = torch.zeros(nb * bs * R, dtype=torch.uint8, device="cuda")
    rows = torch.full((3, R), 7, dtype=torch.uint8, device="cuda")
    slots = torch.tensor([1, nb * bs, 2], dtype=torch.int64, device="cuda")
    pkv.pkv_cache_write(rows, None, slots, cache, None, pkv.pkv_view(0, 0, bs * R, R, 0), bs, nb)
    kind, index = pkv.pkv_get_device_error()
    assert (kind, index) == (1, 1)
    got = cache.cpu().numpy().reshape(nb * bs, R)
    assert (got[1] == 7).all() and (got[2] == 7).all()
    got[1:3] = 0
    assert got.sum() == 0
    assert pkv.pkv_get_device_error() == (0, -1)  # reading clears it


@pytest.mark.parametrize("row_width,T,vec_note", [
    (24, 430001, "8-byte vectors, a tail past the last 16-byte multiple"),
    (18, 580001, "2-byte vectors, odd tail"),
    (656, 16385, "16-byte vectors, one token past a full item"),
])
def test_large_write_many_items_per_cta(pkv, row_width, T, vec_note):
    """Writes of ~10 MB of rows: several batches per CTA, odd row widths and
    token counts; bytes exact, padding and a bad slot skipped, the bad slot
    recorded once."""
    rng = np.random.default_rng(T)
    bs = 64
    nb = T // bs + 50
    offset, block_stride = 16, bs * row_width + (8 if row_width % 8 == 0 else 2)
    total = offset + nb * block_stride
    init = rng.integers(0, 256, size=total, dtype=np.uint8)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[::1001] = -1
    slots[7] = nb * bs + 3  # out of range: skipped and recorded
    rows = rng.integers(0, 256, size=(T, row_width), dtype=np.uint8)
    cache = torch.from_numpy(init.copy()).cuda()
    view = pkv.pkv_view(offset, 0, block_stride, row_width, 0)
    pkv.pkv_cache_write(torch.from_numpy(rows).cuda(), None, torch.from_numpy(slots).cuda(),
                        cache, None, view, bs, nb)
    assert pkv.pkv_get_device_error() == (1, 7)
    ok = slots < nb * bs
    ref = init.copy()
    oracle.cache_write(ref, rows[ok], slots[ok], offset=offset, layer=0, layer_stride=0,
                       block_stride=block_stride, row_width=row_width, block_size=bs,
                       num_blocks=nb)
    assert np.array_equal(cache.cpu().numpy(), ref), vec_note
