"""GPU parity of the batched multi-view write and of the copy-on-write block
copy against the oracle (bit-exact), and an end-to-end copy-on-write flow on
the device: copy the shared partial block, write the tails, decode."""

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
    m.pkv_get_device_error()
    return m


@pytest.fixture(scope="module")
def dsa():
    return W.config5_dsa_write()


def _oracle_layout(wl, layout):
    ref = wl.init.copy()
    for c, v in wl.views[layout].items():
        for layer in range(wl.num_layers):
            oracle.cache_write(ref, wl.rows[(c, layer)], wl.slot_mapping, offset=v.offset,
                               layer=layer, layer_stride=v.layer_stride,
                               block_stride=v.block_stride, row_width=v.row_width,
                               block_size=wl.block_size, num_blocks=wl.num_blocks)
    return ref


@pytest.mark.parametrize("layout", ["BLHNC", "LBNHC"])
def test_write_multi_dsa_one_launch_bit_exact(pkv, dsa, layout):
    from paged_kv_cache_131_gb300.harness import DeviceWrite
    dev = DeviceWrite(dsa)
    assert dev.write_layout_batched(layout) == 1
    assert np.array_equal(dev.cache.cpu().numpy(), _oracle_layout(dsa, layout))
    assert pkv.pkv_get_device_error() == (0, -1)


def test_write_multi_mixed_alignment_and_padding(pkv):
    rng = np.random.default_rng(21)
    bs, nb, T = 16, 20, 200
    widths = [656, 132, 7, 2048]
    total = 0
    views = []
    for R in widths:  # layer-outer regions one after another, odd offsets for R = 7
        off = total + (3 if R == 7 else 0)
        views.append(pkv.pkv_view(off, nb * bs * R, bs * R, R, 1))
        total = off + 2 * nb * bs * R
    init = rng.integers(0, 256, size=total, dtype=np.uint8)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[::9] = -1
    rows = [rng.integers(0, 256, size=(T, R), dtype=np.uint8) for R in widths]
    cache = torch.from_numpy(init.copy()).cuda()
    writes = [(torch.from_numpy(r).cuda(), cache, v) for r, v in zip(rows, views)]
    pkv.pkv_cache_write_multi(writes, torch.from_numpy(slots).cuda(), bs, nb)
    ref = init.copy()
    for r, v in zip(rows, views):
        oracle.cache_write(ref, r, slots, offset=v.offset, layer=v.layer,
                           layer_stride=v.layer_stride, block_stride=v.block_stride,
                           row_width=v.row_width, block_size=bs, num_blocks=nb)
    assert np.array_equal(cache.cpu().numpy(), ref)
    assert pkv.pkv_get_device_error() == (0, -1)


@pytest.mark.parametrize("layout", ["BLHNC", "LBNHC"])
def test_copy_blocks_dsa_views_bit_exact(pkv, dsa, layout):
    rng = np.random.default_rng(22)
    src = rng.choice(dsa.num_blocks, size=300, replace=False)
    dst = rng.choice(np.setdiff1d(np.arange(dsa.num_blocks), src), size=300, replace=False)
    pairs = np.stack([src, dst], axis=1).astype(np.int64)
    pairs[7] = [pairs[7, 0], pairs[7, 0]]  # src == dst: nothing to do
    cache = torch.from_numpy(dsa.init.copy()).cuda()
    mapping = torch.from_numpy(pairs).cuda()
    ref = dsa.init.copy()
    for c, v in dsa.views[layout].items():
        pkv.pkv_copy_blocks(cache, pkv.pkv_view(v.offset, v.layer_stride, v.block_stride,
                                                v.row_width, 0),
                            dsa.num_layers, dsa.block_size, mapping, dsa.num_blocks)
        oracle.copy_blocks(ref, pairs, offset=v.offset, layer=0, num_layers=dsa.num_layers,
                           layer_stride=v.layer_stride, block_stride=v.block_stride,
                           row_width=v.row_width, block_size=dsa.block_size,
                           num_blocks=dsa.num_blocks)
    assert np.array_equal(cache.cpu().numpy(), ref)
    assert pkv.pkv_get_device_error() == (0, -1)


def test_copy_blocks_bad_id_recorded_and_skipped(pkv):
    bs, R, nb = 16, 64, 8
    init = np.random.default_rng(23).integers(0, 256, size=nb * bs * R, dtype=np.uint8)
    cache = torch.from_numpy(init.copy()).cuda()
    mapping = torch.tensor([[1, 2], [3, nb], [4, 5]], dtype=torch.int64, device="cuda")
    pkv.pkv_copy_blocks(cache, pkv.pkv_view(0, 0, bs * R, R, 0), 1, bs, mapping, nb)
    assert pkv.pkv_get_device_error() == (2, 1)
    ref = init.copy()
    oracle.copy_blocks(ref, [(1, 2), (4, 5)], offset=0, layer=0, num_layers=1, layer_stride=0,
                       block_stride=bs * R, row_width=R, block_size=bs, num_blocks=nb)
    assert np.array_equal(cache.cpu().numpy(), ref)


def test_copy_on_write_end_to_end(pkv):
    """A 1995-token shared prefix ends inside block 124: before the sequences
    write their tails there, every writer but the last copies it
    ("vLLM 技术内幕" §2.2).  Device: pkv_copy_blocks, tail writes, the new
    token's write, decode.  The caches must equal the generator's state and
    the output the oracle's."""
    from paged_kv_cache_131_gb300.harness import DeviceDecode
    S, bs = 4, 16
    wl = W.small_decode(403, [1995 + 23, 1995 + 9, 1995 + 40, 1995 + 2], H=8, Hk=2, D=128,
                        shared_prefix_tokens=1995)
    assert wl.cow_pairs.shape == (S - 1, 2)
    row = wl.num_kv_heads * wl.head_dim * 2
    # the state before copy on write and before any tail token was written
    tail_slots, tail_k, tail_v = [], [], []
    kflat = wl.k_cache.reshape(wl.num_blocks * bs, -1)
    vflat = wl.v_cache.reshape(wl.num_blocks * bs, -1)
    for i in range(S):
        for pos in range(1995, int(wl.seq_lens[i]) - 1):
            s = W.slot_of(wl.block_tables[i], pos, bs)
            tail_slots.append(s)
            tail_k.append(kflat[s].copy())
            tail_v.append(vflat[s].copy())
    k0, v0 = wl.k_cache.copy(), wl.v_cache.copy()
    nan = np.float16(np.nan)
    for cache, flat in ((k0, k0.reshape(wl.num_blocks * bs, -1)),
                        (v0, v0.reshape(wl.num_blocks * bs, -1))):
        flat[tail_slots] = nan
        for _, dst in wl.cow_pairs:
            cache[dst] = nan
    dev = DeviceDecode(W.DecodeWorkload(wl.name, wl.num_heads, wl.num_kv_heads, wl.head_dim, bs,
                                        wl.num_blocks, wl.scale, wl.seq_lens, wl.block_tables,
                                        wl.q, k0, v0, wl.k_new, wl.v_new, wl.slot_mapping))
    mapping = torch.from_numpy(wl.cow_pairs).cuda()
    view = dev.view()
    for cache in (dev.k_cache, dev.v_cache):
        pkv.pkv_copy_blocks(cache, view, 1, bs, mapping, wl.num_blocks)
    ts = torch.tensor(tail_slots, dtype=torch.int64, device="cuda")
    pkv.pkv_cache_write(torch.from_numpy(np.stack(tail_k)).cuda(),
                        torch.from_numpy(np.stack(tail_v)).cuda(), ts, dev.k_cache, dev.v_cache,
                        view, bs, wl.num_blocks)
    out = dev.step().cpu().numpy().astype(np.float64)
    assert pkv.pkv_get_device_error() == (0, -1)
    # caches equal the generator's (oracle-side) state after the new token's write
    k_ref, v_ref = wl.k_cache.copy(), wl.v_cache.copy()
    for cache, new in ((k_ref, wl.k_new), (v_ref, wl.v_new)):
        oracle.cache_write(cache.view(np.uint8).reshape(-1), new.view(np.uint8), wl.slot_mapping,
                           offset=0, layer=0, layer_stride=0, block_stride=bs * row,
                           row_width=row, block_size=bs, num_blocks=wl.num_blocks)
    assert np.array_equal(dev.k_cache.cpu().numpy().view(np.uint16), k_ref.view(np.uint16))
    assert np.array_equal(dev.v_cache.cpu().numpy().view(np.uint16), v_ref.view(np.uint16))
    ref = oracle.decode_attention(wl.q, k_ref, v_ref, wl.block_tables, wl.seq_lens, wl.scale)
    err = np.abs(out - ref)
    assert (err <= 2e-3 + 1e-2 * np.abs(ref)).all(), err.max()
