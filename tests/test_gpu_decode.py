"""GPU parity of paged decode attention against the float64 oracle.

Tolerance (fp16 inputs, fp32 accumulation, fp16 output): every element must
satisfy |gpu - ref| <= 2e-3 + 1e-2 * |ref|.  Small cases and the full-size
workloads (Llama-8B decode layer, long context, shared prefix) compare every
element, plus properties that hold at any size (finite everywhere, inside
the convex hull of the values read).
"""

import numpy as np
import pytest

import oracle
from paged_kv_cache_131_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2
SIMT, MMA = 1, 2
GRID, BALANCED = 1, 2


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_131_gb300 import _build
    _build.build()
    import paged_kv_cache_131_gb300 as m
    assert torch.cuda.is_available()
    m.pkv_get_device_error()
    return m


def assert_close(gpu, ref, pairs=None, what=""):
    g = gpu.astype(np.float64)
    if pairs is not None:
        idx = tuple(np.array(pairs).T)
        g, ref = g[idx], ref[idx]
    assert not np.isnan(ref).any()
    assert np.isfinite(g).all(), f"{what}: {int((~np.isfinite(g)).sum())} non-finite outputs"
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                           f"max |err| {err.max():.3e}, worst excess {(err - bound).max():.3e}")
    return float(err.max())


def oracle_after_write(wl):
    k, v = wl.k_cache.copy(), wl.v_cache.copy()
    if wl.slot_mapping is not None and wl.slot_mapping.size:
        row = wl.num_kv_heads * wl.head_dim * 2
        for cache, new in ((k, wl.k_new), (v, wl.v_new)):
            oracle.cache_write(cache.view(np.uint8).reshape(-1), new.view(np.uint8),
                               wl.slot_mapping, offset=0, layer=0, layer_stride=0,
                               block_stride=wl.block_size * row, row_width=row,
                               block_size=wl.block_size, num_blocks=wl.num_blocks)
    return k, v


def run(wl, **kw):
    from paged_kv_cache_131_gb300.harness import DeviceDecode
    dev = DeviceDecode(wl, **kw)
    out = dev.step().cpu().numpy()
    return dev, out


# ------------------------------------------------------------- small cases


@pytest.mark.parametrize("schedule", [BALANCED, GRID])
@pytest.mark.parametrize("compute", [MMA, SIMT])
def test_config1_tiny_all_elements(pkv, compute, schedule):
    wl = W.config1_tiny()
    dev, out = run(wl, compute=compute, schedule=schedule)
    k, v = oracle_after_write(wl)
    ref = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale)
    assert_close(out, ref, what="config 1")
    assert pkv.pkv_get_device_error() == (0, -1)


SMALL = [
    # (index, lens, H, Hk, D)
    (201, [0, 1, 15, 16, 17, 31, 32, 33, 100, 257, 600, 1100], 8, 8, 128),
    (202, [1, 2, 16, 50, 513, 777], 8, 4, 128),
    (203, [5, 47, 300, 999, 1024, 1500], 16, 4, 128),
    (204, [3, 64, 129, 700], 16, 2, 128),
    (205, [7, 19, 81, 530], 4, 4, 64),
    (206, [16, 33, 400, 1030], 8, 4, 64),
    (207, [9, 200, 520], 16, 2, 64),
    (208, [2, 48, 333, 2049], 8, 1, 64),
]


@pytest.fixture(scope="module", params=SMALL, ids=lambda c: f"{c[0]}-G{c[2]//c[3]}-D{c[4]}")
def small_case(request):
    index, lens, H, Hk, D = request.param
    wl = W.small_decode(index, lens, H=H, Hk=Hk, D=D)
    k, v = oracle_after_write(wl)
    ref = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale)
    return wl, ref


SCHEDULES = [(BALANCED, 0, MMA), (BALANCED, 0, SIMT)] + [
    (GRID, p, c) for p in (0, 16, 48, 128, 8192) for c in (MMA, SIMT)]


@pytest.mark.parametrize("schedule,partition_size,compute", SCHEDULES,
                         ids=lambda v: str(v))
def test_small_all_elements(pkv, small_case, schedule, partition_size, compute):
    wl, ref = small_case
    _, out = run(wl, partition_size=partition_size, compute=compute, schedule=schedule)
    assert_close(out, ref, what=f"s{schedule} P{partition_size} c{compute}")
    assert pkv.pkv_get_device_error() == (0, -1)


def test_balanced_many_short_sequences(pkv):
    """More sequences than CTAs, many empty or one-token ones: every range
    boundary case of the balanced split (whole sequences, cut ones, empty)."""
    lens = [0, 1, 2, 15, 16, 17, 0, 3, 31, 33, 1, 0] * 30 + [700, 5, 1200]
    wl = W.small_decode(217, lens, H=8, Hk=2, D=64)
    k, v = oracle_after_write(wl)
    ref = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale)
    for compute in (MMA, SIMT):
        _, out = run(wl, compute=compute, schedule=BALANCED)
        assert_close(out, ref, what=f"c{compute}")
    assert pkv.pkv_get_device_error() == (0, -1)


@pytest.mark.parametrize("index,lens,H,Hk,D", [
    (221, [0, 1, 17, 600, 1500, 33, 2100], 32, 16, 128),  # 2 groups of 8 KV heads
    (222, [5, 300, 999, 64], 128, 16, 64),                # G 8, 2 groups
    (223, [1, 250, 1300, 16, 700], 12, 12, 128),          # 2 groups of 6
    (224, [40, 700, 3], 40, 40, 64),                      # 5 groups of 8
])
@pytest.mark.parametrize("compute", [MMA, SIMT])
def test_balanced_more_kv_heads_than_a_cta_holds(pkv, index, lens, H, Hk, D, compute):
    """More than 8 KV heads: the balanced schedule takes them in groups (each
    CTA range walks (group, sequence, block)), every element as the oracle."""
    wl = W.small_decode(index, lens, H=H, Hk=Hk, D=D)
    k, v = oracle_after_write(wl)
    ref = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale)
    _, out = run(wl, compute=compute, schedule=BALANCED)
    assert_close(out, ref, what=f"Hk {Hk}")
    assert pkv.pkv_get_device_error() == (0, -1)


REPEAT = [
    # (index, lens, H, Hk, D): ranges of many blocks per CTA
    (231, [3000 + 37 * i for i in range(16)], 32, 8, 128),         # long sequences
    (232, [200 + (i * 53) % 300 for i in range(256)], 32, 8, 128),  # many short ones
    (233, [5000, 17, 2500, 1, 4000, 300] * 4, 64, 8, 128),          # mixed lengths, G 8
    (234, [2000 + 11 * i for i in range(24)], 32, 16, 128),         # 2 head groups
]


@pytest.mark.parametrize("case", REPEAT, ids=lambda c: str(c[0]))
def test_repeated_calls_every_element_same_bits(pkv, case):
    """Calls in a row on one workspace: every call within tolerance of the
    oracle on every element (outputs poisoned before each call, so a merge
    that did not happen shows), the same bits every call (the split is fixed
    by the lengths), the scratch left clean for the next call."""
    from paged_kv_cache_131_gb300.harness import DeviceDecode
    index, lens, H, Hk, D = case
    wl = W.small_decode(index, lens, H=H, Hk=Hk, D=D)
    k, v = oracle_after_write(wl)
    ref = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale,
                                  workers=oracle.default_workers())
    dev = DeviceDecode(wl, schedule=BALANCED)
    dev.write()
    first = None
    for _ in range(4):
        dev.out.fill_(float("nan"))
        out = dev.decode().clone()
        assert_close(out.cpu().numpy(), ref, what=f"case {index}")
        if first is None:
            first = out
        assert torch.equal(out, first)
    assert pkv.pkv_get_device_error() == (0, -1)


def test_schedules_agree(pkv):
    wl = W.small_decode(218, [100, 900, 1600, 3], H=32, Hk=8, D=128)
    a = run(wl, schedule=BALANCED)[1].astype(np.float64)
    b = run(wl, schedule=GRID)[1].astype(np.float64)
    assert np.max(np.abs(a - b)) < 4e-3


def test_single_partition_results_do_not_depend_on_partition_size(pkv):
    """Sequences that fit one partition take the same path: bit-equal outputs."""
    wl = W.small_decode(209, [1, 40, 300, 512], H=8, Hk=2, D=128)
    a = run(wl, partition_size=512, schedule=GRID)[1]
    b = run(wl, partition_size=8192, schedule=GRID)[1]
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


@pytest.mark.parametrize("schedule", [BALANCED, GRID])
def test_physical_permutation_bit_exact(pkv, schedule):
    wl = W.small_decode(210, [33, 700, 1200, 5], H=16, Hk=4, D=128, write_last=False)
    _, out = run(wl, schedule=schedule)
    perm = np.random.default_rng(3).permutation(wl.num_blocks)
    k2 = np.empty_like(wl.k_cache)
    v2 = np.empty_like(wl.v_cache)
    k2[perm] = wl.k_cache
    v2[perm] = wl.v_cache
    bt = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)
    wl2 = W.DecodeWorkload(wl.name, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                           wl.num_blocks, wl.scale, wl.seq_lens, bt, wl.q, k2, v2, None, None,
                           None)
    _, out2 = run(wl2, schedule=schedule)
    assert np.array_equal(out.view(np.uint16), out2.view(np.uint16))


@pytest.mark.parametrize("schedule", [BALANCED, GRID])
def test_shared_prefix_equals_private_copies_bit_exact(pkv, schedule):
    wl = W.small_decode(211, [600, 650, 700, 777], H=16, Hk=2, D=128, shared_prefix_tokens=512)
    dev, out = run(wl, schedule=schedule)
    k = dev.k_cache.cpu().numpy()
    v = dev.v_cache.cpu().numpy()
    S, nshared = wl.num_seqs, 512 // 16
    k2 = np.concatenate([k, np.zeros((S * nshared,) + k.shape[1:], k.dtype)])
    v2 = np.concatenate([v, np.zeros((S * nshared,) + v.shape[1:], v.dtype)])
    bt2 = wl.block_tables.copy()
    nxt = wl.num_blocks
    for i in range(S):
        for j in range(nshared):
            k2[nxt], v2[nxt] = k[bt2[i, j]], v[bt2[i, j]]
            bt2[i, j] = nxt
            nxt += 1
    wl2 = W.DecodeWorkload(wl.name, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                           nxt, wl.scale, wl.seq_lens, bt2, wl.q, k2, v2, None, None, None)
    _, out2 = run(wl2, schedule=schedule)
    assert np.array_equal(out.view(np.uint16), out2.view(np.uint16))


def test_mma_and_simt_agree(pkv):
    wl = W.small_decode(212, [100, 900, 1600], H=32, Hk=8, D=128)
    a = run(wl, compute=MMA)[1].astype(np.float64)
    b = run(wl, compute=SIMT)[1].astype(np.float64)
    assert np.max(np.abs(a - b)) < 4e-3


@pytest.mark.parametrize("schedule", [BALANCED, GRID])
def test_workspace_reuse_and_left_zeroed(pkv, schedule):
    from paged_kv_cache_131_gb300.harness import DeviceDecode
    wl = W.small_decode(213, [1000, 1300, 20], H=8, Hk=2, D=128)
    dev = DeviceDecode(wl, partition_size=64, schedule=schedule)
    first = dev.step().clone()
    for _ in range(3):
        again = dev.decode().clone()
        assert torch.equal(first, again)
    torch.cuda.synchronize()
    tickets = dev.workspace[: wl.num_seqs * wl.num_heads * 4]
    assert int(tickets.sum()) == 0


def test_non_default_stream(pkv):
    from paged_kv_cache_131_gb300.harness import DeviceDecode
    wl = W.small_decode(214, [77, 880], H=8, Hk=2, D=64)
    dev = DeviceDecode(wl)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = dev.step(stream=s)
    s.synchronize()
    k, v = oracle_after_write(wl)
    ref = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale)
    assert_close(out.cpu().numpy(), ref)


def test_concurrent_streams_own_workspaces(pkv):
    """Calls in flight together on four streams, each with its own workspace
    (fp16 on both schedules and FP8): each result matches the oracle, so no
    state is shared between calls beyond the device error record."""
    from paged_kv_cache_131_gb300.harness import DeviceDecode, DeviceDecodeFp8
    cases = [(221, [3000 + 53 * i for i in range(8)], BALANCED),
             (222, [2500 + 71 * i for i in range(12)], BALANCED),
             (223, [1800 + 37 * i for i in range(10)], GRID)]
    devs = []
    for index, lens, schedule in cases:
        wl = W.small_decode(index, lens, H=32, Hk=8, D=128)
        dev = DeviceDecode(wl, schedule=schedule)
        dev.write()
        devs.append((wl, dev))
    wl8 = W.small_decode(224, [2200 + 89 * i for i in range(9)], H=32, Hk=8, D=128)
    dev8 = DeviceDecodeFp8(wl8)
    dev8.write()
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(4)]
    for _ in range(3):
        for (wl, dev), s in zip(devs, streams):
            with torch.cuda.stream(s):
                dev.out.fill_(float("nan"))
                dev.decode(stream=s)
        with torch.cuda.stream(streams[3]):
            dev8.out.fill_(float("nan"))
            dev8.decode(stream=streams[3])
    torch.cuda.synchronize()
    for wl, dev in devs:
        k, v = oracle_after_write(wl)
        ref = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale,
                                      workers=oracle.default_workers())
        assert_close(dev.out.cpu().numpy(), ref)
    from test_gpu_fp8 import _oracle_fp8_state
    k8, v8, ks, vs = _oracle_fp8_state(wl8, workers=oracle.default_workers())
    ref8 = oracle.decode_attention_fp8(wl8.q, k8, v8, ks, vs, wl8.block_tables, wl8.seq_lens,
                                       wl8.scale, workers=oracle.default_workers())
    assert_close(dev8.out.cpu().numpy(), ref8)
    assert pkv.pkv_get_device_error() == (0, -1)


# ------------------------------------------------------------- bad data


@pytest.mark.parametrize("schedule", [BALANCED, GRID])
def test_bad_block_id_recorded_skipped_no_fault(pkv, schedule):
    from paged_kv_cache_131_gb300.harness import DeviceDecode
    wl = W.small_decode(215, [40, 40], H=4, Hk=4, D=128, write_last=False)
    dev = DeviceDecode(wl, schedule=schedule)
    bt = dev.block_tables.clone()
    bt[1, 1] = wl.num_blocks + 7  # second block of sequence 1
    dev.block_tables.copy_(bt)
    out = dev.decode().cpu().numpy()
    kind, index = pkv.pkv_get_device_error()
    assert kind == 2 and index == 1 * wl.max_blocks_per_seq + 1
    # sequence 0 is untouched by the bad entry
    ref = oracle.decode_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.seq_lens,
                                  wl.scale)
    assert_close(out[:1], ref[:1])
    # sequence 1 equals attention over its remaining (valid) positions
    keep = [j for j in range(40) if j // 16 != 1]
    k1 = np.concatenate([wl.k_cache[wl.block_tables[1, j // 16], j % 16][None] for j in keep])
    v1 = np.concatenate([wl.v_cache[wl.block_tables[1, j // 16], j % 16][None] for j in keep])
    q1 = wl.q[1].astype(np.float64)
    s = np.einsum("hd,jhd->hj", q1, k1.astype(np.float64)) * wl.scale
    w = np.exp(s - s.max(axis=1, keepdims=True))
    exp = np.einsum("hj,jhd->hd", w / w.sum(axis=1, keepdims=True), v1.astype(np.float64))
    assert_close(out[1:2], exp[None])


@pytest.mark.parametrize("schedule", [BALANCED, GRID])
def test_seq_len_beyond_table_recorded_no_fault(pkv, schedule):
    from paged_kv_cache_131_gb300.harness import DeviceDecode
    wl = W.small_decode(216, [20, 30], H=4, Hk=4, D=64, write_last=False)
    dev = DeviceDecode(wl, schedule=schedule)
    sl = dev.seq_lens.clone()
    sl[0] = wl.max_blocks_per_seq * 16 + 100
    dev.seq_lens.copy_(sl)
    dev.decode()
    kind, index = pkv.pkv_get_device_error()
    assert (kind, index) == (3, 0)
    sl[0] = -5
    dev.seq_lens.copy_(sl)
    out = dev.decode().cpu().numpy()
    assert pkv.pkv_get_device_error() == (3, 0)
    assert np.all(out[0] == 0)


# ------------------------------------------------------------- full size


def _hull_check(out, v_after):
    """Every output lies inside [min v, max v] of its KV head's values (a
    convex combination), and nothing is NaN (poisoned slots never leak in)."""
    assert np.isfinite(out).all()
    vmax = float(np.nanmax(np.abs(v_after[np.isfinite(v_after)])))
    assert np.abs(out.astype(np.float64)).max() <= vmax + ATOL


_FULL = {}


@pytest.fixture(scope="module", params=[2, 3, 4], ids=lambda c: f"config{c}")
def full_case(request):
    """Workload, post-write caches and the oracle's every output row of a
    full-size config, computed once per config (the oracle's rows are split
    over the host's cores; each row is the same single-threaded float64
    computation)."""
    cfg = request.param
    if cfg not in _FULL:
        _FULL.clear()
        wl = W.config(cfg)
        k, v = oracle_after_write(wl)
        ref = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale,
                                      workers=oracle.default_workers())
        _FULL[cfg] = (cfg, wl, k, v, ref)
    return _FULL[cfg]


@pytest.mark.parametrize("schedule,compute", [(BALANCED, MMA), (BALANCED, SIMT), (GRID, MMA),
                                              (GRID, SIMT)])
def test_full_size_configs_all_elements(pkv, full_case, schedule, compute):
    cfg, wl, k, v, ref = full_case
    dev, out = run(wl, compute=compute, schedule=schedule)
    assert pkv.pkv_get_device_error() == (0, -1)
    assert_close(out, ref, what=f"config {cfg}")
    _hull_check(out, v)
