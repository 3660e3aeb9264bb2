"""Pins of the oracle to things other than itself (CPU only).

Each pin is one of: a value the pages print (tests/golden/, cited there), a
closed form, an invariant, a special case that reduces to a library routine,
or an independent brute force on tiny inputs.  test_oracle_mutations.py then
plants plausible mistakes in a copy of the oracle and checks that these pins
catch every one of them.
"""

import math

import numpy as np
import pytest

from conftest import golden
from paged_kv_cache_131_gb300 import workloads as W


# ---------------------------------------------------------------- fp16 -> f64


def test_half_to_double_exhaustive(orc, lib=None):
    """All 65536 binary16 patterns against numpy's float16 -> float64 conversion."""
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(b), lib=lib) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero too
    assert math.copysign(1.0, orc.half_to_double(0x8000, lib=lib)) == -1.0


# ---------------------------------------------------------------- write side


def test_slot_mapping_worked_example(orc, lib=None):
    g = golden("slot_mapping_example.json")
    bs = g["block_size"]
    # scheduler side (input generator): block_table[130 // 64] = 5 -> slot 322
    table = [0] * 8
    table[g["logical_block"]] = g["block_table_entry_2"]
    assert W.slot_of(table, g["token_position"], bs) == g["slot_mapping"]
    # kernel side (oracle): split the slot back
    assert orc.split_slot(g["slot_mapping"], bs, lib=lib) == (
        g["block_table_entry_2"], g["in_block"])


def test_dsa_block_outer_addresses(orc, lib=None):
    g = golden("dsa_two_cache.json")
    views = W.block_outer_views(W.DSA_PAGES, g["num_layers"], g["block_size"])
    for c in ("mla", "idx"):
        v = views[c]
        assert vars(v) == g["views"][c]
        assert g["block_size"] * v.row_width == g["page_bytes"][c]
    assert views["mla"].block_stride == g["block_bytes"]
    # in-block offsets of [MLA L0 | MLA L1 | IDX L0 | IDX L1]: address of slot 0
    # of block 0 in each (cache, layer)
    offs = []
    for c in ("mla", "idx"):
        v = views[c]
        for layer in range(2):
            offs.append(orc.slot_address(0, g["block_size"], v.offset, layer, v.layer_stride,
                                         v.block_stride, v.row_width, lib=lib))
    assert offs == g["in_block_offsets"][:4]
    # the next block starts at the block size
    v = views["mla"]
    assert orc.slot_address(g["block_size"], g["block_size"], v.offset, 0, v.layer_stride,
                            v.block_stride, v.row_width, lib=lib) == g["in_block_offsets"][4]
    # layer 1, slot 322 (block 5, position 2): the page's term lists
    for c in ("mla", "idx"):
        v = views[c]
        a = orc.slot_address(322, g["block_size"], v.offset, 1, v.layer_stride, v.block_stride,
                             v.row_width, lib=lib)
        assert a == sum(g["layer1_slot322_terms"][c])
    assert sum(g["layer1_slot322_terms"]["mla"]) == 547616
    assert sum(g["layer1_slot322_terms"]["idx"]) == 597000


def test_dsa_layer_outer_addresses(orc, lib=None):
    """LBNHC for NB = 4096 from the layer-outer stride rule (block_stride = page,
    layer_stride = page * NB); slot 322, layer 1."""
    views = W.layer_outer_views(W.DSA_PAGES, 2, 64, 4096)
    assert vars(views["mla"]) == dict(offset=0, layer_stride=171966464, block_stride=41984,
                                      row_width=656)
    assert vars(views["idx"]) == dict(offset=343932928, layer_stride=34603008, block_stride=8448,
                                      row_width=132)
    got = {c: orc.slot_address(322, 64, v.offset, 1, v.layer_stride, v.block_stride,
                               v.row_width, lib=lib) for c, v in views.items()}
    assert got == {"mla": 172177696, "idx": 378578440}


def _write_all(orc, wl, layout, lib=None):
    cache = wl.init.copy()
    for c, v in wl.views[layout].items():
        for layer in range(wl.num_layers):
            orc.cache_write(cache, wl.rows[(c, layer)], wl.slot_mapping, offset=v.offset,
                            layer=layer, layer_stride=v.layer_stride,
                            block_stride=v.block_stride, row_width=v.row_width,
                            block_size=wl.block_size, num_blocks=wl.num_blocks, lib=lib)
    return cache


@pytest.fixture(scope="module")
def small_dsa():
    return W.config5_dsa_write(num_tokens=512, num_blocks=64)


def test_write_ranges_disjoint_and_in_bounds(small_dsa):
    """Distinct (cache, layer, slot) rows occupy disjoint byte ranges inside the
    allocation, for both layouts (pure address arithmetic, brute force)."""
    wl = small_dsa
    for layout, views in wl.views.items():
        spans = []
        for c, v in views.items():
            for layer in range(wl.num_layers):
                for slot in range(wl.num_blocks * wl.block_size):
                    b, o = divmod(slot, wl.block_size)
                    a = v.offset + layer * v.layer_stride + b * v.block_stride + o * v.row_width
                    spans.append((a, a + v.row_width))
        spans.sort()
        assert spans[0][0] == 0 and spans[-1][1] == wl.cache_bytes, layout
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 == b0, layout  # disjoint and gap-free: the layout tiles the buffer


def test_write_round_trip_and_untouched(orc, small_dsa, lib=None):
    wl = small_dsa
    for layout in ("BLHNC", "LBNHC"):
        cache = _write_all(orc, wl, layout, lib=lib)
        touched = np.zeros(wl.cache_bytes, dtype=bool)
        for c, v in wl.views[layout].items():
            for layer in range(wl.num_layers):
                rows = wl.rows[(c, layer)]
                for t, slot in enumerate(wl.slot_mapping):
                    b, o = divmod(int(slot), wl.block_size)
                    a = v.offset + layer * v.layer_stride + b * v.block_stride + o * v.row_width
                    assert np.array_equal(cache[a:a + v.row_width], rows[t])
                    touched[a:a + v.row_width] = True
        assert np.array_equal(cache[~touched], wl.init[~touched])


def test_write_layouts_hold_same_map(orc, small_dsa, lib=None):
    """BLHNC and LBNHC hold the same (cache, layer, block, slot) -> bytes map."""
    wl = small_dsa
    a = _write_all(orc, wl, "BLHNC", lib=lib)
    b = _write_all(orc, wl, "LBNHC", lib=lib)
    va, vb = wl.views["BLHNC"], wl.views["LBNHC"]
    for c in W.DSA_PAGES:
        for layer in range(wl.num_layers):
            for blk in range(wl.num_blocks):
                for o in range(0, wl.block_size, 7):
                    pa = va[c].offset + layer * va[c].layer_stride + blk * va[c].block_stride \
                        + o * va[c].row_width
                    pb = vb[c].offset + layer * vb[c].layer_stride + blk * vb[c].block_stride \
                        + o * vb[c].row_width
                    slot = blk * wl.block_size + o
                    if slot in set(wl.slot_mapping.tolist()):
                        assert np.array_equal(a[pa:pa + va[c].row_width],
                                              b[pb:pb + vb[c].row_width])


def test_write_negative_slot_skipped_and_range_error(orc, lib=None):
    cache = np.zeros(4 * 2 * 8, dtype=np.uint8)  # 4 blocks, bs 2, rows of 8 B
    src = np.arange(3 * 8, dtype=np.uint8).reshape(3, 8)
    n = orc.cache_write(cache, src, np.array([-1, 5, -7]), offset=0, layer=0, layer_stride=0,
                        block_stride=16, row_width=8, block_size=2, num_blocks=4, lib=lib)
    assert n == 1
    assert np.array_equal(cache[40:48], src[1]) and cache[:40].sum() == 0
    with pytest.raises(ValueError):
        orc.cache_write(cache, src[:1], np.array([8]), offset=0, layer=0, layer_stride=0,
                        block_stride=16, row_width=8, block_size=2, num_blocks=4, lib=lib)


# ---------------------------------------------------------------- read side


def brute_force_attention(wl: W.DecodeWorkload, k_cache, v_cache):
    """Independent restatement for tiny inputs: reads each key/value element in
    place from the caches' raw bytes at its byte address (no gather), numpy's
    float16 -> float64, and softmax weights w_j = 1 / sum_k exp(s_k - s_j)."""
    S, H, D = wl.q.shape
    Hk, bs = wl.num_kv_heads, wl.block_size
    kb = k_cache.view(np.uint8).reshape(-1)
    vb = v_cache.view(np.uint8).reshape(-1)
    row_width = Hk * D * 2
    block_stride = bs * row_width

    def elem(buf, slot, kvh, d):
        blk, o = divmod(slot, bs)
        a = blk * block_stride + o * row_width + kvh * D * 2 + d * 2
        return float(buf[a:a + 2].view(np.float16)[0])

    out = np.zeros((S, H, D))
    for i in range(S):
        L = int(wl.seq_lens[i])
        for h in range(H):
            kvh = h // (H // Hk)
            qv = [float(x) for x in wl.q[i, h]]
            slots = [int(wl.block_tables[i, j // bs]) * bs + j % bs for j in range(L)]
            s = [wl.scale * math.fsum(qv[d] * elem(kb, sl, kvh, d) for d in range(D))
                 for sl in slots]
            w = [1.0 / math.fsum(math.exp(sk - sj) for sk in s) for sj in s]
            for d in range(D):
                out[i, h, d] = math.fsum(w[j] * elem(vb, slots[j], kvh, d) for j in range(L))
    return out


def _after_write(orc, wl):
    """The cache state after the new token of each sequence is written (oracle)."""
    k, v = wl.k_cache.copy(), wl.v_cache.copy()
    if wl.slot_mapping is not None:
        row = wl.num_kv_heads * wl.head_dim * 2
        for cache, new in ((k, wl.k_new), (v, wl.v_new)):
            orc.cache_write(cache.view(np.uint8).reshape(-1), new.view(np.uint8), wl.slot_mapping,
                            offset=0, layer=0, layer_stride=0,
                            block_stride=wl.block_size * row, row_width=row,
                            block_size=wl.block_size, num_blocks=wl.num_blocks)
    return k, v


@pytest.mark.parametrize("case", [
    dict(index=101, lens=[1, 5, 16, 17, 33], H=2, Hk=2, D=8),
    dict(index=102, lens=[3, 20, 40], H=4, Hk=2, D=8),
    dict(index=103, lens=[0, 2, 31], H=8, Hk=1, D=4),
])
def test_decode_matches_brute_force(orc, case, lib=None):
    wl = W.small_decode(case["index"], case["lens"], H=case["H"], Hk=case["Hk"], D=case["D"])
    k, v = _after_write(orc, wl)
    got = orc.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale, lib=lib)
    ref = brute_force_attention(wl, k, v)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_decode_config1_brute_force(orc, lib=None):
    wl = W.config1_tiny()
    k, v = _after_write(orc, wl)
    got = orc.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale, lib=lib)
    np.testing.assert_allclose(got, brute_force_attention(wl, k, v), rtol=1e-12, atol=1e-12)


def _one_seq(L, D=16, Hk=1, H=1, bs=4, seed=7):
    """A single sequence in consecutive blocks, the caller fills K and V rows."""
    nb = max(W.blocks_needed(L, bs), 1)
    k = np.zeros((nb, bs, Hk, D), dtype=np.float16)
    v = np.zeros_like(k)
    bt = np.arange(nb, dtype=np.int32)[None, :]
    q = np.zeros((1, H, D), dtype=np.float16)
    return q, k, v, bt, np.array([L], dtype=np.int32)


def test_decode_special_cases(orc, lib=None):
    rng = np.random.default_rng(0)
    # seq_len 1 -> exactly v_0
    q, k, v, bt, sl = _one_seq(1)
    q[:] = W.fp16_normal(rng, q.shape)
    k[0, 0] = W.fp16_normal(rng, k[0, 0].shape)
    v[0, 0] = W.fp16_normal(rng, v[0, 0].shape)
    out = orc.decode_attention(q, k, v, bt, sl, 0.25, lib=lib)
    assert np.array_equal(out[0, 0], v[0, 0, 0].astype(np.float64))
    # all keys equal -> uniform weights -> mean of V
    L = 13
    q, k, v, bt, sl = _one_seq(L)
    q[:] = W.fp16_normal(rng, q.shape)
    k[:] = W.fp16_normal(rng, (1, 1, 1, 16))
    v[:] = W.fp16_normal(rng, v.shape)
    out = orc.decode_attention(q, k, v, bt, sl, 0.25, lib=lib)
    mean = v.reshape(-1, 16)[:L].astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(out[0, 0], mean, rtol=1e-13, atol=1e-13)
    # q = 0 -> mean of V whatever the keys
    q[:] = 0
    k[:] = W.fp16_normal(rng, k.shape)
    out = orc.decode_attention(q, k, v, bt, sl, 0.25, lib=lib)
    np.testing.assert_allclose(out[0, 0], mean, rtol=1e-13, atol=1e-13)
    # two keys: closed-form two-way softmax
    q, k, v, bt, sl = _one_seq(2, D=2)
    q[0, 0] = [1.0, 0.5]
    k[0, 0, 0] = [2.0, 0.0]
    k[0, 1, 0] = [0.0, 3.0]
    v[0, 0, 0] = [1.0, 0.0]
    v[0, 1, 0] = [0.0, 1.0]
    out = orc.decode_attention(q, k, v, bt, sl, 0.5, lib=lib)
    s0, s1 = 0.5 * 2.0, 0.5 * 1.5  # scale * q.k
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    np.testing.assert_allclose(out[0, 0], [w0, 1.0 - w0], rtol=1e-15, atol=1e-15)
    # empty sequence -> zeros
    q, k, v, bt, sl = _one_seq(0)
    out = orc.decode_attention(q, k, v, bt, sl, 0.25, lib=lib)
    assert np.array_equal(out, np.zeros_like(out))


def test_decode_gqa_equals_mha_with_duplicated_kv(orc, lib=None):
    wl = W.small_decode(104, [9, 30, 47], H=8, Hk=2, D=8, write_last=False)
    out = orc.decode_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.seq_lens,
                               wl.scale, lib=lib)
    G = wl.num_heads // wl.num_kv_heads
    k_mha = np.ascontiguousarray(np.repeat(wl.k_cache, G, axis=2))
    v_mha = np.ascontiguousarray(np.repeat(wl.v_cache, G, axis=2))
    ref = orc.decode_attention(wl.q, k_mha, v_mha, wl.block_tables, wl.seq_lens, wl.scale,
                               lib=lib)
    assert np.array_equal(out, ref)
    # and head h really reads KV head h // G: swapping the two KV heads moves
    # each query group's result
    swapped_k = np.ascontiguousarray(wl.k_cache[:, :, ::-1])
    swapped_v = np.ascontiguousarray(wl.v_cache[:, :, ::-1])
    q2 = np.ascontiguousarray(np.concatenate([wl.q[:, G:], wl.q[:, :G]], axis=1))
    out2 = orc.decode_attention(q2, swapped_k, swapped_v, wl.block_tables, wl.seq_lens,
                                wl.scale, lib=lib)
    assert np.array_equal(np.concatenate([out2[:, G:], out2[:, :G]], axis=1), out)


def test_decode_physical_permutation_invariance(orc, lib=None):
    """Relabelling physical blocks (moving their contents along) leaves the
    output unchanged, bit for bit."""
    wl = W.small_decode(105, [7, 16, 40, 64], H=4, Hk=2, D=8, write_last=False)
    out = orc.decode_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.seq_lens,
                               wl.scale, lib=lib)
    perm = np.random.default_rng(1).permutation(wl.num_blocks)
    k2 = np.empty_like(wl.k_cache)
    v2 = np.empty_like(wl.v_cache)
    k2[perm] = wl.k_cache
    v2[perm] = wl.v_cache
    bt2 = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1)
    out2 = orc.decode_attention(wl.q, k2, v2, bt2.astype(np.int32), wl.seq_lens, wl.scale,
                                lib=lib)
    assert np.array_equal(out, out2)


def test_decode_shared_prefix_equals_private_copies(orc, lib=None):
    wl = W.small_decode(106, [40, 45, 57], H=4, Hk=2, D=8, shared_prefix_tokens=32)
    k, v = _after_write(orc, wl)
    out = orc.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale, lib=lib)
    # give every sequence a private copy of its prefix blocks
    S = wl.num_seqs
    nshared = 2
    extra = S * nshared
    k2 = np.concatenate([k, np.zeros((extra,) + k.shape[1:], k.dtype)])
    v2 = np.concatenate([v, np.zeros((extra,) + v.shape[1:], v.dtype)])
    bt2 = wl.block_tables.copy()
    nxt = wl.num_blocks
    for i in range(S):
        for j in range(nshared):
            k2[nxt] = k[bt2[i, j]]
            v2[nxt] = v[bt2[i, j]]
            bt2[i, j] = nxt
            nxt += 1
    assert len(set(wl.block_tables[:, 0])) == 1 and len(set(bt2[:, 0])) == S
    out2 = orc.decode_attention(wl.q, k2, v2, bt2, wl.seq_lens, wl.scale, lib=lib)
    assert np.array_equal(out, out2)


def test_decode_sampled_pairs_match_full(orc, lib=None):
    wl = W.small_decode(107, [10, 33], H=4, Hk=2, D=8, write_last=False)
    full = orc.decode_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.seq_lens,
                                wl.scale, lib=lib)
    pairs = [(1, 3), (0, 0)]
    part = orc.decode_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.seq_lens,
                                wl.scale, pairs=pairs, lib=lib)
    for i, h in pairs:
        assert np.array_equal(part[i, h], full[i, h])
    assert np.isnan(part[1, 0]).all()


def test_decode_bad_block_id_is_an_error(orc, lib=None):
    wl = W.small_decode(108, [20], H=2, Hk=2, D=4, write_last=False)
    bt = wl.block_tables.copy()
    bt[0, 1] = wl.num_blocks
    with pytest.raises(ValueError):
        orc.decode_attention(wl.q, wl.k_cache, wl.v_cache, bt, wl.seq_lens, wl.scale, lib=lib)


# ---------------------------------------------------------------- copy on write


def test_copy_blocks_pages_only(orc, lib=None):
    """Each pair copies exactly the page (block_size * row_width bytes) of every
    requested layer of the source block onto the destination block; nothing
    else changes; src == dst is a no-op (block-outer two-layer view)."""
    rng = np.random.default_rng(11)
    bs, R, NB, L = 4, 12, 6, 3
    page = bs * R
    block_stride = L * page + 8          # block-outer, with a gap after each block
    layer_stride = page
    total = NB * block_stride
    init = rng.integers(0, 256, size=total, dtype=np.uint8)
    cache = init.copy()
    pairs = [(1, 4), (2, 2), (5, 0)]
    n = orc.copy_blocks(cache, pairs, offset=0, layer=1, num_layers=2, layer_stride=layer_stride,
                        block_stride=block_stride, row_width=R, block_size=bs, num_blocks=NB,
                        lib=lib)
    assert n == 4
    exp = init.copy()
    for s, d in pairs:
        if s == d:
            continue
        for layer in (1, 2):
            a = layer * layer_stride + s * block_stride
            b = layer * layer_stride + d * block_stride
            exp[b:b + page] = init[a:a + page]
    assert np.array_equal(cache, exp)
    with pytest.raises(ValueError):
        orc.copy_blocks(cache, [(0, NB)], offset=0, layer=0, num_layers=1,
                        layer_stride=layer_stride, block_stride=block_stride, row_width=R,
                        block_size=bs, num_blocks=NB, lib=lib)
