"""Host-side logic of the input generators (CPU only): the block pool and
table builder against the pages' worked numbers, copy on write, the fp16
normal sampler, and the shapes of the five workloads."""

import math

import numpy as np
import pytest

from conftest import golden
from paged_kv_cache_131_gb300 import workloads as W


def test_block_counts_of_the_worked_example():
    """"deep-dive-into-vllm-05" §1.3: 2050 prompt tokens -> 129 blocks (the last
    holds 2), 2350 after 300 generated -> 147, a 2000-token prompt = 125 full."""
    g = golden("block_counts.json")
    bs = g["block_size"]
    for case in g["cases"]:
        assert W.blocks_needed(case["tokens"], bs) == case["blocks"]
    # the same through the pool: prefill, then decode token by token
    pool = W.BlockPool(1000)
    seq = W.Sequence()
    W.prefill(pool, seq, 2050, bs)
    assert len(seq.block_table) == 129 and 2050 - 128 * bs == 2
    for _ in range(300):
        W.append_slot(pool, seq, bs)
    assert len(seq.block_table) == 147 and seq.seq_len == 2350
    assert pool.num_free() == 1000 - 147


def test_decode_takes_a_block_only_on_a_boundary():
    pool = W.BlockPool(8, order=[7, 6, 5, 4, 3, 2, 1, 0])
    seq = W.Sequence()
    W.prefill(pool, seq, 16, 16)
    assert seq.block_table == [0]
    logical, pos, cow = W.append_slot(pool, seq, 16)  # token 16 starts block 1
    assert (logical, pos, cow) == (1, 0, None) and seq.block_table == [0, 1]
    for _ in range(15):
        W.append_slot(pool, seq, 16)
    assert seq.block_table == [0, 1]
    W.append_slot(pool, seq, 16)
    assert seq.block_table == [0, 1, 2]


def test_block_table_example_and_slot_formula():
    """"deep-dive-into-vllm-05" §1.2: VB0->PB7, VB1->PB13, VB2->PB21 for tokens
    t1..t48 in blocks of 16; slot = physical block * bs + offset."""
    g = golden("block_tables.json")
    table = g["example_1"]["table"]
    bs = g["example_1"]["block_size"]
    assert [W.slot_of(table, p, bs) for p in (0, 15, 16, 31, 32, 47)] == \
        [7 * 16, 7 * 16 + 15, 13 * 16, 13 * 16 + 15, 21 * 16, 21 * 16 + 15]
    # "KV Cache 与推理服务内存管理": a pool whose free list yields 17, 3, 25 then
    # 8, 11 builds Request A's and Request B's tables
    pool = W.BlockPool(32, order=[11, 8, 25, 3, 17])
    a, b = W.Sequence(), W.Sequence()
    W.prefill(pool, a, 40, 16)
    W.prefill(pool, b, 20, 16)
    assert a.block_table == g["example_2"]["A"] and b.block_table == g["example_2"]["B"]


def test_out_of_blocks_and_double_free():
    pool = W.BlockPool(3)
    seq = W.Sequence()
    with pytest.raises(W.OutOfBlocks):
        W.prefill(pool, seq, 4 * 16, 16)
    blocks = pool.allocate(2)
    pool.free(blocks)
    assert pool.num_free() == 3
    with pytest.raises(RuntimeError):
        pool.free(blocks)


def test_shared_prefix_ref_counts_and_copy_on_write():
    """"vLLM 技术内幕" §2.2: writing into a block with ref_cnt > 1 first copies it.
    A 2000-token prefix is 125 full blocks: no copy; a 1995-token one ends in a
    shared partial block that each writer but the last copies."""
    wl = W.small_decode(401, [2000 + 7, 2000 + 20, 2000 + 1], H=2, Hk=2, D=8,
                        shared_prefix_tokens=2000)
    shared = wl.block_tables[:, :125]
    assert (shared == shared[0]).all() and (wl.ref_cnt[shared[0]] == 3).all()
    assert len({int(wl.block_tables[i, 125]) for i in range(3)}) == 3  # private tails

    S = 4
    wl = W.small_decode(402, [1995 + 10] * S, H=2, Hk=2, D=8, shared_prefix_tokens=1995)
    last_shared = wl.block_tables[:, 124]
    # every sequence but the last got a private copy of logical block 124; the
    # last writes into the original, whose count has dropped to one
    assert len(set(last_shared.tolist())) == S
    assert all(wl.ref_cnt[b] == 1 for b in last_shared)
    # every copy holds the prefix rows 1984..1994 (positions 0..10 of block 124)
    first = wl.k_cache[last_shared[0], :11].view(np.uint16)
    for i in range(1, S):
        assert np.array_equal(wl.k_cache[last_shared[i], :11].view(np.uint16), first)
    assert not np.isnan(wl.k_cache[last_shared[0], :11].astype(np.float32)).any()


def test_fp16_normal_sampler():
    t = W.normal_fp16_table().astype(np.float64)
    assert np.all(np.diff(t) >= 0)  # quantiles are non-decreasing
    assert abs(t.mean()) < 1e-6  # symmetric quantile grid
    assert abs(t.std() - 1.0) < 2e-3
    x = W.fp16_normal(np.random.Generator(np.random.PCG64(0)), (1 << 20,)).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    # seeded: same seed, same values
    a = W.fp16_normal(W.rng_for(9), (64,))
    b = W.fp16_normal(W.rng_for(9), (64,))
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_config1_shapes_and_poison():
    wl = W.config1_tiny()
    assert wl.seq_lens.tolist() == [1, 17, 33, 50]
    assert (wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size) == (4, 4, 64, 16)
    assert wl.scale == 1 / 8
    used = wl.block_tables[wl.block_tables >= 0]
    assert used.size == 1 + 2 + 3 + 4 and len(set(used.tolist())) == used.size  # no reuse
    # the new token's slot is the last position of each sequence
    for i, L in enumerate(wl.seq_lens):
        assert wl.slot_mapping[i] == W.slot_of(wl.block_tables[i], int(L) - 1, 16)
    # every slot no sequence has written yet is NaN (poison)
    flat = wl.k_cache.reshape(32 * 16, -1)
    written = {W.slot_of(wl.block_tables[i], p, 16)
               for i, L in enumerate(wl.seq_lens) for p in range(int(L) - 1)}
    for s in range(32 * 16):
        assert np.isnan(flat[s]).all() != (s in written)


def test_dsa_workload_shapes():
    wl = W.config5_dsa_write(num_tokens=256, num_blocks=16)
    assert wl.cache_bytes == 16 * 100864
    assert len(set(wl.slot_mapping.tolist())) == 256  # without replacement
    assert wl.slot_mapping.min() >= 0 and wl.slot_mapping.max() < 16 * 64
    assert wl.rows[("mla", 1)].shape == (256, 656) and wl.rows[("idx", 0)].shape == (256, 132)


def test_config_sequence_length_mix():
    """Lengths of configs 2 and 4 follow their stated ranges (lengths only:
    the full caches are not built here)."""
    rng = W.rng_for(2)
    lens = rng.integers(256, 4096, size=64, endpoint=True)
    assert lens.min() >= 256 and lens.max() <= 4096
    tails = W.rng_for(4).integers(1, 300, size=256, endpoint=True)
    assert tails.min() >= 1 and tails.max() <= 300
    assert math.ceil(2000 / 16) == 125
