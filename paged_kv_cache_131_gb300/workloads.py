"""Seeded synthetic workloads for the paged KV-cache hot path.

This module produces INPUTS only -- block tables, sequence lengths, slot
mappings, fp16 query/key/value data, cache byte images and cache views.  It
holds none of the arithmetic of the write (the slot split and the address
formula) or of attention; both the CUDA library's callers and the oracle take
their inputs from here.

Sources for the shapes (page title -- section):
  - "deep-dive-into-vllm-05" §1.2: per-layer KV layout
    [num_blocks, block_size, num_kv_heads, head_dim], fp16; §1.3 worked block
    counts (2050 tokens -> 129 blocks, 2350 -> 147, a 2000-token prompt is 125
    full blocks).
  - "KV Cache 与推理服务内存管理" (PagedAttention pseudo-code): a pool of free
    physical block ids; prefill takes ceil(len / BLOCK_SIZE) blocks, decode
    takes a new block only when it crosses a block boundary, finish returns the
    blocks.  Physical ids need not be contiguous.
  - "vLLM KV Cache Layout 可视化": slot_mapping = block * block_size +
    in-block position is computed by the scheduler, once per token, and is
    shared by every cache and layer (查一个 token); the layout stride rules and
    the two-cache (MLA 656 B + indexer 132 B per token) example
    (layout 是什么 / 两种 cache 共用一张 block table / 具体例子).
  - "vLLM 技术内幕" §2.2: shared blocks carry a reference count; writing to a
    block whose count is above one first copies it (copy on write).

Random numbers: numpy PCG64 seeded with 1000 + the workload's index.  fp16
N(0, 1) values are drawn by inverse transform at fp16 resolution: a uniform
16-bit integer u indexes a table holding the standard normal quantile at
(u + 0.5) / 65536, rounded to fp16 (nearest-even).  This is N(0, 1) sampled
on a 2^-16 probability grid (|x| <= 4.3); it is an order of magnitude faster
than float32 normal draws followed by a float16 cast, which matters for the
gigabyte-sized caches.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from statistics import NormalDist

import numpy as np

FP16_NAN_BITS = 0x7E00  # quiet NaN: poison for every slot no sequence owns


def rng_for(index: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(1000 + index))


def blocks_needed(num_tokens: int, block_size: int) -> int:
    """ceil(num_tokens / block_size): the blocks a prefill of that many tokens takes."""
    return -(-num_tokens // block_size)


class OutOfBlocks(RuntimeError):
    """The pool cannot supply the blocks a request needs (it cannot be scheduled)."""


class BlockPool:
    """Host free list of physical block ids with reference counts.

    ``order`` fixes the free list (popped from the end, as the pages' pool
    does); by default a seeded shuffle of range(num_blocks).
    """

    def __init__(self, num_blocks: int, rng: np.random.Generator | None = None,
                 order=None):
        if order is None:
            order = np.arange(num_blocks) if rng is None else rng.permutation(num_blocks)
        self.num_blocks = num_blocks
        self.free_list = [int(b) for b in order]
        self.ref_cnt = np.zeros(num_blocks, dtype=np.int64)

    def num_free(self) -> int:
        return len(self.free_list)

    def allocate(self, n: int) -> list[int]:
        if n > len(self.free_list):
            raise OutOfBlocks(f"need {n} blocks, {len(self.free_list)} free")
        out = [self.free_list.pop() for _ in range(n)]
        self.ref_cnt[out] += 1
        return out

    def share(self, blocks) -> None:
        """Another sequence maps these blocks too (ref_cnt += 1)."""
        self.ref_cnt[list(blocks)] += 1

    def free(self, blocks) -> None:
        """Drop one reference per block; blocks that reach zero go back to the pool."""
        for b in reversed(list(blocks)):
            if self.ref_cnt[b] <= 0:
                raise RuntimeError(f"double free of block {b}")
            self.ref_cnt[b] -= 1
            if self.ref_cnt[b] == 0:
                self.free_list.append(int(b))


@dataclass
class Sequence:
    block_table: list[int] = field(default_factory=list)
    seq_len: int = 0


def prefill(pool: BlockPool, seq: Sequence, num_tokens: int, block_size: int) -> None:
    """Take ceil(num_tokens / block_size) new blocks for a prompt."""
    seq.block_table.extend(pool.allocate(blocks_needed(num_tokens, block_size)))
    seq.seq_len = num_tokens


def append_slot(pool: BlockPool, seq: Sequence, block_size: int):
    """Reserve the slot of the next token; a new block only on a boundary.

    Returns (logical block, in-block position) of the new token.  A shared
    last block (ref_cnt > 1) is copied on write first: the sequence gets a
    private block and the caller must copy the old block's rows; the copy is
    reported as ``(src, dst)`` in the third element (None when no copy).
    """
    pos = seq.seq_len
    logical, in_block = pos // block_size, pos % block_size
    cow = None
    if logical >= len(seq.block_table):
        seq.block_table.extend(pool.allocate(1))
    else:
        b = seq.block_table[logical]
        if pool.ref_cnt[b] > 1:
            (nb,) = pool.allocate(1)
            pool.free([b])
            seq.block_table[logical] = nb
            cow = (b, nb)
    seq.seq_len += 1
    return logical, in_block, cow


def slot_of(block_table, pos: int, block_size: int) -> int:
    """The scheduler's slot number of position ``pos``: physical block * block_size + offset."""
    return int(block_table[pos // block_size]) * block_size + pos % block_size


def pad_tables(tables, width: int | None = None, fill: int = -1) -> np.ndarray:
    width = max((len(t) for t in tables), default=0) if width is None else width
    out = np.full((len(tables), max(width, 1)), fill, dtype=np.int32)
    for i, t in enumerate(tables):
        out[i, : len(t)] = t
    return out


_NORMAL_FP16 = None


def normal_fp16_table() -> np.ndarray:
    """fp16 standard-normal quantiles at (u + 0.5) / 65536, u = 0..65535."""
    global _NORMAL_FP16
    if _NORMAL_FP16 is None:
        inv = NormalDist().inv_cdf
        _NORMAL_FP16 = np.array([inv((u + 0.5) / 65536.0) for u in range(65536)],
                                dtype=np.float64).astype(np.float16)
    return _NORMAL_FP16


def fp16_normal(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0, 1) fp16 values of the given shape (inverse transform, see the module doc)."""
    n = int(np.prod(shape))
    u = np.frombuffer(rng.bytes(2 * n), dtype="<u2")
    return normal_fp16_table()[u].reshape(shape)


# --------------------------------------------------------------------------
# Decode workloads (configs 1-4 of the hot-path scope)


@dataclass
class DecodeWorkload:
    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    seq_lens: np.ndarray  # int32 [S] (lengths after the new token, if any)
    block_tables: np.ndarray  # int32 [S, MB], -1 past each table's end
    q: np.ndarray  # fp16 [S, H, D]
    k_cache: np.ndarray  # fp16 [NB, bs, Hk, D] (state before the write)
    v_cache: np.ndarray
    k_new: np.ndarray | None  # fp16 [T, Hk*D] rows to write, or None
    v_new: np.ndarray | None
    slot_mapping: np.ndarray | None  # int64 [T]
    ref_cnt: np.ndarray | None = None
    cow_pairs: np.ndarray | None = None  # int64 [n, 2] (shared block, private copy)
    shared_prefix_tokens: int = 0

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.seq_lens.size else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def kv_bytes(self) -> int:
        """Key+value bytes one decode call must read: sum_i L_i * Hk * D * 2 B * 2."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * self.head_dim * 4


def _fill_rows(rng, cache_rows: np.ndarray, slots: np.ndarray, row_elems: int,
               chunk: int = 1 << 15) -> None:
    """Write fresh N(0,1) fp16 rows at ``slots`` of a [NB*bs, row] view, in slot-list order."""
    for s in range(0, slots.size, chunk):
        part = slots[s:s + chunk]
        cache_rows[part] = fp16_normal(rng, (part.size, row_elems))


def _decode_workload(name, rng, seq_lens, *, H, Hk, D, bs, NB, write_last=True,
                     shared_prefix_tokens=0, order=None, mb_width=None) -> DecodeWorkload:
    S = len(seq_lens)
    pool = BlockPool(NB, rng=None if order is not None else rng, order=order)
    seqs = [Sequence() for _ in range(S)]
    prefix_blocks: list[int] = []
    if shared_prefix_tokens:
        # one prefill of the common prompt, mapped by every sequence (ref_cnt = S)
        prefix_blocks = pool.allocate(blocks_needed(shared_prefix_tokens, bs))
        for _ in range(S - 1):
            pool.share(prefix_blocks)
    cows = []
    for seq, L in zip(seqs, seq_lens):
        L = int(L)
        before = L - 1 if write_last else L
        if shared_prefix_tokens:
            seq.block_table = list(prefix_blocks)
            seq.seq_len = shared_prefix_tokens
            while seq.seq_len < before:
                *_, cow = append_slot(pool, seq, bs)
                if cow:
                    cows.append(cow)
        else:
            prefill(pool, seq, max(before, 0), bs)
        if write_last and L > 0:
            *_, cow = append_slot(pool, seq, bs)
            if cow:
                cows.append(cow)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    tables = pad_tables([s.block_table for s in seqs], mb_width)

    q = fp16_normal(rng, (S, H, D))
    row = Hk * D
    k_cache = np.full((NB, bs, Hk, D), FP16_NAN_BITS, dtype=np.uint16).view(np.float16)
    v_cache = np.full((NB, bs, Hk, D), FP16_NAN_BITS, dtype=np.uint16).view(np.float16)
    kr = k_cache.reshape(NB * bs, row)
    vr = v_cache.reshape(NB * bs, row)
    # prior tokens, as earlier steps left them: the shared prefix once; copy on
    # write (a private block starts as a copy of the shared one); then each
    # sequence's private positions, in token order
    if shared_prefix_tokens:
        pre = np.asarray([slot_of(prefix_blocks, p, bs) for p in range(shared_prefix_tokens)],
                         dtype=np.int64)
        _fill_rows(rng, kr, pre, row)
        _fill_rows(rng, vr, pre, row)
    for src, dst in cows:
        k_cache[dst] = k_cache[src]
        v_cache[dst] = v_cache[src]
    slots = []
    for seq, L in zip(seqs, seq_lens):
        start = shared_prefix_tokens
        stop = int(L) - 1 if write_last else int(L)
        slots.extend(slot_of(seq.block_table, p, bs) for p in range(start, max(stop, start)))
    slots = np.asarray(slots, dtype=np.int64)
    _fill_rows(rng, kr, slots, row)
    _fill_rows(rng, vr, slots, row)

    k_new = v_new = slot_mapping = None
    if write_last:
        live = [i for i in range(S) if seq_lens[i] > 0]
        slot_mapping = np.asarray(
            [slot_of(seqs[i].block_table, int(seq_lens[i]) - 1, bs) for i in live], dtype=np.int64)
        k_new = fp16_normal(rng, (len(live), row))
        v_new = fp16_normal(rng, (len(live), row))
    return DecodeWorkload(name, H, Hk, D, bs, NB, 1.0 / math.sqrt(D), seq_lens, tables, q,
                          k_cache, v_cache, k_new, v_new, slot_mapping, pool.ref_cnt.copy(),
                          np.asarray(cows, dtype=np.int64).reshape(-1, 2), shared_prefix_tokens)


def config1_tiny() -> DecodeWorkload:
    """4 sequences of lengths {1,17,33,50}, bs 16, 32 blocks handed out by a seeded
    permutation, H = Hk = 4, D = 64; the last token of each sequence is written first."""
    rng = rng_for(1)
    order = rng.permutation(32)
    return _decode_workload("tiny", rng, [1, 17, 33, 50], H=4, Hk=4, D=64, bs=16, NB=32,
                            order=order[::-1])


def config2_llama8b(num_seqs: int = 64, num_kv_heads: int = 8) -> DecodeWorkload:
    """Llama-3-8B-shaped decode layer: 64 sequences, lengths U[256, 4096], bs 16,
    H 32 / Hk 8, D 128, 16384 blocks from a seeded shuffled free list, one new
    token per sequence written.  ``num_kv_heads`` widens the layer with the
    same group size (H = 4 * Hk) and the same lengths and block tables."""
    rng = rng_for(2)
    lens = rng.integers(256, 4096, size=num_seqs, endpoint=True)
    return _decode_workload("llama8b", rng, lens, H=4 * num_kv_heads, Hk=num_kv_heads, D=128,
                            bs=16, NB=16384, order=rng.permutation(16384))


def config3_long(num_seqs: int = 8, seq_len: int = 32768) -> DecodeWorkload:
    """Long context: 8 sequences of 32768 tokens (2048 blocks each), H 32 / Hk 8,
    D 128, blocks scattered by a seeded shuffle; decode only (no write)."""
    rng = rng_for(3)
    return _decode_workload("long", rng, [seq_len] * num_seqs, H=32, Hk=8, D=128, bs=16,
                            NB=16384, write_last=False, order=rng.permutation(16384))


def config4_shared_prefix(num_seqs: int = 256) -> DecodeWorkload:
    """Parallel sampling: 256 sequences share a 2000-token prefix (125 full blocks,
    ref_cnt 256), each with a private tail of U[1, 300] tokens, H 64 / Hk 8, D 128,
    16384 blocks; the last token of each sequence is written."""
    rng = rng_for(4)
    tails = rng.integers(1, 300, size=num_seqs, endpoint=True)
    return _decode_workload("shared_prefix", rng, 2000 + tails, H=64, Hk=8, D=128, bs=16,
                            NB=16384, shared_prefix_tokens=2000, order=rng.permutation(16384))


def small_decode(index: int, seq_lens, *, H, Hk, D, bs=16, NB=None, write_last=True,
                 shared_prefix_tokens=0) -> DecodeWorkload:
    """A small decode case for parity tests (seeded by ``index``)."""
    need = sum(blocks_needed(int(L), bs) for L in seq_lens) + 8
    NB = NB or max(need, 4)
    rng = rng_for(index)
    return _decode_workload(f"small{index}", rng, list(seq_lens), H=H, Hk=Hk, D=D, bs=bs,
                            NB=NB, write_last=write_last,
                            shared_prefix_tokens=shared_prefix_tokens,
                            order=rng.permutation(NB))


# --------------------------------------------------------------------------
# Chunk workloads: several new tokens per sequence (chunked prefill, draft
# verification).  The new tokens' rows are written (slot_mapping) before the
# attention, as in config 1; sequence i's query rows are
# query_start[i] .. query_start[i+1]-1, new token j at position L_i - Q_i + j.


@dataclass
class ChunkWorkload:
    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    seq_lens: np.ndarray  # int32 [S], new tokens included
    query_start: np.ndarray  # int32 [S+1]
    block_tables: np.ndarray  # int32 [S, MB]
    q: np.ndarray  # fp16 [Tq, H, D]
    k_cache: np.ndarray  # fp16 [NB, bs, Hk, D] (state before the write)
    v_cache: np.ndarray
    k_new: np.ndarray  # fp16 [Tq, Hk*D] rows of the new tokens
    v_new: np.ndarray
    slot_mapping: np.ndarray  # int64 [Tq]

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_query_tokens(self) -> int:
        return int(self.query_start[-1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.seq_lens.size else 0

    @property
    def max_query_len(self) -> int:
        return int(np.diff(self.query_start).max()) if self.seq_lens.size else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def kv_bytes(self) -> int:
        """K+V bytes of every sequence's cache: sum_i L_i * Hk * D * 2 B * 2."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * self.head_dim * 4

    def flops(self) -> int:
        """2 * (QK + PV) multiply-adds of the causal attention: each new token at
        position p attends p + 1 keys, for all H heads: sum 4 * (p+1) * D * H."""
        total = 0
        for i in range(self.num_seqs):
            L = int(self.seq_lens[i])
            nq = int(self.query_start[i + 1] - self.query_start[i])
            # positions L-nq .. L-1 attend L-nq+1 .. L keys
            total += (nq * (2 * L - nq + 1)) // 2
        return 4 * total * self.head_dim * self.num_heads


def chunk_workload(index: int, seq_lens, query_lens, *, H, Hk, D, bs=16, NB=None,
                   order=None) -> ChunkWorkload:
    """Sequences of total lengths ``seq_lens`` whose last ``query_lens`` tokens
    are new this step (seeded by ``index``)."""
    rng = rng_for(index)
    S = len(seq_lens)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    query_lens = np.asarray(query_lens, dtype=np.int32)
    assert query_lens.shape == seq_lens.shape and (query_lens <= seq_lens).all()
    need = sum(blocks_needed(int(L), bs) for L in seq_lens) + 8
    NB = NB or max(need, 4)
    pool = BlockPool(NB, rng=None if order is not None else rng,
                     order=order if order is not None else rng.permutation(NB))
    seqs = [Sequence() for _ in range(S)]
    for seq, L, nq in zip(seqs, seq_lens, query_lens):
        prefill(pool, seq, int(L - nq), bs)
        for _ in range(int(nq)):
            append_slot(pool, seq, bs)
    tables = pad_tables([s.block_table for s in seqs])
    query_start = np.zeros(S + 1, dtype=np.int32)
    query_start[1:] = np.cumsum(query_lens)
    Tq = int(query_start[-1])
    row = Hk * D
    k_cache = np.full((NB, bs, Hk, D), FP16_NAN_BITS, dtype=np.uint16).view(np.float16)
    v_cache = np.full((NB, bs, Hk, D), FP16_NAN_BITS, dtype=np.uint16).view(np.float16)
    kr = k_cache.reshape(NB * bs, row)
    vr = v_cache.reshape(NB * bs, row)
    prior = np.asarray([slot_of(seq.block_table, p, bs) for seq, L, nq in
                        zip(seqs, seq_lens, query_lens) for p in range(int(L - nq))],
                       dtype=np.int64)
    _fill_rows(rng, kr, prior, row)
    _fill_rows(rng, vr, prior, row)
    slot_mapping = np.asarray([slot_of(seq.block_table, p, bs) for seq, L, nq in
                               zip(seqs, seq_lens, query_lens) for p in range(int(L - nq), int(L))],
                              dtype=np.int64)
    q = fp16_normal(rng, (Tq, H, D))
    k_new = fp16_normal(rng, (Tq, row))
    v_new = fp16_normal(rng, (Tq, row))
    return ChunkWorkload(f"chunk{index}", H, Hk, D, bs, NB, 1.0 / math.sqrt(D), seq_lens,
                         query_start, tables, q, k_cache, v_cache, k_new, v_new, slot_mapping)


def config6_chunked_prefill(num_decodes: int = 63) -> ChunkWorkload:
    """One engine step of "vLLM 技术内幕" §3.2's example under a 2048-token
    budget: the second chunk of a 3000-token prompt (positions 2048..2999, 952
    new tokens) beside ``num_decodes`` running decode requests (one new token
    each, lengths U[256, 4096] as in config 2); H 32 / Hk 8, D 128, bs 16,
    16384 shuffled blocks."""
    rng = rng_for(6)
    L_dec = rng.integers(256, 4097, size=num_decodes)
    seq_lens = [3000] + [int(x) for x in L_dec]
    query_lens = [952] + [1] * num_decodes
    return chunk_workload(6, seq_lens, query_lens, H=32, Hk=8, D=128, bs=16, NB=16384,
                          order=rng.permutation(16384))


def config7_draft_verify(num_seqs: int = 64, num_query: int = 4) -> ChunkWorkload:
    """Speculative-decode verification ("vLLM 技术内幕" §7.4): every sequence
    checks ``num_query`` new tokens at once; lengths U[256, 4096] as in config
    2, H 32 / Hk 8, D 128, bs 16, 16384 shuffled blocks."""
    rng = rng_for(7)
    seq_lens = [int(x) for x in rng.integers(256, 4097, size=num_seqs)]
    return chunk_workload(7, seq_lens, [num_query] * num_seqs, H=32, Hk=8, D=128, bs=16,
                          NB=16384, order=rng.permutation(16384))


# --------------------------------------------------------------------------
# Byte-strided two-cache write workload (config 5)


@dataclass
class View:
    offset: int
    layer_stride: int
    block_stride: int
    row_width: int


def block_outer_views(pages: dict[str, int], num_layers: int, block_size: int) -> dict[str, View]:
    """Views for block-outer layouts (BLHNC): each block packs every cache's
    layers, in dict order; layer_stride = page, block_stride = whole block."""
    page = {c: block_size * r for c, r in pages.items()}
    block_bytes = sum(num_layers * p for p in page.values())
    out, off = {}, 0
    for c, r in pages.items():
        out[c] = View(off, page[c], block_bytes, r)
        off += num_layers * page[c]
    return out


def layer_outer_views(pages: dict[str, int], num_layers: int, block_size: int,
                      num_blocks: int) -> dict[str, View]:
    """Views for layer-outer layouts (LBNHC): each (cache, layer) is one run of
    all blocks; block_stride = page, layer_stride = page * num_blocks."""
    out, off = {}, 0
    for c, r in pages.items():
        page = block_size * r
        out[c] = View(off, page * num_blocks, page, r)
        off += num_layers * page * num_blocks
    return out


DSA_PAGES = {"mla": 656, "idx": 132}  # bytes per token: 512+16+128 and 128+4


@dataclass
class WriteWorkload:
    name: str
    num_layers: int
    block_size: int
    num_blocks: int
    cache_bytes: int
    slot_mapping: np.ndarray  # int64 [T]
    rows: dict  # (cache, layer) -> uint8 [T, row_width]
    init: np.ndarray  # uint8 [cache_bytes], the cache's prior content
    views: dict  # layout -> {cache: View}


def config5_dsa_write(num_tokens: int = 16384, num_blocks: int = 4096) -> WriteWorkload:
    """Two caches (MLA 656 B/token, indexer 132 B/token), 2 layers, bs 64, 4096
    blocks, 16384 tokens of random bytes written to seeded slots drawn without
    replacement; BLHNC and LBNHC views of the same byte budget."""
    rng = rng_for(5)
    L, bs = 2, 64
    views = {"BLHNC": block_outer_views(DSA_PAGES, L, bs),
             "LBNHC": layer_outer_views(DSA_PAGES, L, bs, num_blocks)}
    cache_bytes = num_blocks * sum(L * bs * r for r in DSA_PAGES.values())
    slots = rng.choice(num_blocks * bs, size=num_tokens, replace=False).astype(np.int64)
    rows = {}
    for c, r in DSA_PAGES.items():
        for layer in range(L):
            rows[(c, layer)] = rng.integers(0, 256, size=(num_tokens, r), dtype=np.uint8)
    init = rng.integers(0, 256, size=cache_bytes, dtype=np.uint8)
    return WriteWorkload("dsa_write", L, bs, num_blocks, cache_bytes, slots, rows, init, views)


def config(index: int):
    return {1: config1_tiny, 2: config2_llama8b, 3: config3_long, 4: config4_shared_prefix,
            5: config5_dsa_write, 6: config6_chunked_prefill, 7: config7_draft_verify}[index]()
