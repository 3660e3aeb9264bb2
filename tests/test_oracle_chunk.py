"""Pins of the oracle's chunk attention (CPU only): several new tokens per
sequence, each attending causally to its cache ("vLLM 技术内幕" §3.2 chunked
prefill, §7.4 draft verification).

The pins tie it to the decode oracle (itself pinned by closed forms and an
independent brute force in test_oracle_pins.py) -- a one-token chunk is a
decode, and new token j of a sequence is a decode of that sequence cut at
j's position -- and to an independent causal brute force on tiny inputs.
"""

import math

import numpy as np

from paged_kv_cache_131_gb300 import workloads as W


def written_caches(wl: W.ChunkWorkload):
    """The caches after this step's write of the new tokens' rows."""
    NB, bs, Hk, D = wl.k_cache.shape
    k = wl.k_cache.copy()
    v = wl.v_cache.copy()
    k.reshape(NB * bs, Hk * D)[wl.slot_mapping] = wl.k_new
    v.reshape(NB * bs, Hk * D)[wl.slot_mapping] = wl.v_new
    return k, v


def run(orc, wl, rows=None, lib=None):
    k, v = written_caches(wl)
    return orc.chunk_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.query_start,
                               wl.scale, rows=rows, lib=lib)


def test_one_token_chunks_are_decodes(orc, lib=None):
    wl = W.chunk_workload(201, [1, 17, 33, 50, 2], [1, 1, 1, 1, 1], H=4, Hk=2, D=16)
    k, v = written_caches(wl)
    got = run(orc, wl, lib=lib)
    ref = orc.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale)
    assert np.array_equal(got, ref)


def test_each_new_token_is_a_decode_of_its_prefix(orc, lib=None):
    wl = W.chunk_workload(202, [5, 16, 33, 40, 19], [5, 3, 1, 7, 16], H=4, Hk=2, D=16)
    k, v = written_caches(wl)
    got = run(orc, wl, lib=lib)
    for i in range(wl.num_seqs):
        L = int(wl.seq_lens[i])
        r0, r1 = int(wl.query_start[i]), int(wl.query_start[i + 1])
        for r in range(r0, r1):
            pos = L - (r1 - r0) + (r - r0)
            ref = orc.decode_attention(wl.q[r:r + 1], k, v, wl.block_tables[i:i + 1],
                                       np.array([pos + 1], np.int32), wl.scale)
            assert np.array_equal(got[r], ref[0]), (i, r)


def test_first_prompt_token_is_its_value(orc, lib=None):
    # a whole prompt as one chunk: token 0 attends only to itself
    wl = W.chunk_workload(203, [9, 21], [9, 21], H=2, Hk=1, D=8)
    got = run(orc, wl, lib=lib)
    for i in range(2):
        r = int(wl.query_start[i])
        v0 = wl.v_new[r].reshape(wl.num_kv_heads, wl.head_dim).astype(np.float64)
        for h in range(wl.num_heads):
            assert np.array_equal(got[r, h], v0[h // (wl.num_heads // wl.num_kv_heads)])


def brute_force_chunk(wl: W.ChunkWorkload, k_cache, v_cache):
    """Independent causal restatement for tiny inputs: new token j of a
    sequence with Q new tokens is at position L - Q + j and weighs keys
    0..that position with w_p = 1 / sum_k exp(s_k - s_p); elements are read in
    place from the caches' raw bytes at their byte address."""
    Tq, H, D = wl.q.shape
    Hk, bs = wl.num_kv_heads, wl.block_size
    kb = k_cache.view(np.uint8).reshape(-1)
    vb = v_cache.view(np.uint8).reshape(-1)
    row_width = Hk * D * 2

    def elem(buf, slot, kvh, d):
        a = slot * row_width + kvh * D * 2 + d * 2
        return float(buf[a:a + 2].view(np.float16)[0])

    out = np.zeros((Tq, H, D))
    for i in range(wl.num_seqs):
        L = int(wl.seq_lens[i])
        r0, r1 = int(wl.query_start[i]), int(wl.query_start[i + 1])
        for r in range(r0, r1):
            last = L - (r1 - r0) + (r - r0)
            slots = [int(wl.block_tables[i, p // bs]) * bs + p % bs for p in range(last + 1)]
            for h in range(H):
                kvh = h // (H // Hk)
                qv = [float(x) for x in wl.q[r, h]]
                s = [wl.scale * math.fsum(qv[d] * elem(kb, sl, kvh, d) for d in range(D))
                     for sl in slots]
                w = [1.0 / math.fsum(math.exp(sk - sj) for sk in s) for sj in s]
                for d in range(D):
                    out[r, h, d] = math.fsum(w[p] * elem(vb, slots[p], kvh, d)
                                             for p in range(len(slots)))
    return out


def test_chunk_matches_brute_force(orc, lib=None):
    wl = W.chunk_workload(204, [7, 18, 3], [4, 6, 3], H=4, Hk=2, D=8)
    k, v = written_caches(wl)
    got = run(orc, wl, lib=lib)
    ref = brute_force_chunk(wl, k, v)
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_rows_subset(orc, lib=None):
    wl = W.chunk_workload(205, [12, 30], [5, 9], H=4, Hk=1, D=8)
    full = run(orc, wl, lib=lib)
    rows = [0, 4, 7, 13]
    part = run(orc, wl, rows=rows, lib=lib)
    assert np.array_equal(part[rows], full[rows])
    others = [r for r in range(wl.num_query_tokens) if r not in rows]
    assert np.isnan(part[others]).all()


def test_config6_and_7_shapes():
    # the workload generators: budgets and positions as the pages' example
    wl = W.chunk_workload(206, [3000, 300], [952, 1], H=2, Hk=1, D=8, NB=400)
    assert wl.num_query_tokens == 953 and wl.max_query_len == 952
    # the new tokens' slots are the sequence's last positions
    bs = wl.block_size
    first = int(wl.slot_mapping[0])
    assert first == int(wl.block_tables[0, 2048 // bs]) * bs + 2048 % bs
