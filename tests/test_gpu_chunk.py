"""GPU parity of pkv_chunk_attention against the oracle (chunked prefill /
draft verification: each sequence's new tokens attend causally to its cache).

Every case writes the new tokens' rows with pkv_cache_write first, as a step
does, then compares the attention element by element with the float64 oracle
at the tolerance |gpu - ref| <= 2e-3 + 1e-2 |ref|."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import paged_kv_cache_131_gb300 as pkv  # noqa: E402
from paged_kv_cache_131_gb300 import workloads as W  # noqa: E402
from paged_kv_cache_131_gb300.harness import DeviceChunk  # noqa: E402
from test_oracle_chunk import written_caches  # noqa: E402

pytestmark = pytest.mark.gpu
ATOL, RTOL = 2e-3, 1e-2


@pytest.fixture(scope="module")
def pkv_lib():
    from paged_kv_cache_131_gb300 import _build
    _build.build()
    assert torch.cuda.is_available()
    pkv.pkv_get_device_error()
    return pkv


def assert_close(got, ref, what=""):
    got = got.astype(np.float64)
    bad = np.abs(got - ref) > ATOL + RTOL * np.abs(ref)
    assert np.isfinite(got).all(), f"{what}: non-finite outputs"
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} out of tolerance, max err "
                           f"{np.abs(got - ref).max():.3e}")


def run(wl, reps=1):
    dev = DeviceChunk(wl)
    out = None
    for _ in range(reps):
        dev.step()
        out = dev.out.float().cpu().numpy()
    kind, idx = pkv.pkv_get_device_error()
    assert kind == 0, f"device error {pkv.DEVICE_ERRORS.get(kind)} at {idx}"
    return dev, out


def oracle(orc, wl, rows=None):
    k, v = written_caches(wl)
    return orc.chunk_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.query_start,
                               wl.scale, rows=rows, workers=orc.default_workers())


SMALL = [
    # (index, lens, query lens, H, Hk, D)
    (301, [5, 16, 33, 40, 19], [5, 3, 1, 7, 16], 4, 2, 64),           # pure prefill, ragged
    (302, [1, 17, 50, 2], [1, 1, 1, 1], 32, 8, 128),                  # one-token chunks
    (303, [700, 1100, 40], [60, 300, 40], 32, 8, 128),                # tiles and partitions
    (304, [1300, 613], [513, 97], 8, 8, 128),                         # G = 1, many tiles
    (305, [530, 1040, 77], [17, 9, 77], 16, 2, 64),                   # G = 8
    (306, [0, 12, 0, 600], [0, 4, 0, 2], 8, 4, 128),                  # empty sequences
    (307, [2049, 513, 512], [1025, 2, 512], 8, 2, 128),               # partition edges
    (309, [2048, 4096, 4097], [200, 130, 300], 8, 2, 128),            # 4096-token edges
    (313, [9000, 300, 4500], [150, 20, 64], 8, 2, 64),               # three partitions
    (312, [300, 40, 1, 600], [100, 40, 1, 3], 16, 16, 64),           # Hk 16: 2 head groups
]


@pytest.mark.parametrize("case", SMALL, ids=[str(c[0]) for c in SMALL])
def test_small_all_elements(pkv_lib, orc, case):
    index, lens, qlens, H, Hk, D = case
    wl = W.chunk_workload(index, lens, qlens, H=H, Hk=Hk, D=D)
    _, got = run(wl)
    assert_close(got, oracle(orc, wl), what=f"case {index}")


def test_repeated_calls_are_identical(pkv_lib):
    # tickets are left at zero: the second step merges exactly as the first
    wl = W.chunk_workload(308, [1500, 900], [200, 33], H=32, Hk=8, D=128)
    dev = DeviceChunk(wl)
    dev.step()
    a = dev.out.clone()
    dev.step()
    assert torch.equal(a, dev.out)


def test_config6_chunked_prefill(pkv_lib, orc):
    """The chunked-prefill step: all 63 decodes, and every row of the
    952-token chunk that starts or ends one of the tile kernel's 128-row query
    tiles (32 tokens x G 4), plus rows spread over the chunk."""
    wl = W.config6_chunked_prefill()
    _, got = run(wl)
    G = wl.num_heads // wl.num_kv_heads
    per_tile = 128 // G
    r0, r1 = _rows_of(wl, 0)
    edges = {r for t in range(r0, r1, per_tile) for r in (t, min(t + per_tile, r1) - 1)}
    rng = np.random.default_rng(16)
    rows = sorted(edges | set(range(r1, wl.q.shape[0])) |
                  set(int(x) for x in rng.integers(r0, r1, size=24)))
    ref = oracle(orc, wl, rows=rows)
    assert_close(got[rows], ref[rows], what="config 6")
    assert np.isfinite(got).all()


def test_config7_draft_verify_all_rows(pkv_lib, orc):
    wl = W.config7_draft_verify()
    _, got = run(wl)
    assert_close(got, oracle(orc, wl), what="config 7")


def test_sm_split_extremes(pkv_lib, orc):
    # the plan kernel hands the balanced schedule most of the SMs (24 long
    # decodes beside a 3-token chunk: as many as HBM rewards, ~2/3) or the
    # fewest it gives (a 1500-token prompt beside one short decode: 2); every
    # row is still computed, once
    rng = np.random.default_rng(318)
    many = [int(x) for x in rng.integers(2500, 4097, size=24)]
    wl = W.chunk_workload(318, [50] + many, [3] + [1] * 24, H=32, Hk=8, D=128)
    _, got = run(wl)
    assert_close(got, oracle(orc, wl), what="decode-heavy split")

    wl = W.chunk_workload(319, [1500, 20], [1500, 1], H=32, Hk=8, D=128)
    _, got = run(wl)
    rows = sorted({0, 1, 31, 32, 767, 768, 1499, 1500} |
                  set(int(x) for x in np.random.default_rng(319).integers(0, 1500, size=24)))
    ref = oracle(orc, wl, rows=rows)
    assert_close(got[rows], ref[rows], what="tile-heavy split")
    assert np.isfinite(got).all()


def _rows_of(wl, i):
    return int(wl.query_start[i]), int(wl.query_start[i + 1])


def test_bad_block_id_is_skipped_and_recorded(pkv_lib, orc):
    # sequence 0: a 300-token chunk (tcgen05 tile kernel: the bad block is
    # staged as zeros and its keys masked), sequence 1: 2 new tokens x G 4 =
    # 8 rows (balanced decode schedule: the bad block is skipped), sequence 2
    # untouched.  The error is recorded; the other sequence is exact and no
    # output is NaN.
    wl = W.chunk_workload(310, [700, 200, 500], [300, 2, 40], H=16, Hk=4, D=128)
    ref = oracle(orc, wl)
    dev = DeviceChunk(wl)
    dev.write()
    dev.block_tables[0, 2] = wl.num_blocks + 7
    dev.block_tables[1, 1] = -5
    dev.attend()
    got = dev.out.float().cpu().numpy()
    kind, _ = pkv.pkv_get_device_error()
    assert pkv.DEVICE_ERRORS.get(kind) == "block_id"
    r0, r1 = _rows_of(wl, 2)
    assert_close(got[r0:r1], ref[r0:r1], what="sequence without bad blocks")
    assert np.isfinite(got[:r0]).all()


def test_bad_sequence_length_is_skipped_and_recorded(pkv_lib, orc):
    # a length past the block table's capacity: that sequence's rows are not
    # written, the error is recorded, the others are exact
    wl = W.chunk_workload(311, [900, 300, 60], [200, 40, 60], H=8, Hk=2, D=64)
    ref = oracle(orc, wl)
    dev = DeviceChunk(wl)
    dev.write()
    dev.seq_lens[1] = wl.block_tables.shape[1] * wl.block_size + 16
    dev.out.fill_(7.0)
    dev.attend()
    got = dev.out.float().cpu().numpy()
    kind, _ = pkv.pkv_get_device_error()
    assert pkv.DEVICE_ERRORS.get(kind) == "seq_len"
    r0, r1 = _rows_of(wl, 1)
    assert (got[r0:r1] == 7.0).all()
    keep = np.r_[0:r0, r1:got.shape[0]]
    assert_close(got[keep], ref[keep], what="valid sequences")
