"""Host-side logic of bench.py that needs no GPU: the committed DRAM-traffic
record it attaches to the roofline, and the kernel count of a multi-token
step that it reports as gpu_launches."""

import os
import sys
from types import SimpleNamespace

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

# algorithmic bytes per decode launch of the Llama-8B decode layer (S=64,
# L~U[256,4096], Hk 8, D 128): K+V rows, q, out, block tables, lengths
ALGORITHMIC = {"config2.fp16": 545_891_164, "config2.fp8": 281_999_324,
               # draft verification (64 x 4 new tokens, query-column mode)
               "config7.fp16": 614_122_464}


@pytest.mark.parametrize("key", sorted(ALGORITHMIC))
def test_traffic_record_is_at_least_the_algorithmic_bytes(key):
    got = bench.recorded_traffic(key)
    if got is None:
        pytest.skip("traffic record taken on other decode sources (re-capture with ncu)")
    # DRAM carries every algorithmic byte once, plus a little (partials,
    # sector granularity); far more would mean re-reads
    assert ALGORITHMIC[key] <= got <= 1.05 * ALGORITHMIC[key]


def test_traffic_record_ignored_for_other_sources(monkeypatch):
    monkeypatch.setattr(bench, "decode_source_hash", lambda: "0" * 16)
    assert bench.recorded_traffic("config2.fp16") is None


def test_traffic_record_unknown_workload():
    assert bench.recorded_traffic("no-such-workload") is None


@pytest.mark.parametrize("H,Hk,max_q,launches", [
    (32, 8, 952, 4),  # chunked prefill beside decodes: write, balanced, plan, tile
    (32, 8, 4, 2),    # draft verification, 16 rows per KV head: write, balanced
    (32, 8, 2, 2),    # 8 rows: one column tile of the balanced schedule
    (32, 8, 5, 4),    # 20 rows: past both column tiles, so the tile kernel too
    (8, 8, 8, 2),     # G = 1: 8 rows
    (64, 8, 2, 2),    # G = 8: 16 rows in two column tiles
])
def test_chunk_launches_per_step_follow_the_routing(H, Hk, max_q, launches):
    wl = SimpleNamespace(num_heads=H, num_kv_heads=Hk, max_query_len=max_q)
    assert bench.chunk_launches_per_step(wl) == launches


def test_passes_needed_reaches_the_timed_budget():
    # 20 steps of 0.1 ms = 2 ms per pass: 500 passes make a second
    assert bench.passes_needed(2.0, 1.0) == 500
    assert bench.passes_needed(2000.0, 1.0) == 1      # one long pass is enough
    assert bench.passes_needed(0.001, 1.0) == bench.MAX_PASSES
    assert bench.passes_needed(0.0, 1.0) == bench.MAX_PASSES


def test_spread_is_median_and_deciles():
    s = bench.spread(list(range(1, 102)))  # 1..101
    assert s["median"] == 51 and s["p10"] == 11 and s["p90"] == 91


def test_write_traffic_record_gated_by_write_source(monkeypatch):
    monkeypatch.setattr(bench, "write_source_hash", lambda: "0" * 16)
    assert bench.recorded_write_traffic("config5.BLHNC.one_launch") is None


def test_default_run_is_short_and_times_every_workload():
    args = bench.parse([])
    assert (args.gpus, args.steps, args.warmup, args.config) == (1, 20, 5, 2)
    keys = args.extras.split(",")
    assert {"3", "4", "5", "2.fp8", "3.fp8", "6", "6.chunk", "7"} == set(keys)


def test_config5_write_bytes_count_the_slot_mapping_once():
    pytest.importorskip("torch")
    from paged_kv_cache_131_gb300 import workloads as W
    from paged_kv_cache_131_gb300.harness import DeviceWrite
    dev = DeviceWrite(W.config5_dsa_write(), device="cpu")
    # rows read + rows written for 2 caches x 2 layers, plus 8 bytes per slot
    for layout in ("BLHNC", "LBNHC"):
        assert dev.layout_bytes(layout) == 2 * 16384 * (656 + 132) * 2 + 8 * 16384
    # the packed per-step inputs hold every row set and the slot mapping
    for key, rows in dev.wl.rows.items():
        assert np.array_equal(dev.rows[key].numpy(), rows)
    assert np.array_equal(dev.slot_mapping.numpy(), dev.wl.slot_mapping)


def test_unique_kv_bytes_of_the_shared_prefix_workload():
    from paged_kv_cache_131_gb300 import workloads as W
    wl = W.small_decode(40, [40, 50, 35], H=8, Hk=2, D=64, shared_prefix_tokens=32)
    # the 2 shared blocks once, then each private tail (40-32, 50-32, 35-32 rows
    # in the third block of each sequence, the last of which holds the new token)
    rows = 32 + (40 - 32) + (50 - 32 - 16) + 16 + (35 - 32)
    assert bench.unique_kv_bytes(wl) == rows * 2 * 64 * 4


def test_chunk_traffic_record_gated_by_chunk_source(monkeypatch):
    monkeypatch.setattr(bench, "chunk_source_hash", lambda: "0" * 16)
    assert bench.recorded_chunk_traffic("config6.chunk") is None


def test_chunk_traffic_record_reads_the_inputs_once():
    got = bench.recorded_chunk_traffic("config6.chunk")
    if got is None:
        pytest.skip("traffic record taken on other tile-kernel sources (re-capture with ncu)")
    # the 3000-token prompt's keys and values (bs 16, Hk 8, D 128, fp16) and
    # the 952 chunk tokens' query rows (H 32): each read once from DRAM; the
    # output may stay in L2
    kv = 2 * 3000 * 8 * 128 * 2
    q = 952 * 32 * 128 * 2
    assert kv + q <= got <= 1.1 * (kv + q)
