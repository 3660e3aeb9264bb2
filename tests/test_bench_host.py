"""Host-side logic of bench.py that needs no GPU: the committed DRAM-traffic
record it attaches to the roofline, and the kernel count of a multi-token
step that it reports as gpu_launches."""

import os
import sys
from types import SimpleNamespace

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

# algorithmic bytes per decode launch of the Llama-8B decode layer (S=64,
# L~U[256,4096], Hk 8, D 128): K+V rows, q, out, block tables, lengths
ALGORITHMIC = {"config2.fp16": 545_891_164, "config2.fp8": 281_999_324}


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
