#!/usr/bin/env python3
"""Benchmark of the paged KV-cache hot path on GB300.

One step = one pass of the whole hot path over one batch: the cache write of
each sequence's new K/V token (pkv_cache_write), then paged decode attention
over every sequence (pkv_decode_attention: block-table walk, online softmax,
split-KV with the in-kernel log-sum-exp combine).

Default workload: the Llama-3-8B-shaped decode layer -- 64 sequences, lengths
uniform in [256, 4096], block_size 16, 32 query / 8 KV heads, head_dim 128,
fp16 KV cache [16384, 16, 8, 128] from a seeded shuffled free list, one new
token per sequence.  Synthetic seeded data; the KV cache is resident state.

Prints one JSON line.  `value` is KV-read GB/s of the whole step (key+value
bytes the decode must read / step time, inputs resident in HBM, L2 flushed
between timed steps).  The K-step timed pass is repeated until about a second
of timed device work has accumulated (`passes`); `value` and `ms_per_step`
are the median over passes, `spread` gives the 10th / 90th percentiles.
`e2e` is the same metric through the public API with the step's inputs
copied from pinned host memory and the output copied back inside the timed
region.  `roofline` is the decode kernel's algorithmic bytes per launch / its
event-timed duration against the measured HBM copy bandwidth.
`cpu_baseline` times the float64 oracle on the host.

With the default workload (N=1) the line also carries `configs`: the other
workloads of the hot path, each event-timed the same way (L2 flushed before
every step) with its own roofline and clock record -- long-context decode,
shared-prefix decode (logical bytes, DRAM bytes and L2 hit rate), the
two-cache byte-strided write in both layouts (one launch and one launch per
(cache, layer) view), FP8 decode of the first two, the multi-token steps
(chunked prefill, draft verification), and the chunked-prefill chunk alone
(`6.chunk`: the tcgen05 tile kernel on every SM, tensor-bound).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config 2|3|4|5|6|7] [--compute auto|simt|mma] [--kv fp16|fp8]
                  [--extras LIST|none]

Config 5 times the two-cache write alone (MLA 656-byte and indexer 132-byte
rows, 2 layers, block-outer and layer-outer views).  Configs 6 and 7 time the
multi-token step instead: the write of every new token's row, then the causal
attention of each sequence's new tokens (pkv_chunk_attention) -- 6 is one
engine step of chunked prefill (a 952-token prompt chunk beside 63 decodes),
7 is 4-token draft verification on 64 sequences.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode KV-read GB/s (% of HBM peak), seqs/s; cache-write GB/s"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0

# the headline's K-step pass is repeated until this much timed device work
# has accumulated; each `configs` entry gets EXTRA_TIMED_S per timed pass kind
HEADLINE_TIMED_S = 1.0
EXTRA_TIMED_S = 0.3
MAX_PASSES = 4000
EXTRAS_DEFAULT = "3,4,5,2.fp8,3.fp8,6,6.chunk,7"

CHUNK_ONLY_NAME = ("chunked-prefill chunk alone: the 952-token chunk of config 6 (positions "
                   "2048..2999 of a 3000-token prompt) without the decodes, bs=16, H=32, Hk=8, "
                   "D=128, new rows written first")
WORKLOAD_NAMES = {
    2: "llama3-8b decode layer: S=64, L~U[256,4096], bs=16, H=32, Hk=8, D=128, "
       "fp16 cache [16384,16,8,128], 1 new token/seq written",
    3: "long context: S=8, L=32768, bs=16, H=32, Hk=8, D=128, 16384 shuffled blocks, decode only",
    4: "shared prefix: S=256, 2000-token shared prefix + tail U[1,300], bs=16, H=64, Hk=8, "
       "D=128, 16384 blocks, 1 new token/seq written",
    5: "two-cache DSA write: 2 layers, bs=64, 4096 blocks, 16384 tokens of random bytes at "
       "seeded slots (no repeats), MLA 656 B + indexer 132 B rows, block-outer (BLHNC) and "
       "layer-outer (LBNHC) views",
    6: "chunked-prefill step: 952-token chunk of a 3000-token prompt (positions 2048..2999) + "
       "63 decodes L~U[256,4096], bs=16, H=32, Hk=8, D=128, 16384 shuffled blocks, new rows "
       "written first",
    7: "draft verification: S=64, 4 new tokens each, L~U[256,4096], bs=16, H=32, Hk=8, D=128, "
       "16384 shuffled blocks, new rows written first",
}

L2_NOTE = ("flushed between timed steps (write a 2x L2 buffer, then read another 2x L2 buffer: "
           "cold, clean L2)")

CSRC = os.path.join(ROOT, "paged_kv_cache_131_gb300", "csrc")
DECODE_SOURCES = [os.path.join(CSRC, f)
                  for f in ("pkv_decode_balanced.cu", "pkv_decode_common.cuh", "pkv_device.cuh",
                            "pkv_tensor_map.cu")]
WRITE_SOURCES = [os.path.join(CSRC, "pkv_write.cu")]
CHUNK_SOURCES = [os.path.join(CSRC, f)
                 for f in ("pkv_chunk.cu", "pkv_tcgen05.cuh", "pkv_device.cuh",
                           "pkv_decode_common.cuh", "pkv_decode_host.h", "pkv_tensor_map.cu")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_kernel_dram_traffic.txt")
WRITE_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "cache_write_kernel_dram_traffic.txt")
CHUNK_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "chunk_attention_kernel_dram_traffic.txt")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, choices=[2, 3, 4, 5, 6, 7])
    ap.add_argument("--compute", choices=["auto", "simt", "mma"], default="auto")
    ap.add_argument("--schedule", choices=["auto", "grid", "balanced"], default="auto")
    ap.add_argument("--kv", choices=["fp16", "fp8"], default="fp16",
                    help="KV cache format (fp8: E4M3 codes + per-row fp32 scales)")
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--kv-heads", type=int, default=8,
                    help="config 2 only: KV heads of the layer (query heads = 4x), same lengths")
    ap.add_argument("--chunk-only", action="store_true",
                    help="config 6 only: the chunk without the decodes (the tile kernel alone)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--timed-s", type=float, default=HEADLINE_TIMED_S,
                    help="repeat the K-step timed pass until this much timed device work")
    ap.add_argument("--extras", default=EXTRAS_DEFAULT,
                    help="comma list of other workloads timed into `configs` with the default "
                         "workload (3, 4, 5, 2.fp8, 3.fp8, 6, 6.chunk, 7), or 'none'")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_bf16_tflops() -> float:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f).get("bf16_tflops", 1900.0))
    return 1900.0


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def host_cpu_info() -> dict:
    """The host's CPU count and the size of this process's affinity set (the
    oracle runs single-threaded on one of them)."""
    try:
        aff = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        aff = None
    return {"host_cpus": os.cpu_count(), "affinity_cpus": aff}


# --------------------------------------------------------------------------- ncu records


def source_hash(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def decode_source_hash() -> str:
    return source_hash(DECODE_SOURCES)


def write_source_hash() -> str:
    return source_hash(WRITE_SOURCES)


def chunk_source_hash() -> str:
    return source_hash(CHUNK_SOURCES)


def _read_record(path: str, current_hash: str) -> dict:
    """key = value lines of a committed ncu summary, or {} when the file is
    missing or was taken on other kernel sources than the current ones."""
    if not os.path.exists(path):
        return {}
    rec = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                rec[k.strip()] = v.strip()
    return rec if rec.get("source_hash") == current_hash else {}


def recorded_traffic(workload_key: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode kernel source (else None)."""
    v = _read_record(TRAFFIC_FILE, decode_source_hash()).get(
        f"traffic_bytes_per_launch.{workload_key}")
    return float(v) if v else None


def recorded_decode_value(key: str):
    """Another figure of the decode ncu record (e.g. an L2 hit rate), same gate."""
    v = _read_record(TRAFFIC_FILE, decode_source_hash()).get(key)
    return float(v) if v else None


def recorded_chunk_traffic(workload_key: str):
    """DRAM bytes per tile-kernel launch from its committed ncu summary, if it
    was taken on the current tile kernel source (else None)."""
    v = _read_record(CHUNK_TRAFFIC_FILE, chunk_source_hash()).get(
        f"traffic_bytes_per_launch.{workload_key}")
    return float(v) if v else None


def recorded_write_traffic(workload_key: str):
    """DRAM bytes per cache-write launch from its committed ncu summary, if it
    was taken on the current write kernel source (else None)."""
    v = _read_record(WRITE_TRAFFIC_FILE, write_source_hash()).get(
        f"traffic_bytes_per_launch.{workload_key}")
    return float(v) if v else None


# --------------------------------------------------------------------------- timing helpers


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """Max of a per-rank float over the process group (the rank's own value
    when there is none).  NCCL reduces a CUDA tensor, gloo a CPU one."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    import torch
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank: int, world: int, step_ms_max: float) -> float:
    """Weak scaling: every rank reads its own replica's bytes each step; the
    job's step takes as long as its slowest rank."""
    return world * bytes_per_rank / (step_ms_max * 1e-3) / 1e9


def passes_needed(first_pass_ms: float, min_s: float, max_passes: int = MAX_PASSES) -> int:
    """Passes (the first included) that bring the timed device work to at
    least ``min_s`` seconds, given the first pass's total."""
    if first_pass_ms <= 0:
        return max_passes
    return int(min(max_passes, max(1, math.ceil(min_s * 1e3 / first_pass_ms))))


def spread(values) -> dict:
    """Median and 10th / 90th percentiles."""
    a = np.asarray(values, dtype=np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)),
            "p90": float(np.percentile(a, 90))}


def timed_passes(K, step, flush, stream, min_s, split=False, dist=None, device=None):
    """K-step passes, repeated until ``min_s`` seconds of timed device work.

    ``step(mid)`` enqueues one step; with ``split`` it records the event
    ``mid`` between the step's two parts (else ``mid`` is None).  L2 is
    flushed before every step, outside the events.  Returns the per-pass mean
    step times (ms) and, with ``split``, every step's two part times."""
    import torch

    means, first, second = [], [], []
    target = None
    while target is None or len(means) < target:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        for i in range(K):
            flush()
            ev[i][0].record(stream)
            step(ev[i][1] if split else None)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        ms = [e[0].elapsed_time(e[2]) for e in ev]
        means.append(sum(ms) / K)
        if split:
            first += [e[0].elapsed_time(e[1]) for e in ev]
            second += [e[1].elapsed_time(e[2]) for e in ev]
        if target is None:
            target = passes_needed(sum(ms), min_s)
            # every rank runs the same number of passes
            target = int(max_over_ranks(float(target), dist, device))
    return means, first, second


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed loop runs."""

    QUERY = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, p in zip(names, parts[2:]):
                if p.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- reference arm


def oracle_step_sample(wl, k, v, units, orc):
    """The oracle's write of every new row, then its decode of the sampled
    (sequence, kv_head) units (all G query heads of each).  Returns the KV
    bytes the sample reads."""
    row = wl.num_kv_heads * wl.head_dim * 2
    if wl.slot_mapping is not None:
        for cache, new in ((k, wl.k_new), (v, wl.v_new)):
            orc.cache_write(cache.view(np.uint8).reshape(-1), new.view(np.uint8),
                            wl.slot_mapping, offset=0, layer=0, layer_stride=0,
                            block_stride=wl.block_size * row, row_width=row,
                            block_size=wl.block_size, num_blocks=wl.num_blocks)
    G = wl.num_heads // wl.num_kv_heads
    pairs = [(i, kvh * G + g) for i, kvh in units for g in range(G)]
    orc.decode_attention(wl.q, k, v, wl.block_tables, wl.seq_lens, wl.scale, pairs=pairs)
    return sum(int(wl.seq_lens[i]) for i, _ in units) * wl.head_dim * 4


class OracleSampler:
    """Times the float64 oracle on rotating (sequence, kv_head) units."""

    def __init__(self, wl):
        import oracle as orc

        orc.build()
        self.orc, self.wl = orc, wl
        self.k, self.v = wl.k_cache.copy(), wl.v_cache.copy()
        self.units = [(i, h) for i in range(wl.num_seqs) for h in range(wl.num_kv_heads)]
        self.pos = 0

    def step(self, n_units):
        units = [self.units[(self.pos + j) % len(self.units)] for j in range(n_units)]
        self.pos += n_units
        t0 = time.perf_counter()
        nbytes = oracle_step_sample(self.wl, self.k, self.v, units, self.orc)
        return nbytes, time.perf_counter() - t0

    def calibrate(self) -> float:
        """Seconds per unit (one sequence's KV head, all its query heads)."""
        nb, t = self.step(4)
        return t / 4

    def run(self, n_units, steps=None, budget_s=None):
        total_b, total_t, n = 0, 0.0, 0
        while (steps is not None and n < steps) or (budget_s is not None and total_t < budget_s):
            b, t = self.step(n_units)
            total_b, total_t, n = total_b + b, total_t + t, n + 1
        return (total_b / total_t / 1e9 if total_t > 0 else 0.0), total_t, n


class ChunkOracleSampler:
    """Times the float64 chunk oracle on rotating query rows (all heads of a
    row); bytes = the key+value bytes each row's causal attention reads."""

    def __init__(self, wl):
        import oracle as orc

        orc.build()
        self.orc, self.wl = orc, wl
        NB, bs, Hk, D = wl.k_cache.shape
        self.k, self.v = wl.k_cache.copy(), wl.v_cache.copy()
        self.k.reshape(NB * bs, Hk * D)[wl.slot_mapping] = wl.k_new
        self.v.reshape(NB * bs, Hk * D)[wl.slot_mapping] = wl.v_new
        qs, L = wl.query_start, wl.seq_lens
        self.pos_of = {}
        for i in range(wl.num_seqs):
            for r in range(int(qs[i]), int(qs[i + 1])):
                self.pos_of[r] = int(L[i]) - int(qs[i + 1] - qs[i]) + r - int(qs[i])
        self.rows = sorted(self.pos_of)
        self.cur = 0

    def step(self, n_rows):
        rows = [self.rows[(self.cur + j) % len(self.rows)] for j in range(n_rows)]
        self.cur += n_rows
        wl = self.wl
        t0 = time.perf_counter()
        self.orc.chunk_attention(wl.q, self.k, self.v, wl.block_tables, wl.seq_lens,
                                 wl.query_start, wl.scale, rows=rows)
        t = time.perf_counter() - t0
        nbytes = sum(self.pos_of[r] + 1 for r in rows) * wl.num_kv_heads * wl.head_dim * 4
        return nbytes, t

    def calibrate(self) -> float:
        nb, t = self.step(2)
        return t / 2

    def run(self, n_rows, steps=None, budget_s=None):
        total_b, total_t, n = 0, 0.0, 0
        while (steps is not None and n < steps) or (budget_s is not None and total_t < budget_s):
            b, t = self.step(n_rows)
            total_b, total_t, n = total_b + b, total_t + t, n + 1
        return (total_b / total_t / 1e9 if total_t > 0 else 0.0), total_t, n


class WriteOracleSampler:
    """Times the oracle's two-cache write: every (cache, layer) view of one
    layout per step, alternating block-outer and layer-outer layouts; bytes =
    rows read + written + the slot mapping once."""

    def __init__(self, wl):
        import oracle as orc

        orc.build()
        self.orc, self.wl = orc, wl
        self.cache = wl.init.copy()
        self.layouts = sorted(wl.views)
        self.n = 0

    def step(self):
        wl = self.wl
        layout = self.layouts[self.n % len(self.layouts)]
        self.n += 1
        nbytes = 8 * wl.slot_mapping.size
        t0 = time.perf_counter()
        for c, v in wl.views[layout].items():
            for layer in range(wl.num_layers):
                self.orc.cache_write(self.cache, wl.rows[(c, layer)], wl.slot_mapping,
                                     offset=v.offset, layer=layer, layer_stride=v.layer_stride,
                                     block_stride=v.block_stride, row_width=v.row_width,
                                     block_size=wl.block_size, num_blocks=wl.num_blocks)
                nbytes += 2 * wl.slot_mapping.size * v.row_width
        return nbytes, time.perf_counter() - t0

    def run(self, steps=None, budget_s=None):
        total_b, total_t, n = 0, 0.0, 0
        while (steps is not None and n < steps) or (budget_s is not None and total_t < budget_s):
            b, t = self.step()
            total_b, total_t, n = total_b + b, total_t + t, n + 1
        return (total_b / total_t / 1e9 if total_t > 0 else 0.0), total_t, n


def reference_line(args, gbs, t, n, sample):
    return {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t / max(n, 1) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64" if args.config != 5 else "u8",
        "data": "synthetic",
        "config": {"workload": CHUNK_ONLY_NAME if args.chunk_only else WORKLOAD_NAMES[args.config],
                   "sample": sample},
        "cpu_baseline": {"value": round(gbs, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, **host_cpu_info()},
        "e2e": {"value": round(gbs, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_reference(args, wl, rank):
    if rank != 0:
        return
    if args.config == 5:
        sampler = WriteOracleSampler(wl)
        if args.warmup > 0:
            sampler.run(steps=args.warmup)
        gbs, t, n = sampler.run(steps=max(1, args.steps))
        sample = ("every (cache, layer) view of one layout per step, block-outer and "
                  "layer-outer alternating, all 16384 tokens; single-threaded")
        print(json.dumps(reference_line(args, gbs, t, n, sample)), flush=True)
        return
    if args.config in (6, 7):
        sampler = ChunkOracleSampler(wl)
        t_row = sampler.calibrate()
        n_rows = max(1, int(90.0 / max(1, args.steps + args.warmup) / t_row))
        if args.warmup > 0:
            sampler.run(n_rows, steps=args.warmup)
        gbs, t, n = sampler.run(n_rows, steps=max(1, args.steps))
        sample = (f"{n_rows} query rows (all heads) per step, rotating over all "
                  f"{len(sampler.rows)}; single-threaded float64")
        print(json.dumps(reference_line(args, gbs, t, n, sample)), flush=True)
        return
    sampler = OracleSampler(wl)
    t_unit = sampler.calibrate()
    per_step_budget = 90.0 / max(1, args.steps + args.warmup)
    n_units = max(1, int(per_step_budget / t_unit))
    if args.warmup > 0:
        sampler.run(n_units, steps=args.warmup)
    gbs, t, n = sampler.run(n_units, steps=max(1, args.steps))
    sample = (f"{n_units} (sequence, kv_head) units per step, rotating over all "
              f"{len(sampler.units)}, plus the write of all new rows; single-threaded float64")
    print(json.dumps(reference_line(args, gbs, t, n, sample)), flush=True)


# --------------------------------------------------------------------------- our arm


def chunk_launches_per_step(wl) -> int:
    """Kernels of one multi-token step: the write, the balanced decode
    schedule for chunks of up to 8 (or 16) query rows per KV head, and the
    plan + tcgen05 tile kernels for longer chunks (the routing of
    pkv_chunk_attention)."""
    G = wl.num_heads // wl.num_kv_heads
    rows = int(wl.max_query_len) * G
    col_tiles = 1 if (rows <= 8 or rows > 16) else 2
    return 1 + 1 + (2 if rows > 8 * col_tiles else 0)


def decode_alg_bytes(wl, kv_bytes: int) -> int:
    """Algorithmic bytes of one decode launch: the key/value bytes, q in, out,
    the block-table entries of every sequence's blocks and the lengths."""
    S, H, D = wl.num_seqs, wl.num_heads, wl.head_dim
    nblk = int(sum(-(-int(L) // wl.block_size) for L in wl.seq_lens))
    return kv_bytes + S * H * D * 2 * 2 + nblk * 4 + S * 4


def check_device_error(pkv):
    kind, idx = pkv.pkv_get_device_error()
    if kind:
        raise RuntimeError(f"device error {pkv.DEVICE_ERRORS.get(kind)} at {idx}")


def setup_device(args, local, world):
    import torch

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import paged_kv_cache_131_gb300 as pkv
    from paged_kv_cache_131_gb300 import _build

    if int(os.environ.get("RANK", "0")) == 0 or not os.path.exists(_build.LIB):
        _build.build()
    if dist is not None:
        dist.barrier()
    return pkv, dist


def measure_decode(wl, args, kv, local, flush, stream, min_s, dist=None, compute=0, schedule=0,
                   partition=0):
    """Warm up, then time the decode step (write + decode) in K-step passes:
    whole steps, then with an event between the write and the decode for each
    kernel's own time.  Returns the device staging and the measurements."""
    import torch

    import paged_kv_cache_131_gb300 as pkv
    from paged_kv_cache_131_gb300.harness import DeviceDecode, DeviceDecodeFp8

    if kv == "fp8":
        dev = DeviceDecodeFp8(wl, device=f"cuda:{local}")
    else:
        dev = DeviceDecode(wl, device=f"cuda:{local}", partition_size=partition,
                           compute=compute, schedule=schedule)

    def step(mid):
        dev.write()
        if mid is not None:
            mid.record(stream)
        dev.decode()

    for _ in range(max(args.warmup, 3)):
        flush()
        step(None)
    torch.cuda.synchronize()
    check_device_error(pkv)
    K = args.steps
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        means, _, _ = timed_passes(K, step, flush, stream, min_s, dist=dist,
                                   device=f"cuda:{local}")
        t_wall = time.perf_counter() - t_wall
        split_means, w_ms, d_ms = timed_passes(K, step, flush, stream, min_s / 2, split=True,
                                               dist=dist, device=f"cuda:{local}")
    check_device_error(pkv)
    launches = (1 if dev.has_write else 0) + 1
    return dev, {
        "step_passes": means, "write_ms": w_ms, "decode_ms": d_ms, "clocks": clocks.summary(),
        "wall_s": t_wall, "passes": len(means), "split_passes": len(split_means),
        "gpu_launches": launches * K * (len(means) + len(split_means)),
    }


def decode_entry(key, wl, dev, m, kv, peak, peak_kind):
    """One `configs` entry for a decode workload."""
    kv_bytes = dev.kv_bytes() if kv == "fp8" else wl.kv_bytes()
    alg = decode_alg_bytes(wl, kv_bytes)
    st, dk = spread(m["step_passes"]), spread(m["decode_ms"])
    achieved = alg / (dk["median"] * 1e-3) / 1e9
    entry = {
        "workload": WORKLOAD_NAMES[int(key.split(".")[0])] + (", FP8 (E4M3) cache" if kv == "fp8"
                                                               else ""),
        "kv": kv,
        "value": round(kv_bytes / (st["median"] * 1e-3) / 1e9, 2), "unit": UNIT,
        "ms_per_step": round(st["median"], 5),
        "ms_per_step_p10_p90": [round(st["p10"], 5), round(st["p90"], 5)],
        "decode_kernel_ms": round(dk["median"], 5),
        "decode_kernel_ms_p10_p90": [round(dk["p10"], 5), round(dk["p90"], 5)],
        "seqs_per_s": round(wl.num_seqs / (st["median"] * 1e-3), 1),
        "passes": m["passes"], "steps": len(m["decode_ms"]) // max(m["split_passes"], 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic(f"config{key.split('.')[0]}.{kv}"),
                     "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth)",
                     "kernel": "decode_balanced_kernel" + (" (FP8 MMA policy)" if kv == "fp8"
                                                           else " (MMA policy)"),
                     "alg_bytes_per_launch": alg},
        "gpu_launches": m["gpu_launches"],
        "clocks": m["clocks"],
    }
    if dev.has_write:
        wk = spread(m["write_ms"])
        entry["write_kernel_ms"] = round(wk["median"], 5)
    return entry


def measure_chunk(wl, args, local, flush, stream, min_s, dist=None):
    """The multi-token step (write + attention call), captured as CUDA graphs
    and replayed: whole steps, then write and call with an event between."""
    import torch

    import paged_kv_cache_131_gb300 as pkv
    from paged_kv_cache_131_gb300.harness import DeviceChunk

    dev = DeviceChunk(wl, device=f"cuda:{local}")
    for _ in range(max(args.warmup, 3)):
        flush()
        dev.step()
    torch.cuda.synchronize()
    check_device_error(pkv)
    # the step's launches (write; one or two attention kernels and the plan
    # kernel) are captured once as CUDA graphs and replayed, so no Python
    # enqueue sits inside the timed region (one graph for the whole step, so
    # the attention call may overlap the write's tail as it does on a stream;
    # two for the pass that times each)
    g_step, g_write, g_attend = (torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(),
                                 torch.cuda.CUDAGraph())
    with torch.cuda.graph(g_step):
        dev.write()
        dev.attend()
    with torch.cuda.graph(g_write):
        dev.write()
    with torch.cuda.graph(g_attend):
        dev.attend()
    torch.cuda.synchronize()

    def step(mid):
        if mid is None:
            g_step.replay()
        else:
            g_write.replay()
            mid.record(stream)
            g_attend.replay()

    K = args.steps
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        means, _, _ = timed_passes(K, step, flush, stream, min_s, dist=dist,
                                   device=f"cuda:{local}")
        split_means, w_ms, a_ms = timed_passes(K, step, flush, stream, min_s / 2, split=True,
                                               dist=dist, device=f"cuda:{local}")
    check_device_error(pkv)
    Tq, H, D = wl.q.shape
    nblk = int(sum(-(-int(L) // wl.block_size) for L in wl.seq_lens))
    # algorithmic bytes of the attention: every sequence's K and V once, q in,
    # out, block tables, lengths and query offsets
    attn_bytes = wl.kv_bytes() + Tq * H * D * 2 * 2 + nblk * 4 + wl.num_seqs * 8 + 4
    return dev, {"step_passes": means, "write_ms": w_ms, "attn_ms": a_ms,
                 "clocks": clocks.summary(), "passes": len(means),
                 "split_passes": len(split_means), "attn_bytes": attn_bytes,
                 "gpu_launches": chunk_launches_per_step(wl) * K * (len(means) +
                                                                    len(split_means))}


def chunk_roofline(wl, m, peak_hbm, peak_kind):
    peak_tf = measured_bf16_tflops()
    attn_ms = spread(m["attn_ms"])["median"]
    flops = wl.flops()
    gbs = m["attn_bytes"] / (attn_ms * 1e-3) / 1e9
    tfs = flops / (attn_ms * 1e-3) / 1e12
    hbm_frac, tf_frac = gbs / peak_hbm, tfs / peak_tf
    if hbm_frac >= tf_frac:
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                "frac": round(hbm_frac, 4), "traffic": None,
                "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth)"}
    else:
        roof = {"bound": "tensor", "achieved": round(tfs, 2), "peak": peak_tf, "unit": "TFLOP/s",
                "frac": round(tf_frac, 4), "traffic": None,
                "peak_source": "measured bf16_tflops (cuBLAS, burst); the fp16 tcgen05 MMA "
                               "runs at the bf16 rate"}
    # the attention call is one or two kernels: short chunks (and decodes) on
    # the balanced decode schedule, longer ones on the tcgen05 tile kernel
    roof.update({"kernel": "attention call (decode_balanced_kernel for short chunks, "
                           "chunk_attention_kernel on tcgen05 for the rest)",
                 "alg_bytes_per_launch": m["attn_bytes"],
                 "flops_per_launch": flops, "achieved_gbs": round(gbs, 1),
                 "achieved_tflops": round(tfs, 2), "hbm_frac": round(hbm_frac, 4),
                 "tensor_frac": round(tf_frac, 4)})
    return roof, attn_ms


def chunk_entry(key, wl, m, peak, peak_kind):
    roof, attn_ms = chunk_roofline(wl, m, peak, peak_kind)
    st, ak = spread(m["step_passes"]), spread(m["attn_ms"])
    Tq = wl.q.shape[0]
    if key.endswith(".chunk"):
        roof["kernel"] = ("attention call = chunk_plan_kernel (one CTA) + chunk_attention_kernel "
                          "(tcgen05) on every SM")
        # DRAM bytes of the dominant kernel, the tile kernel (ncu record)
        roof["traffic"] = recorded_chunk_traffic("config6.chunk")
    elif key == "7":
        # the call is the balanced schedule alone (query-column mode)
        roof["traffic"] = recorded_traffic("config7.fp16")
    return {
        "workload": CHUNK_ONLY_NAME if key.endswith(".chunk") else WORKLOAD_NAMES[int(key)],
        "value": round(wl.kv_bytes() / (st["median"] * 1e-3) / 1e9, 2), "unit": UNIT,
        "ms_per_step": round(st["median"], 5),
        "ms_per_step_p10_p90": [round(st["p10"], 5), round(st["p90"], 5)],
        "attention_call_ms": round(attn_ms, 5),
        "attention_call_ms_p10_p90": [round(ak["p10"], 5), round(ak["p90"], 5)],
        "write_kernel_ms": round(spread(m["write_ms"])["median"], 5),
        "query_tokens_per_s": round(Tq / (st["median"] * 1e-3), 1),
        "passes": m["passes"], "roofline": roof, "gpu_launches": m["gpu_launches"],
        "clocks": m["clocks"],
    }


def measure_write(wl, args, local, flush, stream, min_s, peak, peak_kind, dist=None):
    """The two-cache write of config 5: for each layout, all (cache, layer)
    views in one launch and in one launch per view.  Returns the device
    staging and the entries per layout and mode."""
    import torch

    import paged_kv_cache_131_gb300 as pkv
    from paged_kv_cache_131_gb300.harness import DeviceWrite

    dev = DeviceWrite(wl, device=f"cuda:{local}")
    out = {}
    K = args.steps
    for layout in ("BLHNC", "LBNHC"):
        out[layout] = {}
        alg = dev.layout_bytes(layout)
        for mode, fn in (("one_launch", dev.write_layout_batched),
                         ("per_view_launches", dev.write_layout)):
            nviews = len(wl.views[layout]) * wl.num_layers
            for _ in range(max(args.warmup, 3)):
                flush()
                fn(layout)
            torch.cuda.synchronize()
            check_device_error(pkv)
            if dist is not None:
                dist.barrier()
            with ClockSampler(local) as clocks:
                means, _, _ = timed_passes(K, lambda mid: fn(layout), flush, stream, min_s,
                                           dist=dist, device=f"cuda:{local}")
            check_device_error(pkv)
            sp = spread(means)
            gbs = alg / (sp["median"] * 1e-3) / 1e9
            launches = 1 if mode == "one_launch" else nviews
            out[layout][mode] = {
                "ms": round(sp["median"], 5), "ms_p10_p90": [round(sp["p10"], 5),
                                                             round(sp["p90"], 5)],
                "value": round(gbs, 2), "unit": UNIT,
                "tokens_per_s": round(wl.slot_mapping.size / (sp["median"] * 1e-3), 1),
                "launches_per_step": launches, "passes": len(means),
                "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                             "unit": "GB/s", "frac": round(gbs / peak, 4),
                             "traffic": recorded_write_traffic(f"config5.{layout}.{mode}"),
                             "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth)",
                             "kernel": "cache_write_kernel",
                             "alg_bytes_per_launch" if launches == 1 else "alg_bytes_per_step":
                                 alg},
                "gpu_launches": launches * K * len(means),
                "clocks": clocks.summary(),
            }
    return dev, out


def run_extras(args, keys, local, flush, stream, peak, peak_kind):
    """The `configs` entries: every other workload, measured one after the
    other on this GPU (each staged, timed and freed in turn)."""
    import torch

    from paged_kv_cache_131_gb300 import workloads as W

    out = {}
    for key in keys:
        cfg = int(key.split(".")[0])
        kv = "fp8" if key.endswith(".fp8") else "fp16"
        # "6.chunk": the chunk of config 6 without its decodes
        wl = (W.config6_chunked_prefill(num_decodes=0) if key.endswith(".chunk")
              else W.config(cfg))
        if cfg == 5:
            dev, entry = measure_write(wl, args, local, flush, stream, EXTRA_TIMED_S, peak,
                                       peak_kind)
            entry = {"workload": WORKLOAD_NAMES[5], **entry}
        elif cfg in (6, 7):
            dev, m = measure_chunk(wl, args, local, flush, stream, EXTRA_TIMED_S)
            entry = chunk_entry(key, wl, m, peak, peak_kind)
        else:
            dev, m = measure_decode(wl, args, kv, local, flush, stream, EXTRA_TIMED_S)
            entry = decode_entry(key, wl, dev, m, kv, peak, peak_kind)
            if cfg == 4:
                # the shared prefix is read once from DRAM and then from L2:
                # logical bytes per second, and the DRAM bytes / L2 hit rate of
                # the committed ncu record for this kernel source
                entry["logical_kv_gbs"] = round(
                    wl.kv_bytes() / (entry["decode_kernel_ms"] * 1e-3) / 1e9, 1)
                entry["dram_bytes_per_launch"] = entry["roofline"]["traffic"]
                entry["l2_sector_hit_rate_pct"] = recorded_decode_value(
                    f"l2_sector_hit_rate_pct.config4.{kv}")
                entry["unique_kv_bytes"] = unique_kv_bytes(wl)
        out[key] = entry
        del dev
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def unique_kv_bytes(wl) -> int:
    """Key+value bytes of the distinct (physical block, in-block slot) rows
    the sequences read: the shared prefix counted once."""
    seen = set()
    for i, L in enumerate(wl.seq_lens):
        L = int(L)
        nb = -(-L // wl.block_size)
        for j in range(nb):
            rows = min(wl.block_size, L - j * wl.block_size)
            seen.add((int(wl.block_tables[i, j]), rows))
    # a block shared by several sequences is read up to its longest use
    longest = {}
    for b, rows in seen:
        longest[b] = max(longest.get(b, 0), rows)
    return sum(longest.values()) * wl.num_kv_heads * wl.head_dim * 4


def main_chunk(args, wl, rank, world, local):
    """Multi-token step: write every new token's row, then the causal
    attention of each sequence's new tokens."""
    import torch

    pkv, dist = setup_device(args, local, world)
    from paged_kv_cache_131_gb300.harness import L2Flush

    flush = L2Flush(f"cuda:{local}")
    stream = torch.cuda.current_stream()
    dev, m = measure_chunk(wl, args, local, flush, stream, args.timed_s, dist=dist)
    st = spread(m["step_passes"])
    step_ms = max_over_ranks(st["median"], dist, f"cuda:{local}")
    if dist is not None:
        dist.barrier()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    peak_hbm, peak_kind = measured_peaks()
    roof, attn_ms = chunk_roofline(wl, m, peak_hbm, peak_kind)
    if args.chunk_only:
        roof["traffic"] = recorded_chunk_traffic("config6.chunk")
    elif args.config == 7:
        roof["traffic"] = recorded_traffic("config7.fp16")
    kv_bytes = wl.kv_bytes()
    Tq = wl.q.shape[0]
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        sampler = ChunkOracleSampler(wl)
        t_row = sampler.calibrate()
        n_rows = max(1, int(1.0 / t_row))
        gbs_cpu, t_cpu, n_cpu = sampler.run(n_rows, budget_s=15.0)
        cpu = {"value": round(gbs_cpu, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
               **host_cpu_info(),
               "sample": f"{n_cpu} x {n_rows} query rows (all heads), rotating, "
                         f"{t_cpu:.1f} s single-threaded float64"}
    line = {
        "metric": METRIC,
        "value": round(whole_job_gbs(kv_bytes, world, step_ms), 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "passes": m["passes"],
        "ms_per_step": round(step_ms, 5),
        "spread": {"ms_per_step_p10": round(st["p10"], 5), "ms_per_step_p90": round(st["p90"], 5)},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16xf16->f32",
        "data": "synthetic (seeded N(0,1) fp16, shuffled physical blocks)",
        "config": {"workload": CHUNK_ONLY_NAME if args.chunk_only else WORKLOAD_NAMES[args.config],
                   "global_batch": wl.num_seqs * world,
                   "query_tokens": Tq, "seq_len": int(wl.max_seq_len),
                   "parallelism": f"replicas x{world}", "l2": L2_NOTE,
                   "kv_cache": "resident in HBM (state), not copied per step"},
        "query_tokens_per_s": round(world * Tq / (step_ms * 1e-3), 1),
        "attention_kernel_ms": round(attn_ms, 5),
        "write_kernel_ms": round(spread(m["write_ms"])["median"], 5),
        "roofline": roof,
        "e2e": None,
        "gpu_launches": m["gpu_launches"],
        "clocks": m["clocks"],
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main_write(args, wl, rank, world, local):
    """Config 5: the two-cache byte-strided write.  Headline = the block-outer
    layout's four (cache, layer) writes in one launch."""
    import torch

    pkv, dist = setup_device(args, local, world)
    from paged_kv_cache_131_gb300.harness import L2Flush

    flush = L2Flush(f"cuda:{local}")
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peaks()
    dev, entries = measure_write(wl, args, local, flush, stream, args.timed_s / 4, peak,
                                 peak_kind, dist=dist)
    head = entries["BLHNC"]["one_launch"]
    step_ms = max_over_ranks(head["ms"], dist, f"cuda:{local}")
    alg = dev.layout_bytes("BLHNC")

    # end to end through the API from pinned host memory: every step copies
    # the rows and slot mapping in (one packed copy), writes, and reads the
    # device error word back (the write's result is the cache itself)
    host = dev.host_inputs(pinned=True)
    e2e_ms = []
    for i in range(5 + args.e2e_steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dev.inputs.copy_(host, non_blocking=True)
        dev.write_layout_batched("BLHNC")
        kind, _ = pkv.pkv_get_device_error()
        e1.record(stream)
        e1.synchronize()
        if kind:
            raise RuntimeError(f"device error {pkv.DEVICE_ERRORS.get(kind)}")
        if i >= 5:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_med = float(np.median(e2e_ms))
    if dist is not None:
        dist.barrier()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        gbs_cpu, t_cpu, n_cpu = WriteOracleSampler(wl).run(budget_s=10.0)
        cpu = {"value": round(gbs_cpu, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
               **host_cpu_info(),
               "sample": f"{n_cpu} steps of every (cache, layer) view of one layout, "
                         f"{t_cpu:.1f} s single-threaded"}
    line = {
        "metric": METRIC,
        "value": round(whole_job_gbs(alg, world, step_ms), 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "passes": head["passes"],
        "ms_per_step": round(step_ms, 5),
        "spread": {"ms_per_step_p10": head["ms_p10_p90"][0],
                   "ms_per_step_p90": head["ms_p10_p90"][1]},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u8",
        "data": "synthetic (seeded random bytes, slots drawn without replacement)",
        "config": {"workload": WORKLOAD_NAMES[5], "global_batch": int(wl.slot_mapping.size),
                   "parallelism": f"replicas x{world}", "l2": L2_NOTE,
                   "headline": "block-outer (BLHNC) layout, 4 (cache, layer) views in one launch"},
        "cache_write_gbs": head["value"],
        "roofline": head["roofline"],
        "layouts": entries,
        "e2e": {"value": round(alg / (e2e_med * 1e-3) / 1e9, 2), "unit": UNIT,
                "h2d_bytes_per_step": int(host.numel()), "d2h_bytes_per_step": 8,
                "ms_per_step": round(e2e_med, 5)},
        "gpu_launches": sum(e["gpu_launches"] for lay in entries.values()
                            for e in lay.values()),
        "clocks": head["clocks"],
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse()
    rank, world, local = dist_env()
    from paged_kv_cache_131_gb300 import workloads as W

    if args.chunk_only and args.config != 6:
        raise SystemExit("--chunk-only goes with --config 6")
    if args.chunk_only:
        wl = W.config6_chunked_prefill(num_decodes=0)
    elif args.config == 2 and args.kv_heads != 8:
        wl = W.config2_llama8b(num_kv_heads=args.kv_heads)
    else:
        wl = W.config(args.config)
    if args.impl == "reference":
        run_reference(args, wl, rank)
        return
    if args.config in (6, 7):
        main_chunk(args, wl, rank, world, local)
        return
    if args.config == 5:
        main_write(args, wl, rank, world, local)
        return

    import torch

    pkv, dist = setup_device(args, local, world)
    from paged_kv_cache_131_gb300.harness import L2Flush

    compute = {"auto": 0, "simt": 1, "mma": 2}[args.compute]
    schedule = {"auto": 0, "grid": 1, "balanced": 2}[args.schedule]
    flush = L2Flush(f"cuda:{local}")
    stream = torch.cuda.current_stream()
    dev, m = measure_decode(wl, args, args.kv, local, flush, stream, args.timed_s, dist=dist,
                            compute=compute, schedule=schedule, partition=args.partition)
    kv_bytes = dev.kv_bytes() if args.kv == "fp8" else wl.kv_bytes()
    S = wl.num_seqs
    alg = decode_alg_bytes(wl, kv_bytes)
    if args.kv == "fp8":
        t = wl.slot_mapping.size if dev.has_write else 0
        write_bytes = t * wl.num_kv_heads * (wl.head_dim * 3 + 4) * 2 + 8 * t
    else:
        write_bytes = dev.write_bytes()
    st = spread(m["step_passes"])
    step_ms = max_over_ranks(st["median"], dist, f"cuda:{local}")
    decode_ms = spread(m["decode_ms"])["median"]
    write_ms = spread(m["write_ms"])["median"] if dev.has_write else None
    if dist is not None:
        dist.barrier()

    # end to end through the public API: pinned host inputs in, output out
    e2e = e2e_measure(dev, wl, args.e2e_steps, stream, flush) if args.kv == "fp16" else None

    extras = None
    keys = [] if args.extras in ("", "none") else args.extras.split(",")
    if (rank == 0 and world == 1 and keys and args.config == 2 and args.kv == "fp16"
            and compute == 0 and schedule == 0 and args.partition == 0 and args.kv_heads == 8):
        del dev
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        peak, peak_kind = measured_peaks()
        extras = run_extras(args, keys, local, flush, stream, peak, peak_kind)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    peak, peak_kind = measured_peaks()
    value = whole_job_gbs(kv_bytes, world, step_ms)
    achieved = alg / (decode_ms * 1e-3) / 1e9
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        sampler = OracleSampler(wl)
        gbs, t_cpu, n_cpu = sampler.run(8, budget_s=15.0)
        cpu = {"value": round(gbs, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
               **host_cpu_info(),
               "sample": f"{n_cpu} steps x 8 (sequence, kv_head) units (all query heads) + the "
                         f"write of all new rows, {t_cpu:.1f} s single-threaded float64"}
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "passes": m["passes"],
        "ms_per_step": round(step_ms, 5),
        "spread": {"ms_per_step_p10": round(st["p10"], 5), "ms_per_step_p90": round(st["p90"], 5),
                   "value_p10": round(whole_job_gbs(kv_bytes, world, st["p90"]), 2),
                   "value_p90": round(whole_job_gbs(kv_bytes, world, st["p10"]), 2)},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16xf16->f32" if args.kv == "fp16" else "e4m3 KV (dequantized to f16) -> f32",
        "data": "synthetic (seeded N(0,1) fp16, shuffled physical blocks)",
        "config": {"workload": WORKLOAD_NAMES[args.config] if args.kv_heads == 8 or
                   args.config != 2 else
                   WORKLOAD_NAMES[2].replace("H=32, Hk=8", f"H={wl.num_heads}, Hk={wl.num_kv_heads}")
                   .replace("[16384,16,8,128]", f"[16384,16,{wl.num_kv_heads},128]"),
                   "global_batch": S * world,
                   "seq_len": int(wl.max_seq_len), "parallelism": f"replicas x{world}",
                   "l2": L2_NOTE + "; KV read per step > L2",
                   "kv_cache": "resident in HBM (state), not copied per step",
                   "compute": args.compute, "schedule": args.schedule, "kv": args.kv},
        "pct_hbm_peak": round(100 * value / world / peak, 2),
        "seqs_per_s": round(world * S / (step_ms * 1e-3), 1),
        "decode_tokens_per_s": round(world * S / (step_ms * 1e-3), 1),
        "cache_write_gbs": round(write_bytes / (write_ms * 1e-3) / 1e9, 2) if write_bytes else None,
        "decode_kernel_ms": round(decode_ms, 5),
        "write_kernel_ms": round(write_ms, 5) if write_ms is not None else None,
        "wall_s_timed_loop": round(m["wall_s"], 3),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     # recorded for the balanced schedule with the MMA policies only
                     "traffic": recorded_traffic(f"config{args.config}.{args.kv}")
                     if schedule != 1 and compute != 1 else None,
                     "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth)",
                     "kernel": ("decode_grid_kernel" if schedule == 1 else
                                "decode_balanced_kernel") +
                               (" (FP8 MMA policy)" if args.kv == "fp8" else
                                " (SIMT policy)" if compute == 1 else " (MMA policy)"),
                     "alg_bytes_per_launch": alg},
        "e2e": e2e,
        "gpu_launches": m["gpu_launches"],
        "clocks": m["clocks"],
        "cpu_baseline": cpu,
    }
    if extras is not None:
        line["configs"] = extras
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def e2e_measure(dev, wl, steps, stream, flush):
    """Same metric through the public API from pinned host buffers: per step the
    step's inputs (q, new K/V rows, slot_mapping, block tables, seq_lens,
    packed in one pinned buffer) go host -> device in one copy, the library
    runs, the output comes back device -> host.  L2 is flushed between steps,
    outside the timed events."""
    import torch

    host = dev.host_inputs(pinned=True)  # all per-step inputs, packed: one copy in
    out_host = torch.empty(tuple(wl.q.shape), dtype=torch.float16).pin_memory()
    h2d = host.numel()
    d2h = out_host.numel() * out_host.element_size()

    def one():
        dev.inputs.copy_(host, non_blocking=True)
        dev.step()
        out_host.copy_(dev.out, non_blocking=True)

    for _ in range(5):
        flush()
        one()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for e0, e1 in ev:
        flush()
        e0.record(stream)
        one()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = float(np.median([e0.elapsed_time(e1) for e0, e1 in ev]))
    return {"value": round(wl.kv_bytes() / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms, 5)}


if __name__ == "__main__":
    main()
