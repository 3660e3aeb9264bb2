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
between timed steps).  `e2e` is the same metric through the public API with
the step's inputs copied from pinned host memory and the output copied back
inside the timed region.  `roofline` is the decode kernel's algorithmic bytes
per launch / its event-timed duration against the measured HBM copy
bandwidth.  `cpu_baseline` times the float64 oracle on the host.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config 2|3|4|6|7] [--compute auto|simt|mma] [--kv fp16|fp8]

Configs 6 and 7 time the multi-token step instead: the write of every new
token's row, then the causal attention of each sequence's new tokens
(pkv_chunk_attention) -- 6 is one engine step of chunked prefill (a
952-token prompt chunk beside 63 decodes), 7 is 4-token draft verification
on 64 sequences.
"""

from __future__ import annotations

import argparse
import hashlib
import json
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

WORKLOAD_NAMES = {
    2: "llama3-8b decode layer: S=64, L~U[256,4096], bs=16, H=32, Hk=8, D=128, "
       "fp16 cache [16384,16,8,128], 1 new token/seq written",
    3: "long context: S=8, L=32768, bs=16, H=32, Hk=8, D=128, 16384 shuffled blocks, decode only",
    4: "shared prefix: S=256, 2000-token shared prefix + tail U[1,300], bs=16, H=64, Hk=8, "
       "D=128, 16384 blocks, 1 new token/seq written",
    6: "chunked-prefill step: 952-token chunk of a 3000-token prompt (positions 2048..2999) + "
       "63 decodes L~U[256,4096], bs=16, H=32, Hk=8, D=128, 16384 shuffled blocks, new rows "
       "written first",
    7: "draft verification: S=64, 4 new tokens each, L~U[256,4096], bs=16, H=32, Hk=8, D=128, "
       "16384 shuffled blocks, new rows written first",
}

DECODE_SOURCES = [os.path.join(ROOT, "paged_kv_cache_131_gb300", "csrc", f)
                  for f in ("pkv_decode_balanced.cu", "pkv_decode_common.cuh", "pkv_device.cuh",
                            "pkv_tensor_map.cu")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_kernel_dram_traffic.txt")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, choices=[2, 3, 4, 6, 7])
    ap.add_argument("--compute", choices=["auto", "simt", "mma"], default="auto")
    ap.add_argument("--schedule", choices=["auto", "grid", "balanced"], default="auto")
    ap.add_argument("--kv", choices=["fp16", "fp8"], default="fp16",
                    help="KV cache format (fp8: E4M3 codes + per-row fp32 scales)")
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=200)
    return ap.parse_args()


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


def decode_source_hash() -> str:
    h = hashlib.sha256()
    for p in DECODE_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_key: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode kernel source (else None)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    rec = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                rec[k.strip()] = v.strip()
    if rec.get("source_hash") != decode_source_hash():
        return None
    v = rec.get(f"traffic_bytes_per_launch.{workload_key}")
    return float(v) if v else None


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


def run_reference(args, wl, rank):
    if rank != 0:
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
        line = {
            "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t / n * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAMES[args.config], "sample": sample},
            "cpu_baseline": {"value": round(gbs, 4), "unit": UNIT, "cores": 1,
                             "kind": "oracle", "sample": sample, **host_cpu_info()},
            "e2e": {"value": round(gbs, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
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
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t / n * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAMES[args.config], "sample": sample},
        "cpu_baseline": {"value": round(gbs, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, **host_cpu_info()},
        "e2e": {"value": round(gbs, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


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


def main_chunk(args, wl, rank, world, local):
    """Multi-token step: write every new token's row, then the causal
    attention of each sequence's new tokens."""
    import torch

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import paged_kv_cache_131_gb300 as pkv
    from paged_kv_cache_131_gb300 import _build
    from paged_kv_cache_131_gb300.harness import DeviceChunk, L2Flush

    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build()
    if dist is not None:
        dist.barrier()
    dev = DeviceChunk(wl, device=f"cuda:{local}")
    flush = L2Flush(f"cuda:{local}")
    stream = torch.cuda.current_stream()
    kv_bytes = wl.kv_bytes()
    flops = wl.flops()
    Tq, H, D = wl.q.shape
    nblk = int(sum(-(-int(L) // wl.block_size) for L in wl.seq_lens))
    # algorithmic bytes of the attention: every sequence's K and V once, q in,
    # out, block tables, lengths and query offsets
    attn_bytes = kv_bytes + Tq * H * D * 2 * 2 + nblk * 4 + wl.num_seqs * 8 + 4
    for _ in range(args.warmup):
        flush()
        dev.step()
    torch.cuda.synchronize()
    kind, idx = pkv.pkv_get_device_error()
    if kind:
        raise RuntimeError(f"device error {pkv.DEVICE_ERRORS.get(kind)} at {idx}")
    K = args.steps
    # the step's launches (write; one or two attention kernels and the plan
    # kernel) are captured once as CUDA graphs and replayed, so no Python
    # enqueue sits inside the timed region
    # (one graph for the whole step, so the attention call may overlap the
    # write's tail as it does on a stream; two for the pass that times each)
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

    def timed_loop(split: bool):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        for i in range(K):
            flush()
            ev[i][0].record(stream)
            if split:
                g_write.replay()
                ev[i][1].record(stream)
                g_attend.replay()
            else:
                g_step.replay()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        step = sum(e[0].elapsed_time(e[2]) for e in ev) / K
        if not split:
            return step, None, None
        return (step, float(np.median([e[0].elapsed_time(e[1]) for e in ev])),
                float(np.median([e[1].elapsed_time(e[2]) for e in ev])))

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        step_ms, _, _ = timed_loop(split=False)
        _, write_ms, attn_ms = timed_loop(split=True)
    if dist is not None:
        step_ms = max_over_ranks(step_ms, dist, f"cuda:{local}")
        dist.barrier()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    peak_hbm, peak_kind = measured_peaks()
    peak_tf = measured_bf16_tflops()
    value = whole_job_gbs(kv_bytes, world, step_ms)
    gbs = attn_bytes / (attn_ms * 1e-3) / 1e9
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
                 "alg_bytes_per_launch": attn_bytes,
                 "flops_per_launch": flops, "achieved_gbs": round(gbs, 1),
                 "achieved_tflops": round(tfs, 2), "hbm_frac": round(hbm_frac, 4),
                 "tensor_frac": round(tf_frac, 4)})
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
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16xf16->f32",
        "data": "synthetic (seeded N(0,1) fp16, shuffled physical blocks)",
        "config": {"workload": WORKLOAD_NAMES[args.config], "global_batch": wl.num_seqs * world,
                   "query_tokens": Tq, "seq_len": int(wl.max_seq_len),
                   "parallelism": f"replicas x{world}",
                   "l2": "flushed between timed steps (write a 2x L2 buffer, then read another "
                         "2x L2 buffer: cold, clean L2)",
                   "kv_cache": "resident in HBM (state), not copied per step"},
        "query_tokens_per_s": round(world * Tq / (step_ms * 1e-3), 1),
        "attention_kernel_ms": round(attn_ms, 5),
        "write_kernel_ms": round(write_ms, 5),
        "roofline": roof,
        "e2e": None,
        "gpu_launches": chunk_launches_per_step(wl) * K,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse()
    rank, world, local = dist_env()
    from paged_kv_cache_131_gb300 import workloads as W

    wl = W.config(args.config)
    if args.impl == "reference":
        run_reference(args, wl, rank)
        return
    if args.config in (6, 7):
        main_chunk(args, wl, rank, world, local)
        return

    import torch

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import paged_kv_cache_131_gb300 as pkv
    from paged_kv_cache_131_gb300 import _build
    from paged_kv_cache_131_gb300.harness import DeviceDecode, L2Flush

    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build()
    if dist is not None:
        dist.barrier()
    compute = {"auto": 0, "simt": 1, "mma": 2}[args.compute]
    schedule = {"auto": 0, "grid": 1, "balanced": 2}[args.schedule]
    if args.kv == "fp8":
        from paged_kv_cache_131_gb300.harness import DeviceDecodeFp8
        dev = DeviceDecodeFp8(wl, device=f"cuda:{local}")
    else:
        dev = DeviceDecode(wl, device=f"cuda:{local}", partition_size=args.partition,
                           compute=compute, schedule=schedule)
    flush = L2Flush(f"cuda:{local}")
    stream = torch.cuda.current_stream()

    kv_bytes = dev.kv_bytes() if args.kv == "fp8" else wl.kv_bytes()
    S, H, D = wl.num_seqs, wl.num_heads, wl.head_dim
    nblk = int(sum(-(-int(L) // wl.block_size) for L in wl.seq_lens))
    decode_alg_bytes = kv_bytes + S * H * D * 2 * 2 + nblk * 4 + S * 4
    if args.kv == "fp8":
        t = wl.slot_mapping.size if dev.has_write else 0
        write_bytes = t * wl.num_kv_heads * (wl.head_dim * 3 + 4) * 2 + 8 * t
    else:
        write_bytes = dev.write_bytes()
    launches_per_step = (1 if dev.has_write else 0) + 1

    for _ in range(args.warmup):
        flush()
        dev.step()
    torch.cuda.synchronize()
    kind, idx = pkv.pkv_get_device_error()
    if kind:
        raise RuntimeError(f"device error {pkv.DEVICE_ERRORS.get(kind)} at {idx}")

    K = args.steps

    def timed_loop(split: bool):
        """K steps, L2 flushed before each (outside the events).  Without
        `split` only the step's ends are marked, so the decode launch may
        overlap the write kernel's tail as it does in use; with `split` an
        event between them gives each kernel's own duration."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        for i in range(K):
            flush()
            ev[i][0].record(stream)
            dev.write()
            if split:
                ev[i][1].record(stream)
            dev.decode()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        step = sum(e[0].elapsed_time(e[2]) for e in ev) / K
        if not split:
            return step, None, None
        # per-kernel durations: medians, so a step where the host fell behind
        # the GPU (launch latency landing between two events) does not skew them
        return (step, float(np.median([e[0].elapsed_time(e[1]) for e in ev])),
                float(np.median([e[1].elapsed_time(e[2]) for e in ev])))

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        step_ms, _, _ = timed_loop(split=False)
        t_wall = time.perf_counter() - t_wall
        _, write_ms, decode_ms = timed_loop(split=True)
    if dist is not None:
        step_ms = max_over_ranks(step_ms, dist, f"cuda:{local}")
        dist.barrier()

    # end to end through the public API: pinned host inputs in, output out
    e2e = e2e_measure(dev, wl, args.e2e_steps, stream, flush) if args.kv == "fp16" else None

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    peak, peak_kind = measured_peaks()
    value = whole_job_gbs(kv_bytes, world, step_ms)
    achieved = decode_alg_bytes / (decode_ms * 1e-3) / 1e9
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
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16xf16->f32" if args.kv == "fp16" else "e4m3 KV (dequantized to f16) -> f32",
        "data": "synthetic (seeded N(0,1) fp16, shuffled physical blocks)",
        "config": {"workload": WORKLOAD_NAMES[args.config], "global_batch": S * world,
                   "seq_len": int(wl.max_seq_len), "parallelism": f"replicas x{world}",
                   "l2": "flushed between timed steps (write a 2x L2 buffer, then read another "
                         "2x L2 buffer: cold, clean L2); KV read per step > L2",
                   "kv_cache": "resident in HBM (state), not copied per step",
                   "compute": args.compute, "schedule": args.schedule, "kv": args.kv},
        "pct_hbm_peak": round(100 * value / world / peak, 2),
        "seqs_per_s": round(world * S / (step_ms * 1e-3), 1),
        "decode_tokens_per_s": round(world * S / (step_ms * 1e-3), 1),
        "cache_write_gbs": round(write_bytes / (write_ms * 1e-3) / 1e9, 2) if write_bytes else None,
        "decode_kernel_ms": round(decode_ms, 5),
        "write_kernel_ms": round(write_ms, 5),
        "wall_s_timed_loop": round(t_wall, 3),
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
                     "alg_bytes_per_launch": decode_alg_bytes},
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
    }
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
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
    return {"value": round(wl.kv_bytes() / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms, 5)}


if __name__ == "__main__":
    main()
