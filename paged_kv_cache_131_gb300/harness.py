"""Device staging of the synthetic workloads, for the benchmark and the tests.

Copies a ``workloads.DecodeWorkload`` / ``WriteWorkload`` into CUDA tensors
and runs the library's calls on them.  Torch is used for device memory and
streams only; every computation runs in libpagedkv's kernels.
"""

from __future__ import annotations

import numpy as np
import torch

from . import (PKV_COMPUTE_AUTO, PKV_SCHEDULE_AUTO, pkv_cache_write, pkv_cache_write_fp8,
               pkv_cache_write_multi, pkv_chunk_attention, pkv_chunk_workspace_bytes,
               pkv_decode_attention, pkv_decode_attention_fp8, pkv_decode_workspace_bytes,
               pkv_view)
from .workloads import ChunkWorkload, DecodeWorkload, WriteWorkload, slot_of


def to_dev(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DeviceDecode:
    """One decode workload resident on the device: caches, tables, q, out, workspace."""

    def __init__(self, wl: DecodeWorkload, device="cuda", partition_size: int = 0,
                 compute: int = PKV_COMPUTE_AUTO, schedule: int = PKV_SCHEDULE_AUTO):
        self.wl = wl
        self.device = torch.device(device)
        self.partition_size = partition_size
        self.compute = compute
        self.schedule = schedule
        self.k_cache = to_dev(wl.k_cache, device)
        self.v_cache = to_dev(wl.v_cache, device)
        self.has_write = wl.slot_mapping is not None and wl.slot_mapping.size > 0
        # the per-step inputs live in one device buffer (256-byte aligned
        # fields), so a host step can bring them in with a single copy
        fields = [("q", wl.q), ("block_tables", wl.block_tables), ("seq_lens", wl.seq_lens)]
        if self.has_write:
            fields += [("k_new", wl.k_new), ("v_new", wl.v_new),
                       ("slot_mapping", wl.slot_mapping)]
        self._layout, off = [], 0
        for name, a in fields:
            a = np.ascontiguousarray(a)
            self._layout.append((name, off, a.dtype, a.shape))
            off += (a.nbytes + 255) // 256 * 256
        self.inputs_nbytes = off
        host = self.host_inputs(pinned=False)
        self.inputs = host.to(device)
        for name, o, dtype, shape in self._layout:
            n = int(np.prod(shape)) * np.dtype(dtype).itemsize
            t = self.inputs[o:o + n].view(torch.from_numpy(np.empty(0, dtype)).dtype)
            setattr(self, name, t.view(shape))
        self.out = torch.empty_like(self.q)
        with torch.cuda.device(self.device):
            nbytes = pkv_decode_workspace_bytes(wl.num_seqs, wl.num_heads, wl.num_kv_heads,
                                                wl.head_dim, wl.max_seq_len, partition_size)
        # zero-filled once; every decode call leaves its tickets at zero again
        self.workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=device) \
            if nbytes else None

    def host_inputs(self, pinned: bool = True) -> torch.Tensor:
        """The per-step inputs packed as in ``self.inputs`` (uint8, host)."""
        buf = np.zeros(self.inputs_nbytes, dtype=np.uint8)
        for name, o, dtype, shape in self._layout:
            a = np.ascontiguousarray(getattr(self.wl, name)).view(np.uint8).reshape(-1)
            buf[o:o + a.size] = a
        t = torch.from_numpy(buf)
        return t.pin_memory() if pinned else t

    @property
    def row_bytes(self) -> int:
        return self.wl.num_kv_heads * self.wl.head_dim * 2

    def view(self) -> pkv_view:
        r = self.row_bytes
        return pkv_view(0, 0, self.wl.block_size * r, r, 0)

    def write(self, stream=None) -> None:
        if self.has_write:
            pkv_cache_write(self.k_new, self.v_new, self.slot_mapping, self.k_cache,
                            self.v_cache, self.view(), self.wl.block_size, self.wl.num_blocks,
                            stream=stream)

    def decode(self, stream=None, out=None) -> torch.Tensor:
        wl = self.wl
        out = self.out if out is None else out
        pkv_decode_attention(out, self.q, self.k_cache, self.v_cache, self.block_tables,
                             self.seq_lens, wl.scale, wl.num_heads, wl.num_kv_heads,
                             wl.head_dim, wl.block_size, wl.max_seq_len, wl.num_blocks,
                             workspace=self.workspace, stream=stream,
                             partition_size=self.partition_size, compute=self.compute,
                             schedule=self.schedule)
        return out

    def step(self, stream=None) -> torch.Tensor:
        """One pass of the hot path: write the new token rows, then decode."""
        self.write(stream)
        return self.decode(stream)

    def write_bytes(self) -> int:
        """Algorithmic bytes of the write: rows read + rows written + slot_mapping."""
        if not self.has_write:
            return 0
        t = self.wl.slot_mapping.size
        return 2 * 2 * t * self.row_bytes + 8 * t


def prior_token_rows(wl: DecodeWorkload):
    """Slots and fp16 K/V rows [n, Hk, D] of every token already in the cache
    before the new tokens (the rows the fp16 workload stored there)."""
    bs = wl.block_size
    seen, slots = set(), []
    new = set(wl.slot_mapping.tolist()) if wl.slot_mapping is not None else set()
    for i, L in enumerate(wl.seq_lens):
        for pos in range(int(L)):
            s = slot_of(wl.block_tables[i], pos, bs)
            if s not in seen and s not in new:
                seen.add(s)
                slots.append(s)
    slots = np.asarray(slots, dtype=np.int64)
    rows_k = wl.k_cache.reshape(-1, wl.num_kv_heads, wl.head_dim)[slots]
    rows_v = wl.v_cache.reshape(-1, wl.num_kv_heads, wl.head_dim)[slots]
    return slots, rows_k, rows_v


class DeviceDecodeFp8:
    """A decode workload held in FP8 (E4M3) caches: the tokens already in the
    fp16 workload's cache are quantized into place by the library's FP8 write
    (unwritten slots keep NaN codes and NaN scales), then each step writes the
    new tokens (FP8) and decodes."""

    def __init__(self, wl: DecodeWorkload, device="cuda"):
        self.wl = wl
        NB, bs, Hk, D = wl.k_cache.shape
        self.k_cache = torch.full((NB, bs, Hk, D), 0x7F, dtype=torch.uint8, device=device)
        self.v_cache = torch.full((NB, bs, Hk, D), 0x7F, dtype=torch.uint8, device=device)
        self.k_scale = torch.full((NB, bs, Hk), float("nan"), dtype=torch.float32, device=device)
        self.v_scale = torch.full((NB, bs, Hk), float("nan"), dtype=torch.float32, device=device)
        self.prior_slots, rk, rv = prior_token_rows(wl)
        if self.prior_slots.size:
            pkv_cache_write_fp8(to_dev(rk, device), to_dev(rv, device),
                                to_dev(self.prior_slots, device), self.k_cache, self.v_cache,
                                self.k_scale, self.v_scale, bs, NB)
        self.q = to_dev(wl.q, device)
        self.block_tables = to_dev(wl.block_tables, device)
        self.seq_lens = to_dev(wl.seq_lens, device)
        self.out = torch.empty_like(self.q)
        self.has_write = wl.slot_mapping is not None and wl.slot_mapping.size > 0
        if self.has_write:
            self.k_new = to_dev(wl.k_new.reshape(-1, Hk, D), device)
            self.v_new = to_dev(wl.v_new.reshape(-1, Hk, D), device)
            self.slot_mapping = to_dev(wl.slot_mapping, device)
        with torch.cuda.device(torch.device(device)):
            nbytes = pkv_decode_workspace_bytes(wl.num_seqs, wl.num_heads, wl.num_kv_heads,
                                                wl.head_dim, max(wl.max_seq_len, 1))
        self.workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=device)

    def write(self, stream=None) -> None:
        if self.has_write:
            pkv_cache_write_fp8(self.k_new, self.v_new, self.slot_mapping, self.k_cache,
                                self.v_cache, self.k_scale, self.v_scale, self.wl.block_size,
                                self.wl.num_blocks, stream=stream)

    def decode(self, stream=None) -> torch.Tensor:
        wl = self.wl
        pkv_decode_attention_fp8(self.out, self.q, self.k_cache, self.v_cache, self.k_scale,
                                 self.v_scale, self.block_tables, self.seq_lens, wl.scale,
                                 wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                                 wl.max_seq_len, wl.num_blocks, self.workspace, stream=stream)
        return self.out

    def step(self, stream=None) -> torch.Tensor:
        self.write(stream)
        return self.decode(stream)

    def kv_bytes(self) -> int:
        """Bytes the FP8 decode reads: codes (1 B) + one fp32 scale per row, K and V."""
        wl = self.wl
        return int(wl.seq_lens.astype(np.int64).sum()) * wl.num_kv_heads * (wl.head_dim + 4) * 2


class DeviceWrite:
    """The byte-strided two-cache write workload resident on the device."""

    def __init__(self, wl: WriteWorkload, device="cuda"):
        self.wl = wl
        self.cache = to_dev(wl.init, device)
        # the per-step inputs (every (cache, layer) row set and the slot
        # mapping) live in one device buffer at 256-byte aligned offsets, so a
        # host step can bring them in with a single copy
        fields = [(key, r) for key, r in wl.rows.items()] + [("slot_mapping", wl.slot_mapping)]
        self._layout, off = [], 0
        for key, a in fields:
            a = np.ascontiguousarray(a)
            self._layout.append((key, off, a.dtype, a.shape))
            off += (a.nbytes + 255) // 256 * 256
        self.inputs_nbytes = off
        self.inputs = self.host_inputs(pinned=False).to(device)
        self.rows = {}
        for key, o, dtype, shape in self._layout:
            n = int(np.prod(shape)) * np.dtype(dtype).itemsize
            t = self.inputs[o:o + n].view(torch.from_numpy(np.empty(0, dtype)).dtype).view(shape)
            if key == "slot_mapping":
                self.slot_mapping = t
            else:
                self.rows[key] = t

    def host_inputs(self, pinned: bool = True) -> torch.Tensor:
        """The per-step inputs packed as in ``self.inputs`` (uint8, host)."""
        buf = np.zeros(self.inputs_nbytes, dtype=np.uint8)
        for key, o, dtype, shape in self._layout:
            src = self.wl.slot_mapping if key == "slot_mapping" else self.wl.rows[key]
            a = np.ascontiguousarray(src).view(np.uint8).reshape(-1)
            buf[o:o + a.size] = a
        t = torch.from_numpy(buf)
        return t.pin_memory() if pinned else t

    def reset(self) -> None:
        self.cache.copy_(torch.from_numpy(self.wl.init))

    def write_layout(self, layout: str, stream=None) -> int:
        """All (cache, layer) writes of one layout; returns the number of calls."""
        n = 0
        for c, v in self.wl.views[layout].items():
            for layer in range(self.wl.num_layers):
                pkv_cache_write(self.rows[(c, layer)], None, self.slot_mapping, self.cache, None,
                                pkv_view(v.offset, v.layer_stride, v.block_stride, v.row_width,
                                         layer),
                                self.wl.block_size, self.wl.num_blocks, stream=stream)
                n += 1
        return n

    def write_layout_batched(self, layout: str, stream=None) -> int:
        """All (cache, layer) writes of one layout in one launch."""
        writes = []
        for c, v in self.wl.views[layout].items():
            for layer in range(self.wl.num_layers):
                writes.append((self.rows[(c, layer)], self.cache,
                               pkv_view(v.offset, v.layer_stride, v.block_stride, v.row_width,
                                        layer)))
        pkv_cache_write_multi(writes, self.slot_mapping, self.wl.block_size, self.wl.num_blocks,
                              stream=stream)
        return 1

    def layout_bytes(self, layout: str) -> int:
        """Algorithmic bytes of one layout's writes: every row read once and
        written once, plus the slot mapping read once (it is shared by all
        (cache, layer) views)."""
        t = self.wl.slot_mapping.size
        per = sum(v.row_width for v in self.wl.views[layout].values()) * self.wl.num_layers
        return 2 * t * per + 8 * t


class DeviceChunk:
    """A chunk workload on the device: each step writes the new tokens' rows
    (pkv_cache_write), then runs the causal attention of every sequence's new
    tokens (pkv_chunk_attention)."""

    def __init__(self, wl: ChunkWorkload, device="cuda"):
        self.wl = wl
        self.device = torch.device(device)
        self.k_cache = to_dev(wl.k_cache, device)
        self.v_cache = to_dev(wl.v_cache, device)
        self.q = to_dev(wl.q, device)
        self.block_tables = to_dev(wl.block_tables, device)
        self.seq_lens = to_dev(wl.seq_lens, device)
        self.query_start = to_dev(wl.query_start, device)
        self.k_new = to_dev(wl.k_new, device)
        self.v_new = to_dev(wl.v_new, device)
        self.slot_mapping = to_dev(wl.slot_mapping, device)
        self.out = torch.empty_like(self.q)
        with torch.cuda.device(self.device):
            nbytes = pkv_chunk_workspace_bytes(wl.num_seqs, wl.num_heads, wl.num_kv_heads,
                                               wl.head_dim, wl.num_query_tokens,
                                               max(wl.max_query_len, 1), max(wl.max_seq_len, 1))
        self.workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=device)

    def view(self) -> pkv_view:
        r = self.wl.num_kv_heads * self.wl.head_dim * 2
        return pkv_view(0, 0, self.wl.block_size * r, r, 0)

    def write(self, stream=None) -> None:
        pkv_cache_write(self.k_new, self.v_new, self.slot_mapping, self.k_cache, self.v_cache,
                        self.view(), self.wl.block_size, self.wl.num_blocks, stream=stream)

    def attend(self, stream=None) -> torch.Tensor:
        wl = self.wl
        pkv_chunk_attention(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                            self.seq_lens, self.query_start, wl.scale, wl.num_heads,
                            wl.num_kv_heads, wl.head_dim, wl.block_size, max(wl.max_query_len, 1),
                            max(wl.max_seq_len, 1), wl.num_blocks, workspace=self.workspace,
                            stream=stream)
        return self.out

    def step(self, stream=None) -> torch.Tensor:
        self.write(stream)
        return self.attend(stream)


class L2Flush:
    """Leaves L2 cold and clean for the next kernel: writes one buffer twice
    the size of L2, then reads another of that size (the reads evict the
    dirty lines of the write, so their write-back is not charged to the
    kernel that follows)."""

    def __init__(self, device="cuda", nbytes: int | None = None):
        if nbytes is None:
            props = torch.cuda.get_device_properties(device)
            nbytes = 2 * max(int(getattr(props, "L2_cache_size", 0)), 128 << 20)
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.clean = torch.ones(nbytes // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self) -> None:
        self.buf.fill_(1)
        torch.sum(self.clean, dim=0, out=self.sink)
