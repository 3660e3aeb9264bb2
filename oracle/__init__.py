"""Oracle for the paged KV-cache hot path -- TEST INFRASTRUCTURE ONLY.

Plain, single-threaded float64 CPU code (``pkv_oracle.c``) that restates what
the pages define: the slot split and byte-address formula of the cache write
("vLLM KV Cache Layout 可视化", 核心 / 查一个 token / kernel 那一侧) and textbook
softmax attention over a sequence's gathered blocks ("deep-dive-into-vllm-05"
§1.2, §2, §3.2; "vLLM 技术内幕" §2.1).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library and the library never calls it.

Every function here is pinned by ``tests/test_oracle_pins.py`` to values the
pages print, closed forms, invariants and an independent brute force.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c with the host C compiler (portable flags only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load(path: str | None = None):
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_slot_address.restype = _i64
    lib.oracle_slot_address.argtypes = [_i64] * 7
    lib.oracle_split_slot.restype = None
    lib.oracle_split_slot.argtypes = [_i64, _i64, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]
    lib.oracle_cache_write.restype = _i64
    lib.oracle_cache_write.argtypes = [_p, _i64, _p, _p, _i64] + [_i64] * 7
    lib.oracle_e4m3_value.restype = ctypes.c_double
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_quantize_row.restype = None
    lib.oracle_quantize_row.argtypes = [_p, _i64, _p, _p]
    lib.oracle_cache_write_fp8.restype = _i64
    lib.oracle_cache_write_fp8.argtypes = [_p, _p, _p, _p] + [_i64] * 5
    lib.oracle_decode_attention_fp8.restype = ctypes.c_int
    lib.oracle_decode_attention_fp8.argtypes = [_p] * 8 + [ctypes.c_double] + [_i64] * 7 + [_p, _i64]
    lib.oracle_copy_blocks.restype = _i64
    lib.oracle_copy_blocks.argtypes = [_p, _i64, _p] + [_i64] * 9
    lib.oracle_decode_attention.restype = ctypes.c_int
    lib.oracle_decode_attention.argtypes = [_p] * 6 + [ctypes.c_double] + [_i64] * 7 + [_p, _i64]
    lib.oracle_chunk_attention.restype = ctypes.c_int
    lib.oracle_chunk_attention.argtypes = [_p] * 7 + [ctypes.c_double] + [_i64] * 7 + [_p, _i64]
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _split_rows(rows, workers: int):
    """Split a list of independent output rows into ``workers`` interleaved
    parts (interleaving spreads long and short rows evenly)."""
    return [rows[w::workers] for w in range(workers) if rows[w::workers]]


def _in_threads(fn, parts):
    """Run ``fn(part)`` for every part on its own thread and return the
    results in order.  The C calls release the GIL, so the parts run on
    several cores; each output row is still computed by one call of the
    same single-threaded function, so the arithmetic of a row does not
    depend on the split."""
    from concurrent.futures import ThreadPoolExecutor

    with ThreadPoolExecutor(max_workers=len(parts)) as ex:
        return list(ex.map(fn, parts))


def default_workers() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        n = os.cpu_count() or 1
    return max(1, n)


# --------------------------------------------------------------------------
# Python-facing functions.  ``lib`` lets a test run the same calls against a
# deliberately mutated build of the C source.


def half_to_double(bits: int, lib=None) -> float:
    return (lib or _load()).oracle_half_to_double(int(bits) & 0xFFFF)


def split_slot(slot: int, block_size: int, lib=None) -> tuple[int, int]:
    b, o = _i64(), _i64()
    (lib or _load()).oracle_split_slot(slot, block_size, ctypes.byref(b), ctypes.byref(o))
    return b.value, o.value


def slot_address(slot: int, block_size: int, offset: int, layer: int, layer_stride: int,
                 block_stride: int, row_width: int, lib=None) -> int:
    return (lib or _load()).oracle_slot_address(slot, block_size, offset, layer, layer_stride,
                                                block_stride, row_width)


def cache_write(cache: np.ndarray, src: np.ndarray, slot_mapping: np.ndarray, *, offset: int,
                layer: int, layer_stride: int, block_stride: int, row_width: int,
                block_size: int, num_blocks: int, lib=None) -> int:
    """Scatter rows of ``src`` (uint8 [T, row_width]) into ``cache`` (uint8, in place)."""
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    src = np.ascontiguousarray(src, dtype=np.uint8)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert src.size == slots.size * row_width
    n = (lib or _load()).oracle_cache_write(
        _ptr(cache), cache.nbytes, _ptr(src), _ptr(slots), slots.size, offset, layer,
        layer_stride, block_stride, row_width, block_size, num_blocks)
    if n < 0:
        raise ValueError(f"oracle_cache_write failed with status {n}")
    return n


def copy_blocks(cache: np.ndarray, pairs, *, offset: int, layer: int, num_layers: int,
                layer_stride: int, block_stride: int, row_width: int, block_size: int,
                num_blocks: int, lib=None) -> int:
    """Copy whole block pages (uint8 ``cache``, in place) for each (src, dst) pair."""
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    pa = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    n = (lib or _load()).oracle_copy_blocks(
        _ptr(cache), cache.nbytes, _ptr(pa), pa.shape[0], offset, layer, num_layers,
        layer_stride, block_stride, row_width, block_size, num_blocks)
    if n < 0:
        raise ValueError(f"oracle_copy_blocks failed with status {n}")
    return n


def decode_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                     block_tables: np.ndarray, seq_lens: np.ndarray, scale: float, *,
                     pairs=None, lib=None, workers: int = 1) -> np.ndarray:
    """Textbook paged decode attention in float64.

    q: fp16 [S, H, D]; caches: fp16 [NB, bs, Hk, D]; block_tables int32 [S, MB];
    seq_lens int32 [S].  Returns float64 [S, H, D]; with ``pairs`` (a list of
    (seq, head)) only those rows are computed (the others are NaN).  With
    ``workers`` > 1 the (seq, head) rows are split over that many threads.
    """
    if workers > 1:
        S, H = q.shape[0], q.shape[1]
        rows = [tuple(p) for p in pairs] if pairs is not None else \
            [(i, h) for i in range(S) for h in range(H)]
        parts = _split_rows(rows, workers)
        outs = _in_threads(lambda part: decode_attention(
            q, k_cache, v_cache, block_tables, seq_lens, scale, pairs=part, lib=lib), parts)
        out = np.full((S, H, q.shape[2]), np.nan, dtype=np.float64)
        for part, o in zip(parts, outs):
            idx = tuple(np.asarray(part).T)
            out[idx] = o[idx]
        return out
    q = np.ascontiguousarray(q, dtype=np.float16)
    assert k_cache.dtype == np.float16 and v_cache.dtype == np.float16
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    S, H, D = q.shape
    NB, bs, Hk, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    assert bt.shape[0] == S and sl.shape == (S,)
    out = np.full((S, H, D), np.nan, dtype=np.float64)
    if pairs is None:
        pp, npairs = None, 0
    else:
        pa = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        pp, npairs = _ptr(pa), pa.shape[0]
    st = (lib or _load()).oracle_decode_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(sl), float(scale),
        S, H, Hk, D, bs, bt.shape[1], NB, pp, npairs)
    if st != 0:
        raise ValueError(f"oracle_decode_attention failed with status {st}")
    return out


# --------------------------------------------------------------------------
# FP8 (E4M3) KV cache


def e4m3_value(code: int, lib=None) -> float:
    return (lib or _load()).oracle_e4m3_value(int(code) & 0xFF)


def e4m3_encode(y: float, lib=None) -> int:
    return (lib or _load()).oracle_e4m3_encode(float(y))


def quantize_row(x: np.ndarray, lib=None):
    """fp16 row -> (uint8 E4M3 codes, fp32 scale)."""
    x = np.ascontiguousarray(x, dtype=np.float16)
    codes = np.empty(x.size, dtype=np.uint8)
    sc = ctypes.c_float()
    (lib or _load()).oracle_quantize_row(_ptr(x), x.size, _ptr(codes), ctypes.byref(sc))
    return codes, sc.value


def cache_write_fp8(cache: np.ndarray, scales: np.ndarray, src: np.ndarray,
                    slot_mapping: np.ndarray, *, block_size: int, lib=None,
                    workers: int = 1) -> int:
    """Quantize fp16 rows src [T, Hk, D] into cache uint8 [NB, bs, Hk, D] and
    scales fp32 [NB, bs, Hk] (both in place).  With ``workers`` > 1 and
    distinct slots (every row then lands in its own place, whatever the
    order), the tokens are split over that many threads."""
    assert cache.dtype == np.uint8 and scales.dtype == np.float32
    assert cache.flags.c_contiguous and scales.flags.c_contiguous
    NB, bs, Hk, D = cache.shape
    assert bs == block_size and scales.shape == (NB, bs, Hk)
    src = np.ascontiguousarray(src, dtype=np.float16).reshape(-1, Hk, D)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert src.shape[0] == slots.size
    if workers > 1 and slots.size > 1 and np.unique(slots).size == slots.size:
        bounds = np.linspace(0, slots.size, min(workers, slots.size) + 1).astype(np.int64)
        parts = [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
        counts = _in_threads(lambda ab: cache_write_fp8(
            cache, scales, src[ab[0]:ab[1]], slots[ab[0]:ab[1]], block_size=block_size,
            lib=lib), parts)
        return int(sum(counts))
    n = (lib or _load()).oracle_cache_write_fp8(_ptr(cache), _ptr(scales), _ptr(src),
                                                _ptr(slots), slots.size, Hk, D, bs, NB)
    if n < 0:
        raise ValueError(f"oracle_cache_write_fp8 failed with status {n}")
    return n


def decode_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens,
                         scale: float, *, pairs=None, lib=None, workers: int = 1) -> np.ndarray:
    """Textbook paged decode attention in float64 over E4M3 caches (dequantized
    exactly: value(code) * scale of the row).  ``workers`` as in
    ``decode_attention``."""
    if workers > 1:
        S, H = q.shape[0], q.shape[1]
        rows = [tuple(p) for p in pairs] if pairs is not None else \
            [(i, h) for i in range(S) for h in range(H)]
        parts = _split_rows(rows, workers)
        outs = _in_threads(lambda part: decode_attention_fp8(
            q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens, scale, pairs=part,
            lib=lib), parts)
        out = np.full((S, H, q.shape[2]), np.nan, dtype=np.float64)
        for part, o in zip(parts, outs):
            idx = tuple(np.asarray(part).T)
            out[idx] = o[idx]
        return out
    q = np.ascontiguousarray(q, dtype=np.float16)
    S, H, D = q.shape
    NB, bs, Hk, D2 = k_cache.shape
    assert D2 == D and k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    assert k_scale.dtype == np.float32 and k_scale.shape == (NB, bs, Hk)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.full((S, H, D), np.nan, dtype=np.float64)
    if pairs is None:
        pp, npairs = None, 0
    else:
        pa = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        pp, npairs = _ptr(pa), pa.shape[0]
    st = (lib or _load()).oracle_decode_attention_fp8(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _ptr(bt), _ptr(sl), float(scale), S, H, Hk, D, bs, bt.shape[1], NB, pp, npairs)
    if st != 0:
        raise ValueError(f"oracle_decode_attention_fp8 failed with status {st}")
    return out


# --------------------------------------------------------------------------
# Chunk of new tokens per sequence (chunked prefill / draft verification)


def chunk_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                    block_tables: np.ndarray, seq_lens: np.ndarray, query_start: np.ndarray,
                    scale: float, *, rows=None, lib=None, workers: int = 1) -> np.ndarray:
    """Causal attention of each sequence's last Q_i = query_start[i+1] -
    query_start[i] tokens over its cache, in float64.

    q: fp16 [Tq, H, D] (Tq = query_start[-1]); caches fp16 [NB, bs, Hk, D];
    block_tables int32 [S, MB]; seq_lens int32 [S] (tokens in the cache,
    the new ones included).  Returns float64 [Tq, H, D]; with ``rows`` only
    those query rows are computed (the others are NaN).  With ``workers`` > 1
    the query rows are split over that many threads.
    """
    if workers > 1:
        all_rows = list(range(q.shape[0])) if rows is None else [int(r) for r in rows]
        parts = _split_rows(all_rows, workers)
        outs = _in_threads(lambda part: chunk_attention(
            q, k_cache, v_cache, block_tables, seq_lens, query_start, scale, rows=part,
            lib=lib), parts)
        out = np.full(q.shape, np.nan, dtype=np.float64)
        for part, o in zip(parts, outs):
            out[part] = o[part]
        return out
    q = np.ascontiguousarray(q, dtype=np.float16)
    assert k_cache.dtype == np.float16 and v_cache.dtype == np.float16
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    Tq, H, D = q.shape
    NB, bs, Hk, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    S = sl.size
    assert bt.shape[0] == S and qs.shape == (S + 1,) and int(qs[-1]) == Tq
    out = np.full((Tq, H, D), np.nan, dtype=np.float64)
    if rows is None:
        rp, nr = None, 0
    else:
        ra = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        rp, nr = _ptr(ra), ra.size
    st = (lib or _load()).oracle_chunk_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(sl), _ptr(qs),
        float(scale), S, H, Hk, D, bs, bt.shape[1], NB, rp, nr)
    if st != 0:
        raise ValueError(f"oracle_chunk_attention failed with status {st}")
    return out
