"""libpagedkv -- paged KV-cache write and paged decode attention for GB300.

Python binding of the C ABI in ``include/pagedkv.h``: every function here has
the C entry point's name and only marshals arguments (torch tensors -> device
pointers, shapes -> sizes, the current torch stream -> cudaStream_t).  All of
the work runs in the CUDA kernels of ``libpagedkv.so``; there is no other
implementation behind these names.  Build the library with
``paged_kv_cache_131_gb300._build.build()`` (or ``__graft_entry__.build()``).
"""

from __future__ import annotations

import ctypes
import os

__all__ = [
    "PkvError", "pkv_view", "pkv_write_desc", "pkv_decode_options", "library_path", "load",
    "pkv_cache_write", "pkv_decode_attention", "pkv_decode_workspace_bytes",
    "pkv_decode_workspace_init", "pkv_get_device_error", "pkv_status_string",
    "pkv_last_error_string", "pkv_version", "EXPORTED_SYMBOLS", "pkv_chunk_attention",
    "pkv_chunk_workspace_bytes",
    "PKV_COMPUTE_AUTO", "PKV_COMPUTE_SIMT", "PKV_COMPUTE_MMA", "PKV_SCHEDULE_AUTO",
    "PKV_SCHEDULE_GRID", "PKV_SCHEDULE_BALANCED", "DEVICE_ERRORS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libpagedkv.so")

PKV_COMPUTE_AUTO, PKV_COMPUTE_SIMT, PKV_COMPUTE_MMA = 0, 1, 2
PKV_SCHEDULE_AUTO, PKV_SCHEDULE_GRID, PKV_SCHEDULE_BALANCED = 0, 1, 2
DEVICE_ERRORS = {0: "none", 1: "slot", 2: "block_id", 3: "seq_len", 4: "timeout"}

EXPORTED_SYMBOLS = [
    "pkv_cache_write", "pkv_decode_attention", "pkv_decode_attention_ex",
    "pkv_decode_workspace_bytes", "pkv_decode_workspace_bytes_ex", "pkv_decode_workspace_init",
    "pkv_get_device_error", "pkv_status_string", "pkv_last_error_string", "pkv_version",
    "pkv_decode_attention_noalloc", "pkv_cache_write_multi", "pkv_copy_blocks",
    "pkv_cache_write_fp8", "pkv_decode_attention_fp8", "pkv_chunk_attention",
    "pkv_chunk_workspace_bytes",
]


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = pkv_status_string(status)
        if status == -6:
            msg += f" [{pkv_last_error_string()}]"
        super().__init__(f"{where}: {msg}")
        self.status = status


class pkv_view(ctypes.Structure):
    _fields_ = [("offset", ctypes.c_int64), ("layer_stride", ctypes.c_int64),
                ("block_stride", ctypes.c_int64), ("row_width", ctypes.c_int64),
                ("layer", ctypes.c_int32)]


class pkv_write_desc(ctypes.Structure):
    _fields_ = [("src", ctypes.c_void_p), ("cache", ctypes.c_void_p), ("view", pkv_view)]


class pkv_decode_options(ctypes.Structure):
    _fields_ = [("partition_size", ctypes.c_int32), ("compute", ctypes.c_int32),
                ("schedule", ctypes.c_int32)]


_lib = None
_i32, _i64, _p, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t


def load(path: str | None = None):
    """Load libpagedkv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or library_path
    if not os.path.exists(path):
        raise ImportError(f"libpagedkv.so is not built ({path}); run "
                          "paged_kv_cache_131_gb300._build.build()")
    lib = ctypes.CDLL(path)
    lib.pkv_cache_write.restype = ctypes.c_int
    lib.pkv_cache_write.argtypes = [_p, _p, _p, _i64, _p, _p, pkv_view, _i32, _i64, _p]
    lib.pkv_cache_write_multi.restype = ctypes.c_int
    lib.pkv_cache_write_multi.argtypes = [ctypes.POINTER(pkv_write_desc), _i32, _p, _i64, _i32,
                                          _i64, _p]
    lib.pkv_cache_write_fp8.restype = ctypes.c_int
    lib.pkv_cache_write_fp8.argtypes = [_p, _p, _p, _i64, _p, _p, _p, _p, _i32, _i32, _i32, _i64,
                                        _p]
    lib.pkv_copy_blocks.restype = ctypes.c_int
    lib.pkv_copy_blocks.argtypes = [_p, pkv_view, _i32, _i32, _p, _i64, _i64, _p]
    dec = [_p, _p, _p, _p, _p, _p, ctypes.c_float, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
           _i64, _p, _sz]
    lib.pkv_decode_attention.restype = ctypes.c_int
    lib.pkv_decode_attention.argtypes = dec + [_p]
    lib.pkv_decode_attention_ex.restype = ctypes.c_int
    lib.pkv_decode_attention_ex.argtypes = dec + [ctypes.POINTER(pkv_decode_options), _p]
    lib.pkv_decode_attention_fp8.restype = ctypes.c_int
    lib.pkv_decode_attention_fp8.argtypes = dec[:4] + [_p, _p] + dec[4:] + [_p]
    lib.pkv_decode_attention_noalloc.restype = ctypes.c_int
    lib.pkv_decode_attention_noalloc.argtypes = dec[:15] + [_p]
    lib.pkv_chunk_attention.restype = ctypes.c_int
    lib.pkv_chunk_attention.argtypes = [_p, _p, _p, _p, _p, _p, _p, ctypes.c_float, _i32, _i32,
                                        _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i64, _p, _sz,
                                        _p]
    lib.pkv_chunk_workspace_bytes.restype = _sz
    lib.pkv_chunk_workspace_bytes.argtypes = [_i32] * 7
    lib.pkv_decode_workspace_bytes.restype = _sz
    lib.pkv_decode_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32]
    lib.pkv_decode_workspace_bytes_ex.restype = _sz
    lib.pkv_decode_workspace_bytes_ex.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
    lib.pkv_decode_workspace_init.restype = ctypes.c_int
    lib.pkv_decode_workspace_init.argtypes = [_p, _sz, _p]
    lib.pkv_get_device_error.restype = ctypes.c_int
    lib.pkv_get_device_error.argtypes = [ctypes.POINTER(_i32), ctypes.POINTER(_i64), _p]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    lib.pkv_last_error_string.restype = ctypes.c_char_p
    lib.pkv_last_error_string.argtypes = []
    lib.pkv_version.restype = ctypes.c_int
    lib.pkv_version.argtypes = []
    if path == library_path:
        _lib = lib
    return lib


# ------------------------------------------------------------------ marshalling


def _dev(t, name, dtype=None):
    """Device pointer of a CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _check(status: int, where: str) -> int:
    if status != 0:
        raise PkvError(status, where)
    return status


def pkv_cache_write(k, v, slot_mapping, k_cache, v_cache, view, block_size: int,
                    num_blocks: int, stream=None, check: bool = True) -> int:
    """Scatter ``k`` (and ``v``) rows to their slots: see pkv_cache_write in pagedkv.h.

    k, v: CUDA tensors of num_tokens rows of ``view.row_width`` bytes; slot_mapping:
    CUDA int64 [num_tokens]; caches: CUDA tensors (any dtype, used as bytes);
    view: pkv_view or an object with offset/layer_stride/block_stride/row_width
    (and optionally layer).
    """
    import torch
    if not isinstance(view, pkv_view):
        view = pkv_view(view.offset, view.layer_stride, view.block_stride, view.row_width,
                        getattr(view, "layer", 0))
    n = slot_mapping.numel()
    if k.numel() * k.element_size() != n * view.row_width:
        raise ValueError("k must hold num_tokens rows of view.row_width bytes")
    if v is not None and v.numel() * v.element_size() != n * view.row_width:
        raise ValueError("v must hold num_tokens rows of view.row_width bytes")
    st = load().pkv_cache_write(
        _dev(k, "k"), _dev(v, "v"), _dev(slot_mapping, "slot_mapping", torch.int64), n,
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), view, block_size, num_blocks,
        _stream(stream))
    return _check(st, "pkv_cache_write") if check else st


def _as_view(view) -> pkv_view:
    if isinstance(view, pkv_view):
        return view
    return pkv_view(view.offset, view.layer_stride, view.block_stride, view.row_width,
                    getattr(view, "layer", 0))


def pkv_cache_write_multi(writes, slot_mapping, block_size: int, num_blocks: int, stream=None,
                          check: bool = True) -> int:
    """One launch for several writes sharing ``slot_mapping``: see pkv_cache_write_multi.

    writes: sequence of (src, cache, view) with CUDA tensors and pkv_view-like views.
    """
    import torch
    n = slot_mapping.numel()
    arr = (pkv_write_desc * max(1, len(writes)))()
    for i, (src, cache, view) in enumerate(writes):
        view = _as_view(view)
        if src.numel() * src.element_size() != n * view.row_width:
            raise ValueError(f"write {i}: src must hold num_tokens rows of row_width bytes")
        arr[i] = pkv_write_desc(_dev(src, f"writes[{i}].src"), _dev(cache, f"writes[{i}].cache"),
                                view)
    st = load().pkv_cache_write_multi(arr, len(writes),
                                      _dev(slot_mapping, "slot_mapping", torch.int64), n,
                                      block_size, num_blocks, _stream(stream))
    return _check(st, "pkv_cache_write_multi") if check else st


def pkv_copy_blocks(cache, view, num_layers: int, block_size: int, block_mapping,
                    num_blocks: int, stream=None, check: bool = True) -> int:
    """Copy whole blocks of a view for each (src, dst) row of ``block_mapping``
    (CUDA int64 [N, 2]): see pkv_copy_blocks in pagedkv.h."""
    import torch
    st = load().pkv_copy_blocks(_dev(cache, "cache"), _as_view(view), num_layers, block_size,
                                _dev(block_mapping, "block_mapping", torch.int64),
                                block_mapping.numel() // 2, num_blocks, _stream(stream))
    return _check(st, "pkv_copy_blocks") if check else st


def pkv_decode_attention(out, q, k_cache, v_cache, block_tables, seq_lens, scale: float,
                         num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                         max_seq_len: int, num_blocks: int, workspace=None, stream=None,
                         partition_size: int = 0, compute: int = PKV_COMPUTE_AUTO,
                         schedule: int = PKV_SCHEDULE_AUTO, check: bool = True) -> int:
    """Paged decode attention: see pkv_decode_attention(_ex) in pagedkv.h.

    out, q: CUDA fp16 [S, H, D]; caches: CUDA fp16 [NB, bs, Hk, D];
    block_tables: CUDA int32 [S, MB]; seq_lens: CUDA int32 [S];
    workspace: CUDA uint8 tensor (zero-filled before first use) or None.
    """
    import torch
    S = q.shape[0]
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have q's shape")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    args = (_dev(out, "out", torch.float16), _dev(q, "q", torch.float16),
            _dev(k_cache, "k_cache", torch.float16), _dev(v_cache, "v_cache", torch.float16),
            _dev(block_tables, "block_tables", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
            float(scale), num_heads, num_kv_heads, head_dim, block_size, S,
            block_tables.shape[1] if block_tables.dim() == 2 else 0, int(max_seq_len),
            int(num_blocks), ws_ptr, ws_bytes)
    lib = load()
    if partition_size == 0 and compute == PKV_COMPUTE_AUTO and schedule == PKV_SCHEDULE_AUTO:
        st = lib.pkv_decode_attention(*args, _stream(stream))
    else:
        opts = pkv_decode_options(partition_size, compute, schedule)
        st = lib.pkv_decode_attention_ex(*args, ctypes.byref(opts), _stream(stream))
    return _check(st, "pkv_decode_attention") if check else st


def pkv_chunk_attention(out, q, k_cache, v_cache, block_tables, seq_lens, query_start,
                        scale: float, num_heads: int, num_kv_heads: int, head_dim: int,
                        block_size: int, max_query_len: int, max_seq_len: int, num_blocks: int,
                        workspace=None, stream=None, check: bool = True) -> int:
    """Causal attention of each sequence's new tokens: see pkv_chunk_attention in
    pagedkv.h.

    out, q: CUDA fp16 [Tq, H, D]; caches: CUDA fp16 [NB, bs, Hk, D];
    block_tables: CUDA int32 [S, MB]; seq_lens: CUDA int32 [S];
    query_start: CUDA int32 [S + 1]; workspace: CUDA uint8 tensor (zero-filled
    before first use).
    """
    import torch
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have q's shape")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    S = seq_lens.numel()
    st = load().pkv_chunk_attention(
        _dev(out, "out", torch.float16), _dev(q, "q", torch.float16),
        _dev(k_cache, "k_cache", torch.float16), _dev(v_cache, "v_cache", torch.float16),
        _dev(block_tables, "block_tables", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        _dev(query_start, "query_start", torch.int32), float(scale), num_heads, num_kv_heads,
        head_dim, block_size, S, block_tables.shape[1] if block_tables.dim() == 2 else 0,
        q.shape[0], int(max_query_len), int(max_seq_len), int(num_blocks), ws_ptr, ws_bytes,
        _stream(stream))
    return _check(st, "pkv_chunk_attention") if check else st


def pkv_chunk_workspace_bytes(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                              num_query_tokens: int, max_query_len: int, max_seq_len: int) -> int:
    return load().pkv_chunk_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim,
                                            num_query_tokens, max_query_len, max_seq_len)


def pkv_cache_write_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, block_size: int,
                        num_blocks: int, stream=None, check: bool = True) -> int:
    """Quantize-on-write of fp16 rows k, v [T, Hk, D] into E4M3 caches
    (uint8 [NB, bs, Hk, D]) and fp32 scales [NB, bs, Hk]: see pagedkv.h."""
    import torch
    NB, bs, Hk, D = k_cache.shape
    st = load().pkv_cache_write_fp8(
        _dev(k, "k", torch.float16), _dev(v, "v", torch.float16),
        _dev(slot_mapping, "slot_mapping", torch.int64), slot_mapping.numel(),
        _dev(k_cache, "k_cache", torch.uint8), _dev(v_cache, "v_cache", torch.uint8),
        _dev(k_scale, "k_scale", torch.float32), _dev(v_scale, "v_scale", torch.float32),
        Hk, D, block_size, num_blocks, _stream(stream))
    return _check(st, "pkv_cache_write_fp8") if check else st


def pkv_decode_attention_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens,
                             scale: float, num_heads: int, num_kv_heads: int, head_dim: int,
                             block_size: int, max_seq_len: int, num_blocks: int, workspace,
                             stream=None, check: bool = True) -> int:
    """Paged decode attention over E4M3 caches: see pkv_decode_attention_fp8."""
    import torch
    st = load().pkv_decode_attention_fp8(
        _dev(out, "out", torch.float16), _dev(q, "q", torch.float16),
        _dev(k_cache, "k_cache", torch.uint8), _dev(v_cache, "v_cache", torch.uint8),
        _dev(k_scale, "k_scale", torch.float32), _dev(v_scale, "v_scale", torch.float32),
        _dev(block_tables, "block_tables", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        float(scale), num_heads, num_kv_heads, head_dim, block_size, q.shape[0],
        block_tables.shape[1], int(max_seq_len), int(num_blocks), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    return _check(st, "pkv_decode_attention_fp8") if check else st


def pkv_decode_workspace_bytes(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                               max_seq_len: int, partition_size: int = 0) -> int:
    return int(load().pkv_decode_workspace_bytes_ex(num_seqs, num_heads, num_kv_heads, head_dim,
                                                    max_seq_len, partition_size))


def pkv_decode_workspace_init(workspace, stream=None) -> int:
    if workspace is None:
        return 0
    return _check(load().pkv_decode_workspace_init(
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)), "pkv_decode_workspace_init")


def pkv_get_device_error(stream=None) -> tuple[int, int]:
    """Synchronise ``stream``; return and clear (kind, index) of the device error record."""
    kind, index = _i32(0), _i64(-1)
    _check(load().pkv_get_device_error(ctypes.byref(kind), ctypes.byref(index), _stream(stream)),
           "pkv_get_device_error")
    return kind.value, index.value


def pkv_status_string(status: int) -> str:
    return load().pkv_status_string(status).decode()


def pkv_last_error_string() -> str:
    return load().pkv_last_error_string().decode()


def pkv_version() -> int:
    return load().pkv_version()
