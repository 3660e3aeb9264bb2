"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, and rejects bad arguments on the host before any CUDA call."""

import ctypes
import os
import re

import pytest

import paged_kv_cache_131_gb300 as pkv
from paged_kv_cache_131_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "pagedkv.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pkv_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pkv_cache_write", "pkv_decode_attention", "pkv_decode_workspace_bytes",
                     "pkv_get_device_error", "pkv_status_string"):
        assert required in names
    assert sorted(pkv.EXPORTED_SYMBOLS) == names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings_and_version(lib):
    for st in range(0, -7, -1):
        s = pkv.pkv_status_string(st)
        assert s.startswith("PKV_")
    assert "unknown" in pkv.pkv_status_string(42)
    assert pkv.pkv_version() >= 10000


FAKE = 0x100000  # 16-byte aligned, never dereferenced: every call below fails validation


def _write(lib, k=FAKE, v=FAKE, slots=FAKE, T=4, kc=FAKE, vc=FAKE, view=None, bs=16, nb=8):
    view = view or pkv.pkv_view(0, 0, 16 * 64, 64, 0)
    return lib.pkv_cache_write(k, v, slots, T, kc, vc, view, bs, nb, None)


def test_write_validation(lib):
    assert _write(lib, T=-1) == -2
    assert _write(lib, k=None) == -1
    assert _write(lib, slots=None) == -1
    assert _write(lib, kc=None) == -1
    assert _write(lib, v=None) == -1  # v_cache given without v
    assert _write(lib, vc=None) == -1
    assert _write(lib, bs=0) == -2
    assert _write(lib, nb=0) == -2
    assert _write(lib, view=pkv.pkv_view(0, 0, 0, 64, 0)) == -2
    assert _write(lib, view=pkv.pkv_view(0, 0, 64, 0, 0)) == -2
    assert _write(lib, view=pkv.pkv_view(-16, 0, 64, 64, 0)) == -2
    assert _write(lib, view=pkv.pkv_view(0, 16, 64, 64, -1)) == -2
    assert _write(lib, slots=FAKE + 4) == -4  # int64 slot_mapping must be 8-byte aligned
    assert _write(lib, T=0) == 0  # nothing to do, nothing launched


def _decode(lib, **kw):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, scale=0.125, H=32, Hk=8, D=128,
             bs=16, S=4, MB=64, maxL=128, NB=64, ws=None, wsb=0, opts=None)
    a.update(kw)
    opts = None if a["opts"] is None else ctypes.byref(pkv.pkv_decode_options(*a["opts"]))
    return lib.pkv_decode_attention_ex(a["out"], a["q"], a["k"], a["v"], a["bt"], a["sl"],
                                       a["scale"], a["H"], a["Hk"], a["D"], a["bs"], a["S"],
                                       a["MB"], a["maxL"], a["NB"], a["ws"], a["wsb"], opts, None)


def test_decode_validation(lib):
    assert _decode(lib, S=-1) == -2
    assert _decode(lib, S=0) == 0
    for key in ("out", "q", "k", "v", "bt", "sl"):
        assert _decode(lib, **{key: None}) == -1, key
    assert _decode(lib, H=30) == -2           # not a multiple of Hk
    assert _decode(lib, H=24, Hk=8) == -3     # group 3 not built
    assert _decode(lib, H=128, Hk=8) == -3    # group 16 not built
    assert _decode(lib, D=96) == -3
    assert _decode(lib, bs=32) == -3
    assert _decode(lib, bs=0) == -2
    assert _decode(lib, MB=0) == -2
    assert _decode(lib, NB=0) == -2
    assert _decode(lib, maxL=-1) == -2
    assert _decode(lib, scale=float("nan")) == -2
    assert _decode(lib, opts=(24, 0, 0)) == -2   # partition not a multiple of 16
    assert _decode(lib, opts=(16384, 0, 0)) == -2
    assert _decode(lib, opts=(512, 7, 0)) == -2  # unknown compute path
    assert _decode(lib, opts=(512, 0, 3)) == -2  # unknown schedule
    assert _decode(lib, q=FAKE + 8) == -4
    assert _decode(lib, k=FAKE + 2) == -4
    assert _decode(lib, maxL=513, ws=FAKE + 8, wsb=1 << 30) == -4
    # grid schedule: two partitions need a workspace
    grid = (0, 0, 1)
    assert _decode(lib, maxL=513, opts=grid) == -5
    need_grid = pkv.load().pkv_decode_workspace_bytes_ex(4, 32, 8, 128, 513, 0)
    a256 = lambda x: (x + 255) // 256 * 256
    grid_bytes = a256(4 * 32 * 4) + a256(4 * 32 * 2 * 8) + 4 * 32 * 2 * 128 * 4
    assert need_grid >= grid_bytes
    assert _decode(lib, maxL=513, ws=FAKE, wsb=grid_bytes - 1, opts=grid) == -5
    # balanced schedule: always needs its workspace; a sequence count whose
    # per-sequence tables overflow its shared memory is unsupported
    bal = (0, 0, 2)
    assert _decode(lib, opts=bal) == -5
    assert _decode(lib, ws=FAKE, wsb=need_grid - 1, opts=bal) == -5 or need_grid == grid_bytes
    assert _decode(lib, S=28000, ws=FAKE, wsb=1 << 30, opts=bal) == -3


def _chunk(lib, out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, qs=FAKE, scale=0.1, H=32,
           Hk=8, D=128, bs=16, S=4, MB=8, Tq=10, maxq=7, maxL=100, NB=64, ws=None, wsb=0):
    return lib.pkv_chunk_attention(out, q, k, v, bt, sl, qs, scale, H, Hk, D, bs, S, MB, Tq,
                                   maxq, maxL, NB, ws, wsb, None)


def test_chunk_validation(lib):
    # every case is refused (or a no-op) on the host, before any CUDA call
    assert _chunk(lib, S=-1) == -2
    assert _chunk(lib, Tq=-1) == -2
    assert _chunk(lib, S=0) == 0 and _chunk(lib, Tq=0) == 0
    for key in ("out", "q", "k", "v", "bt", "sl", "qs"):
        assert _chunk(lib, **{key: None}) == -1, key
    assert _chunk(lib, H=30) == -2
    assert _chunk(lib, H=24, Hk=8) == -3
    assert _chunk(lib, D=96) == -3
    assert _chunk(lib, bs=32) == -3
    assert _chunk(lib, maxq=0) == -2
    assert _chunk(lib, maxL=0) == -2
    assert _chunk(lib, MB=0) == -2
    assert _chunk(lib, NB=0) == -2
    assert _chunk(lib, scale=float("inf")) == -2
    assert _chunk(lib, q=FAKE + 8) == -4
    assert _chunk(lib, qs=FAKE + 2) == -4
    assert _chunk(lib) == -5                      # no workspace
    need = lib.pkv_chunk_workspace_bytes(4, 32, 8, 128, 10, 7, 100)
    assert need > 0
    assert _chunk(lib, ws=FAKE, wsb=need - 1) == -5


def test_chunk_workspace_bytes(lib):
    def a256(x):
        return (x + 255) // 256 * 256

    assert lib.pkv_chunk_workspace_bytes(4, 30, 8, 128, 10, 7, 100) == 0
    assert lib.pkv_chunk_workspace_bytes(4, 32, 8, 128, 10, 0, 100) == 0
    # the balanced schedule's scratch (short chunks: tickets + partial rows of
    # up to 16 query columns) comes first, then the tile kernel's: the work
    # list, a ticket per (sequence, KV head, 128-row tile, softmax warp) and,
    # past one 4096-token partition, partial states of every query row (two
    # copies of (m, l), one O)
    S, H, Hk, D = 4, 32, 8, 128
    one = lib.pkv_chunk_workspace_bytes(S, H, Hk, D, 10, 7, 4096)
    assert one >= a256(S * Hk * 1 * 8 * 4) + a256(S * Hk * 4) + 2 * Hk * 16 * (8 + 4 * D)
    # 952 new tokens x 4 heads per KV head = 30 tiles; 5000 tokens = 2 partitions
    Tq, P, tiles = 1015, 2, 30
    big = lib.pkv_chunk_workspace_bytes(64, H, Hk, D, Tq, 952, 5000)
    assert big >= (a256(64 * Hk * tiles * 8 * 4) + a256(2 * P * Tq * H * 8) +
                   P * Tq * H * D * 4)


def test_workspace_bytes(lib):
    def a256(x):
        return (x + 255) // 256 * 256

    assert pkv.pkv_decode_workspace_bytes(64, 32, 8, 128, 0) == 0
    assert pkv.pkv_decode_workspace_bytes(64, 30, 8, 128, 100) == 0  # H not a multiple of Hk
    # the larger of the grid schedule's partials (one per 512-token partition)
    # and the balanced schedule's (two per CTA; one CTA per SM for this shape)
    S, H, Hk, D, L = 64, 32, 8, 128, 4096
    grid = a256(S * H * 4) + a256(S * H * 8 * 8) + S * H * 8 * D * 4
    got = pkv.pkv_decode_workspace_bytes(S, H, Hk, D, L)
    assert got >= grid
    G = H // Hk
    per_cta = 2 * Hk * G * (8 + D * 4)
    assert (got - a256(S * Hk * 4)) >= per_cta  # room for at least one CTA's partials
    assert pkv.pkv_decode_workspace_bytes(8, 32, 8, 128, 32768, 1024) >= \
        a256(8 * 32 * 4) + a256(8 * 32 * 32 * 8) + 8 * 32 * 32 * 128 * 4


def test_binding_rejects_host_tensors(lib):
    torch = pytest.importorskip("torch")
    t = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError):
        pkv.pkv_cache_write(torch.zeros(4, 64, dtype=torch.uint8), None, t,
                            torch.zeros(1024, dtype=torch.uint8), None,
                            pkv.pkv_view(0, 0, 256, 64, 0), 4, 4)
