"""GPU parity of the FP8 (E4M3) KV path against the oracle: quantize-on-write
bit-exact (codes and scales), and decode over the FP8 caches within the
decode tolerance (|gpu - ref| <= 2e-3 + 1e-2 |ref|) of the oracle's float64
attention on the exactly dequantized values."""

import numpy as np
import pytest

import oracle
from paged_kv_cache_131_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_131_gb300 import _build
    _build.build()
    import paged_kv_cache_131_gb300 as m
    assert torch.cuda.is_available()
    m.pkv_get_device_error()
    return m


def _oracle_fp8_state(wl, seqs=None, workers=1):
    """Oracle caches after quantizing the prior tokens and then the new ones
    (only the rows of `seqs` when given)."""
    from paged_kv_cache_131_gb300.harness import prior_token_rows
    NB, bs, Hk, D = wl.k_cache.shape
    k8 = np.full((NB, bs, Hk, D), 0x7F, np.uint8)
    v8 = np.full((NB, bs, Hk, D), 0x7F, np.uint8)
    ks = np.full((NB, bs, Hk), np.nan, np.float32)
    vs = np.full((NB, bs, Hk), np.nan, np.float32)
    slots, rk, rv = prior_token_rows(wl)
    if seqs is not None:
        mine = {W.slot_of(wl.block_tables[i], p, bs) for i in seqs
                for p in range(int(wl.seq_lens[i]))}
        keep = np.array([s in mine for s in slots.tolist()], dtype=bool)
        slots, rk, rv = slots[keep], rk[keep], rv[keep]
    if slots.size:
        oracle.cache_write_fp8(k8, ks, rk, slots, block_size=bs, workers=workers)
        oracle.cache_write_fp8(v8, vs, rv, slots, block_size=bs, workers=workers)
    if wl.slot_mapping is not None and wl.slot_mapping.size:
        oracle.cache_write_fp8(k8, ks, wl.k_new.reshape(-1, Hk, D), wl.slot_mapping, block_size=bs)
        oracle.cache_write_fp8(v8, vs, wl.v_new.reshape(-1, Hk, D), wl.slot_mapping, block_size=bs)
    return k8, v8, ks, vs


def _same_bits(dev_tensor, ref):
    got = dev_tensor.cpu().numpy()
    return np.array_equal(got.view(np.uint8), np.ascontiguousarray(ref).view(np.uint8))


@pytest.mark.parametrize("Hk,D", [(1, 64), (4, 128), (8, 128), (2, 64)])
def test_fp8_write_bit_exact(pkv, Hk, D):
    rng = np.random.default_rng(31 + Hk + D)
    NB, bs, T = 12, 16, 150
    rows_k = W.fp16_normal(rng, (T, Hk, D))
    rows_v = W.fp16_normal(rng, (T, Hk, D))
    rows_k[::7] *= np.float16(40)          # large rows
    rows_v[3::11] *= np.float16(1e-3)      # small rows (subnormal codes)
    rows_k[5] = 0                          # an all-zero row: scale 0, codes 0
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int64)
    slots[::13] = -1
    dk = torch.full((NB, bs, Hk, D), 0x7F, dtype=torch.uint8, device="cuda")
    dv = torch.full_like(dk, 0x7F)
    dks = torch.full((NB, bs, Hk), float("nan"), dtype=torch.float32, device="cuda")
    dvs = torch.full_like(dks, float("nan"))
    pkv.pkv_cache_write_fp8(torch.from_numpy(rows_k).cuda(), torch.from_numpy(rows_v).cuda(),
                            torch.from_numpy(slots).cuda(), dk, dv, dks, dvs, bs, NB)
    k8 = np.full((NB, bs, Hk, D), 0x7F, np.uint8)
    v8 = np.full_like(k8, 0x7F)
    ks = np.full((NB, bs, Hk), np.nan, np.float32)
    vs = np.full_like(ks, np.nan)
    oracle.cache_write_fp8(k8, ks, rows_k, slots, block_size=bs)
    oracle.cache_write_fp8(v8, vs, rows_v, slots, block_size=bs)
    assert _same_bits(dk, k8) and _same_bits(dv, v8)
    assert _same_bits(dks, ks) and _same_bits(dvs, vs)
    assert pkv.pkv_get_device_error() == (0, -1)


def _close(out, ref, pairs=None):
    g = out.astype(np.float64)
    if pairs is not None:
        idx = tuple(np.array(pairs).T)
        g, ref = g[idx], ref[idx]
    assert np.isfinite(g).all()
    err = np.abs(g - ref)
    assert (err <= ATOL + RTOL * np.abs(ref)).all(), f"max |err| {err.max():.3e}"


@pytest.mark.parametrize("case", [
    dict(index=501, lens=[0, 1, 15, 16, 17, 300, 1100, 2049], H=8, Hk=8, D=128),
    dict(index=502, lens=[5, 47, 999, 1500], H=32, Hk=8, D=128),
    dict(index=503, lens=[3, 64, 700], H=16, Hk=2, D=64),
    dict(index=504, lens=[9, 200, 520], H=8, Hk=1, D=64),
    # more KV heads than a CTA holds: groups of 8, 8 and 2 (64-byte FP8 rows
    # per head: a group must keep whole 128-byte chunks)
    dict(index=505, lens=[1, 33, 1200, 600], H=32, Hk=16, D=128),
    dict(index=506, lens=[700, 17, 2100], H=64, Hk=16, D=64),
    dict(index=507, lens=[250, 999, 5], H=20, Hk=10, D=64),
])
def test_fp8_decode_small(pkv, case):
    from paged_kv_cache_131_gb300.harness import DeviceDecodeFp8
    wl = W.small_decode(case["index"], case["lens"], H=case["H"], Hk=case["Hk"], D=case["D"])
    dev = DeviceDecodeFp8(wl)
    out = dev.step().cpu().numpy()
    assert pkv.pkv_get_device_error() == (0, -1)
    k8, v8, ks, vs = _oracle_fp8_state(wl)
    assert _same_bits(dev.k_cache, k8) and _same_bits(dev.v_scale, vs)
    ref = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.seq_lens,
                                      wl.scale)
    _close(out, ref)


@pytest.mark.parametrize("cfg", [2, 3])
def test_fp8_full_size_all_elements(pkv, cfg):
    """The Llama-8B decode layer and the long-context workload on FP8 caches:
    every code and scale the decode reads is bit-identical to the oracle's
    quantization, and every output element is within tolerance of the
    oracle's float64 attention over the dequantized caches."""
    from paged_kv_cache_131_gb300.harness import DeviceDecodeFp8
    wl = W.config(cfg)
    dev = DeviceDecodeFp8(wl)
    out = dev.step().cpu().numpy()
    assert pkv.pkv_get_device_error() == (0, -1)
    workers = oracle.default_workers()
    k8, v8, ks, vs = _oracle_fp8_state(wl, workers=workers)
    # every row a sequence reads is bit-identical on both sides
    bs, Hk = wl.block_size, wl.num_kv_heads
    slots = np.unique([W.slot_of(wl.block_tables[i], p, bs) for i in range(wl.num_seqs)
                       for p in range(int(wl.seq_lens[i]))])
    g = lambda t: t.cpu().numpy().reshape(wl.num_blocks * bs, -1)[slots]  # noqa: E731
    assert np.array_equal(g(dev.k_cache), k8.reshape(-1, Hk * wl.head_dim)[slots])
    assert np.array_equal(g(dev.v_cache), v8.reshape(-1, Hk * wl.head_dim)[slots])
    assert np.array_equal(g(dev.k_scale).view(np.uint32), ks.reshape(-1, Hk)[slots].view(np.uint32))
    assert np.array_equal(g(dev.v_scale).view(np.uint32), vs.reshape(-1, Hk)[slots].view(np.uint32))
    ref = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.seq_lens,
                                      wl.scale, workers=workers)
    _close(out, ref)


@pytest.mark.parametrize("S,H,Hk", [(800, 32, 8), (400, 64, 16)])
def test_fp8_many_short_sequences_every_element(pkv, S, H, Hk):
    """Many short sequences, several whole ones in every CTA range and cut
    ones at both ends, so each consumer warp finishes, writes and merges
    many times per launch; Hk 16 adds a second head group.  Every element
    against the oracle, two calls in a row."""
    from paged_kv_cache_131_gb300.harness import DeviceDecodeFp8
    lens = [17 + (53 * i) % 250 for i in range(S)]
    wl = W.small_decode(509 + Hk, lens, H=H, Hk=Hk, D=128)
    dev = DeviceDecodeFp8(wl)
    dev.write()
    k8, v8, ks, vs = _oracle_fp8_state(wl, workers=oracle.default_workers())
    ref = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.seq_lens,
                                      wl.scale, workers=oracle.default_workers())
    for _ in range(2):
        dev.out.fill_(float("nan"))
        _close(dev.decode().cpu().numpy(), ref)
    assert pkv.pkv_get_device_error() == (0, -1)


def test_fp8_repeated_calls_every_element(pkv):
    """FP8 decode, calls in a row on one workspace: every call within
    tolerance of the oracle (outputs poisoned before each call)."""
    from paged_kv_cache_131_gb300.harness import DeviceDecodeFp8
    wl = W.small_decode(508, [3000 + 41 * i for i in range(16)], H=32, Hk=8, D=128)
    dev = DeviceDecodeFp8(wl)
    dev.write()
    k8, v8, ks, vs = _oracle_fp8_state(wl, workers=oracle.default_workers())
    ref = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.seq_lens,
                                      wl.scale, workers=oracle.default_workers())
    for _ in range(5):
        dev.out.fill_(float("nan"))
        _close(dev.decode().cpu().numpy(), ref)
    assert pkv.pkv_get_device_error() == (0, -1)
