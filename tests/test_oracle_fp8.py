"""Pins of the oracle's FP8 (E4M3) pieces (CPU only): the code table and the
rounding against torch's float8_e4m3fn conversion (an independent library
routine), the quantizer's closed-form properties, and FP8 decode reducing to
the pinned fp16 oracle when the dequantized values are exact in fp16."""

import numpy as np
import pytest

from paged_kv_cache_131_gb300 import workloads as W

torch = pytest.importorskip("torch")


def _torch_value(codes):
    return torch.tensor(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()


def _torch_encode(ys):
    return torch.tensor(np.asarray(ys, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_e4m3_code_table(orc, lib=None):
    codes = np.arange(256)
    ref = _torch_value(codes)
    got = np.array([orc.e4m3_value(c, lib=lib) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.isnan(got[[0x7F, 0xFF]]).all() and np.isnan(got).sum() == 2
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert orc.e4m3_value(0x7E, lib=lib) == 448.0 and orc.e4m3_value(1, lib=lib) == 2.0 ** -9


def test_e4m3_rounding_matches_library(orc, lib=None):
    vals = np.array([orc.e4m3_value(c) for c in range(127)])  # non-negative finite
    mids = (vals[:-1] + vals[1:]) / 2  # exact ties
    rng = np.random.default_rng(5)
    ys = np.concatenate([vals, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                         rng.uniform(-448, 448, 5000), rng.uniform(-1, 1, 2000),
                         rng.uniform(-2 ** -6, 2 ** -6, 2000)]).astype(np.float32)
    ys = np.concatenate([ys, -ys])
    got = np.array([orc.e4m3_encode(float(y), lib=lib) for y in ys], dtype=np.uint8)
    assert np.array_equal(got, _torch_encode(ys))


def test_e4m3_saturation_and_specials(orc, lib=None):
    assert orc.e4m3_encode(448.0, lib=lib) == 0x7E
    assert orc.e4m3_encode(463.9, lib=lib) == 0x7E
    assert orc.e4m3_encode(1e30, lib=lib) == 0x7E
    assert orc.e4m3_encode(-1e30, lib=lib) == 0xFE
    assert orc.e4m3_encode(float("nan"), lib=lib) == 0x7F
    assert orc.e4m3_encode(-0.0, lib=lib) == 0x80 and orc.e4m3_encode(0.0, lib=lib) == 0


def test_quantize_row_properties(orc, lib=None):
    rng = np.random.default_rng(6)
    for _ in range(50):
        x = W.fp16_normal(rng, (128,)) * np.float16(rng.uniform(0.01, 30))
        codes, s = orc.quantize_row(x, lib=lib)
        xf = x.astype(np.float64)
        amax = np.float32(np.abs(x.astype(np.float32)).max())
        assert s == np.float32(amax / np.float32(448))
        # the largest magnitude lands on +-448
        i = int(np.argmax(np.abs(xf)))
        assert codes[i] & 0x7F == 0x7E
        # every element is the nearest code to x / s (3 mantissa bits: relative
        # error <= 1/16 for normal codes, absolute <= 2^-10 s below them)
        deq = np.array([orc.e4m3_value(c) for c in codes]) * np.float64(s)
        bound = np.maximum(np.abs(xf) / 16, 2.0 ** -10 * s) * (1 + 1e-6)
        assert (np.abs(deq - xf) <= bound).all()
    codes, s = orc.quantize_row(np.zeros(64, np.float16), lib=lib)
    assert s == 0.0 and not codes.any()


def test_cache_write_fp8_rows_and_untouched(orc, lib=None):
    rng = np.random.default_rng(7)
    NB, bs, Hk, D = 6, 16, 2, 64
    cache = np.full((NB, bs, Hk, D), 0x7F, np.uint8)
    scales = np.full((NB, bs, Hk), np.nan, np.float32)
    slots = np.array([3, -1, 40, 95], dtype=np.int64)
    src = W.fp16_normal(rng, (4, Hk, D))
    n = orc.cache_write_fp8(cache, scales, src, slots, block_size=bs, lib=lib)
    assert n == 3 * Hk
    for t, sl in enumerate(slots):
        if sl < 0:
            continue
        b, o = divmod(int(sl), bs)
        for h in range(Hk):
            codes, s = orc.quantize_row(src[t, h], lib=lib)
            assert np.array_equal(cache[b, o, h], codes) and scales[b, o, h] == np.float32(s)
    written = {int(s) for s in slots if s >= 0}
    for s in range(NB * bs):
        if s not in written:
            b, o = divmod(s, bs)
            assert (cache[b, o] == 0x7F).all() and np.isnan(scales[b, o]).all()


def test_decode_fp8_reduces_to_fp16_oracle(orc, lib=None):
    """With power-of-two scales every dequantized value is exact in fp16, so
    FP8 decode must equal the (pinned) fp16 decode on those values exactly."""
    rng = np.random.default_rng(8)
    wl = W.small_decode(405, [5, 16, 40, 71], H=8, Hk=2, D=64, write_last=False)
    NB, bs, Hk, D = wl.k_cache.shape
    k8 = rng.integers(0, 256, size=(NB, bs, Hk, D), dtype=np.uint8)
    v8 = rng.integers(0, 256, size=(NB, bs, Hk, D), dtype=np.uint8)
    k8[(k8 & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    v8[(v8 & 0x7F) == 0x7F] = 0x41
    ks = (2.0 ** rng.integers(-6, -2, size=(NB, bs, Hk))).astype(np.float32)
    vs = (2.0 ** rng.integers(-6, -2, size=(NB, bs, Hk))).astype(np.float32)
    k16 = (_torch_value(k8.reshape(-1)).reshape(k8.shape) * ks[..., None]).astype(np.float16)
    v16 = (_torch_value(v8.reshape(-1)).reshape(v8.shape) * vs[..., None]).astype(np.float16)
    assert np.array_equal(k16.astype(np.float64),
                          _torch_value(k8.reshape(-1)).reshape(k8.shape) * ks[..., None])
    got = orc.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.seq_lens, wl.scale,
                                   lib=lib)
    ref = orc.decode_attention(wl.q, k16, v16, wl.block_tables, wl.seq_lens, wl.scale)
    assert np.array_equal(got, ref)
