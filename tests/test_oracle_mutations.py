"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pins of test_oracle_pins.py catch every one of them.

Each mutation is a textual edit of oracle/pkv_oracle.c compiled into a
throw-away shared library; the committed oracle is never modified.
"""

import os
import subprocess

import pytest

import oracle
import test_oracle_chunk as C
import test_oracle_fp8 as F
import test_oracle_pins as P
from paged_kv_cache_131_gb300 import workloads as W

SRC = os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")

MUTATIONS = {
    "in-block position taken with /":
        ("*in_block = slot % block_size;", "*in_block = slot / block_size;"),
    "block taken with %":
        ("*block = slot / block_size;", "*block = slot % block_size;"),
    "layer term dropped":
        ("offset + layer * layer_stride + block * block_stride",
         "offset + block * block_stride"),
    "block size used as row width":
        ("in_block * row_width;", "in_block * block_size;"),
    "fp16 exponent bias off by one":
        ("expo - 25", "expo - 24"),
    "fp16 subnormal scale wrong":
        ("ldexp((double)frac, -24)", "ldexp((double)frac, -25)"),
    "GQA heads interleaved instead of consecutive":
        ("int64_t h = kvh * group + g;", "int64_t h = g * num_kv_heads + kvh;"),
    "scale not applied":
        ("s *= scale;", "s *= 1.0;"),
    "softmax not normalised":
        ("out[d] /= denom;", "out[d] /= 1.0;"),
    "softmax exponent sign flipped":
        ("double e = exp(scores[j] - m);", "double e = exp(m - scores[j]);"),
    "cache read head-major instead of token-major":
        ("((block * block_size + in_block) * num_kv_heads + kv_head) * head_dim + d",
         "((block * num_kv_heads + kv_head) * block_size + in_block) * head_dim + d"),
    "block table indexed with %":
        ("int64_t logical = j / block_size;", "int64_t logical = j % block_size;"),
    "gathered position taken with /":
        ("int64_t in_block = j % block_size;", "int64_t in_block = j / block_size;"),
    "keys and values swapped":
        ("cache_at(v_cache, phys", "cache_at(k_cache, phys"),
    "query and key head index transposed":
        ("q[(i * num_heads + h) * head_dim + d]", "q[(h * num_seqs + i) * head_dim + d]"),
    "negative slots not skipped":
        ("if (slot < 0)\n            continue;", "if (slot < -1000)\n            continue;"),
    "copy on write copies the wrong way":
        ("memcpy(cache + b, cache + a, (size_t)page);", "memcpy(cache + a, cache + b, (size_t)page);"),
    "E4M3 exponent bias off by one":
        ("ldexp((double)(8 + mant), expo - 10)", "ldexp((double)(8 + mant), expo - 9)"),
    "E4M3 subnormal scale wrong":
        ("mag = ldexp((double)mant, -9);", "mag = ldexp((double)mant, -8);"),
    "E4M3 ties to odd":
        ("(above == below && ((lo + 1) & 1) == 0)", "(above == below && ((lo + 1) & 1) == 1)"),
    "E4M3 rounds down always":
        ("if (above < below ||", "if (0 &&"),
    "FP8 scale for a 240 maximum":
        ("float s = amax / 448.0f;", "float s = amax / 240.0f;"),
    "FP8 quantizer multiplies by the scale":
        ("oracle_e4m3_encode(xi / s)", "oracle_e4m3_encode(xi * s)"),
    "FP8 decode ignores the value scale":
        ("oracle_e4m3_value(v_cache[row * head_dim + d]) * (double)v_scale[row]",
         "oracle_e4m3_value(v_cache[row * head_dim + d]) * 1.0"),
    "FP8 decode scales values by the key scale":
        ("oracle_e4m3_value(v_cache[row * head_dim + d]) * (double)v_scale[row]",
         "oracle_e4m3_value(v_cache[row * head_dim + d]) * (double)k_scale[row]"),
    "copy on write ignores the layer":
        ("int64_t a = offset + l * layer_stride + src * block_stride;",
         "int64_t a = offset + src * block_stride;"),
    "chunk token attends one key too many":
        ("pos + 1, head_dim, scale, scores);", "pos + 2 <= len ? pos + 2 : len, head_dim, scale, scores);"),
    "chunk token attends one key too few":
        ("pos + 1, head_dim, scale, scores);", "pos > 0 ? pos : 1, head_dim, scale, scores);"),
    "chunk positions counted from the sequence start":
        ("int64_t pos = len - nq + (r - r0);", "int64_t pos = r - r0;"),
    "chunk attention not causal":
        ("pos + 1, head_dim, scale, scores);", "len, head_dim, scale, scores);"),
    "chunk query rows taken in reverse":
        ("int64_t pos = len - nq + (r - r0);", "int64_t pos = len - 1 - (r - r0);"),
}


def _pins(orc, lib):
    small_dsa = W.config5_dsa_write(num_tokens=64, num_blocks=8)
    yield lambda: P.test_half_to_double_exhaustive(orc, lib=lib)
    yield lambda: P.test_slot_mapping_worked_example(orc, lib=lib)
    yield lambda: P.test_dsa_block_outer_addresses(orc, lib=lib)
    yield lambda: P.test_dsa_layer_outer_addresses(orc, lib=lib)
    yield lambda: P.test_write_round_trip_and_untouched(orc, small_dsa, lib=lib)
    yield lambda: P.test_write_negative_slot_skipped_and_range_error(orc, lib=lib)
    yield lambda: P.test_decode_config1_brute_force(orc, lib=lib)
    yield lambda: P.test_decode_special_cases(orc, lib=lib)
    yield lambda: P.test_decode_gqa_equals_mha_with_duplicated_kv(orc, lib=lib)
    yield lambda: P.test_decode_bad_block_id_is_an_error(orc, lib=lib)
    yield lambda: P.test_copy_blocks_pages_only(orc, lib=lib)
    yield lambda: F.test_e4m3_code_table(orc, lib=lib)
    yield lambda: F.test_e4m3_rounding_matches_library(orc, lib=lib)
    yield lambda: F.test_quantize_row_properties(orc, lib=lib)
    yield lambda: F.test_cache_write_fp8_rows_and_untouched(orc, lib=lib)
    yield lambda: F.test_decode_fp8_reduces_to_fp16_oracle(orc, lib=lib)
    yield lambda: C.test_each_new_token_is_a_decode_of_its_prefix(orc, lib=lib)
    yield lambda: C.test_chunk_matches_brute_force(orc, lib=lib)
    for case in (dict(index=102, lens=[3, 20, 40], H=4, Hk=2, D=8),
                 dict(index=103, lens=[0, 2, 31], H=8, Hk=1, D=4)):
        yield lambda case=case: P.test_decode_matches_brute_force(orc, case, lib=lib)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(orc, tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert old in src, f"mutation site for {name!r} not found"
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", str(path), "-o",
                           str(so), "-lm"])
    lib = oracle._load(str(so))
    caught = []
    for pin in _pins(orc, lib):
        try:
            pin()
        except (AssertionError, ValueError):
            caught.append(pin)
            break
    assert caught, f"no pin caught the planted mistake {name!r}"
