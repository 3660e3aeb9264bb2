/*
 * pkv_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, single-threaded, float64 CPU restatement of the two operations of
 * the PagedAttention hot path, written from the pages' statement of them and
 * used only to check the CUDA library (tests, the smoke check and the CPU
 * baseline of the benchmark).  It shares no code, header, table or helper
 * with the CUDA library; the product path never calls it.
 *
 * Sources (page title -- section):
 *  - "vLLM KV Cache Layout 可视化" -- 核心 (the byte-address formula
 *    address = offset + layer*layer_stride + block*block_stride
 *              + slot_in_block*row_width),
 *    "查一个 token" (slot_mapping = block * block_size + in-block position) and
 *    "kernel 那一侧" (split the slot back with / and %).
 *  - "deep-dive-into-vllm-05" -- §1.2 (per-layer KV layout
 *    [num_blocks, block_size, num_kv_heads, head_dim], fp16), §2 (the read
 *    loop: for every block of the block table, dot the query with its keys,
 *    softmax over all positions, weighted sum of values), §3.2 (GQA:
 *    consecutive query heads share one KV head).
 *  - "vLLM 技术内幕" -- §2.1 (the query is dotted with the keys of each
 *    physical block in turn and values are accumulated block by block).
 *
 * The attention result is the textbook definition: gather the sequence's
 * blocks into contiguous K and V, then out = sum_j e^{s_j - m} v_j /
 * sum_j e^{s_j - m} with s_j = scale * q.k_j and m = max_j s_j.  The
 * block-wise online softmax of the method reaches this same value (up to
 * rounding order), so the definition is the oracle.
 *
 * Conventions where the pages are silent (each one is stated where it is
 * applied): a negative slot is padding and is skipped; a sequence of length 0
 * yields an all-zero output.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status codes of this file (independent of the library's). */
#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_RANGE (-2)
#define ORC_ERR_NOMEM (-3)

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 -> double, from the format's definition: 1 sign bit,
 * 5 exponent bits with bias 15, 10 fraction bits.  Every binary16 value is
 * exactly representable in binary64. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0) {
        /* zero or subnormal: (frac / 2^10) * 2^(1-15) */
        mag = ldexp((double)frac, -24);
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        /* normal: (1 + frac / 2^10) * 2^(expo-15) */
        mag = ldexp((double)(1024 + frac), expo - 25);
    }
    return sign ? -mag : mag;
}

/* ------------------------------------------------------------------------ */
/* FP8 KV ("deep-dive-into-vllm-05" §3.4: quantize on write, dequantize on
 * read, the scale kept with the block; "vLLM KV Cache Layout 可视化" -- 两种
 * cache: a row of 128 FP8 values carries one FP32 scale).  Format E4M3 as in
 * the OCP 8-bit floating-point specification: 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, largest
 * finite magnitude 448. */

/* Value of an E4M3 code. */
double oracle_e4m3_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 0xf;
    int mant = code & 0x7;
    double mag;
    if (expo == 15 && mant == 7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)mant, -9); /* (mant / 8) * 2^(1-7) */
    else
        mag = ldexp((double)(8 + mant), expo - 10); /* (1 + mant/8) * 2^(expo-7) */
    return sign ? -mag : mag;
}

/* Nearest E4M3 code to y, ties to the even code, magnitudes above 448
 * saturating to 448; NaN gives 0x7F.  The non-negative finite codes 0..126
 * have increasing values, so the nearest one is found by bisection over the
 * codes (each code's value computed from the format as it is needed; no
 * table, no state kept between calls), then the two neighbours are compared
 * (ties -> even code).  A scan of all 127 codes per element gives the same
 * code but is too slow to quantize full-size caches. */
uint8_t oracle_e4m3_encode(float y)
{
    if (isnan(y))
        return 0x7f;
    double a = fabs((double)y);
    if (a > 448.0)
        a = 448.0;
    int lo = 0, hi = 126; /* largest lo with value(lo) <= a */
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (oracle_e4m3_value((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    int best = lo;
    if (lo < 126) {
        double below = a - oracle_e4m3_value((uint8_t)lo);
        double above = oracle_e4m3_value((uint8_t)(lo + 1)) - a;
        if (above < below || (above == below && ((lo + 1) & 1) == 0))
            best = lo + 1;
    }
    return (uint8_t)((signbit(y) ? 0x80 : 0) | best);
}

/* One row of n fp16 values -> n E4M3 codes and one fp32 scale, all in fp32:
 * amax = max |x|, s = amax / 448, code = encode(x / s); s == 0 gives zero
 * codes.  (The pages leave the granularity open; one scale per row of a KV
 * head is our reading, matching the per-token scale of their indexer rows.) */
void oracle_quantize_row(const uint16_t *x, int64_t n, uint8_t *codes, float *scale)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float v = (float)fabs(oracle_half_to_double(x[i]));
        if (v > amax)
            amax = v;
    }
    float s = amax / 448.0f;
    *scale = s;
    for (int64_t i = 0; i < n; ++i) {
        if (s == 0.0f) {
            codes[i] = 0;
        } else {
            float xi = (float)oracle_half_to_double(x[i]);
            codes[i] = oracle_e4m3_encode(xi / s);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* The write side ("vLLM KV Cache Layout 可视化", 核心 and "kernel 那一侧"). */

/* Split a slot back into (physical block, position inside the block). */
void oracle_split_slot(int64_t slot, int64_t block_size, int64_t *block, int64_t *in_block)
{
    *block = slot / block_size;
    *in_block = slot % block_size;
}

/* Byte address of a slot in one view:
 * offset + layer*layer_stride + block*block_stride + in_block*row_width. */
int64_t oracle_slot_address(int64_t slot, int64_t block_size, int64_t offset, int64_t layer,
                            int64_t layer_stride, int64_t block_stride, int64_t row_width)
{
    int64_t block, in_block;
    oracle_split_slot(slot, block_size, &block, &in_block);
    return offset + layer * layer_stride + block * block_stride + in_block * row_width;
}

/* Scatter num_tokens rows of row_width bytes (row t at src + t*row_width)
 * into the cache at the address of slot_mapping[t].  A negative slot is
 * padding and is skipped (our convention).  Bytes that no token addresses
 * keep their prior content.  Returns the number of rows written, or
 * ORC_ERR_RANGE if a row would leave [0, cache_bytes) or a slot is beyond
 * num_blocks*block_size (nothing is written past the first such token). */
int64_t oracle_cache_write(uint8_t *cache, int64_t cache_bytes, const uint8_t *src,
                           const int64_t *slot_mapping, int64_t num_tokens, int64_t offset,
                           int64_t layer, int64_t layer_stride, int64_t block_stride,
                           int64_t row_width, int64_t block_size, int64_t num_blocks)
{
    if (block_size <= 0 || row_width <= 0 || num_tokens < 0)
        return ORC_ERR_ARG;
    int64_t written = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * block_size)
            return ORC_ERR_RANGE;
        int64_t addr = oracle_slot_address(slot, block_size, offset, layer, layer_stride,
                                           block_stride, row_width);
        if (addr < 0 || addr + row_width > cache_bytes)
            return ORC_ERR_RANGE;
        memcpy(cache + addr, src + t * row_width, (size_t)row_width);
        ++written;
    }
    return written;
}

/* Quantize-on-write of fp16 rows [num_tokens][num_kv_heads][head_dim] into
 * an E4M3 cache [num_blocks][block_size][num_kv_heads][head_dim] (bytes)
 * and fp32 scales [num_blocks][block_size][num_kv_heads]: each (token, head)
 * row is quantized by oracle_quantize_row and stored at its slot.  Negative
 * slots are skipped.  Returns rows written or ORC_ERR_RANGE. */
int64_t oracle_cache_write_fp8(uint8_t *cache, float *scales, const uint16_t *src,
                               const int64_t *slot_mapping, int64_t num_tokens,
                               int64_t num_kv_heads, int64_t head_dim, int64_t block_size,
                               int64_t num_blocks)
{
    int64_t written = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * block_size)
            return ORC_ERR_RANGE;
        int64_t block, in_block;
        oracle_split_slot(slot, block_size, &block, &in_block);
        for (int64_t h = 0; h < num_kv_heads; ++h) {
            int64_t row = (block * block_size + in_block) * num_kv_heads + h;
            oracle_quantize_row(src + (t * num_kv_heads + h) * head_dim, head_dim,
                                cache + row * head_dim, scales + row);
            ++written;
        }
    }
    return written;
}

/* Copy on write ("vLLM 技术内幕" §2.2): for each (src, dst) pair and each
 * of num_layers layers starting at `layer`, the page of block_size*row_width
 * bytes of block src is copied to block dst.  src == dst copies nothing.
 * Returns the number of pages copied, or ORC_ERR_RANGE for an id outside
 * [0, num_blocks) or a page outside the cache (nothing after it is copied). */
int64_t oracle_copy_blocks(uint8_t *cache, int64_t cache_bytes, const int64_t *pairs,
                           int64_t num_pairs, int64_t offset, int64_t layer, int64_t num_layers,
                           int64_t layer_stride, int64_t block_stride, int64_t row_width,
                           int64_t block_size, int64_t num_blocks)
{
    int64_t page = block_size * row_width, copied = 0;
    for (int64_t p = 0; p < num_pairs; ++p) {
        int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks)
            return ORC_ERR_RANGE;
        if (src == dst)
            continue;
        for (int64_t l = layer; l < layer + num_layers; ++l) {
            int64_t a = offset + l * layer_stride + src * block_stride;
            int64_t b = offset + l * layer_stride + dst * block_stride;
            if (a < 0 || b < 0 || a + page > cache_bytes || b + page > cache_bytes)
                return ORC_ERR_RANGE;
            memcpy(cache + b, cache + a, (size_t)page);
            ++copied;
        }
    }
    return copied;
}

/* ------------------------------------------------------------------------ */
/* The read side: paged decode attention, one query token per sequence. */

/* Element (block, in_block, kv_head, d) of a [num_blocks, block_size,
 * num_kv_heads, head_dim] fp16 cache ("deep-dive-into-vllm-05" §1.2). */
static double cache_at(const uint16_t *cache, int64_t block, int64_t in_block, int64_t kv_head,
                       int64_t d, int64_t block_size, int64_t num_kv_heads, int64_t head_dim)
{
    int64_t idx = ((block * block_size + in_block) * num_kv_heads + kv_head) * head_dim + d;
    return oracle_half_to_double(cache[idx]);
}

/* Attention for one (sequence, head) over keys/values already gathered into
 * contiguous rows K[len][head_dim], V[len][head_dim]: textbook softmax. */
static void textbook_attention(double *out, const double *q, const double *K, const double *V,
                               int64_t len, int64_t head_dim, double scale, double *scores)
{
    for (int64_t d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    if (len == 0)
        return; /* empty sequence: zeros (our convention) */
    double m = -INFINITY;
    for (int64_t j = 0; j < len; ++j) {
        double s = 0.0;
        for (int64_t d = 0; d < head_dim; ++d)
            s += q[d] * K[j * head_dim + d];
        s *= scale;
        scores[j] = s;
        if (s > m)
            m = s;
    }
    double denom = 0.0;
    for (int64_t j = 0; j < len; ++j) {
        double e = exp(scores[j] - m);
        scores[j] = e;
        denom += e;
    }
    for (int64_t j = 0; j < len; ++j)
        for (int64_t d = 0; d < head_dim; ++d)
            out[d] += scores[j] * V[j * head_dim + d];
    for (int64_t d = 0; d < head_dim; ++d)
        out[d] /= denom;
}

/*
 * out[num_seqs][num_heads][head_dim] (float64) for q[num_seqs][num_heads][head_dim]
 * (fp16 bits), caches [num_blocks][block_size][num_kv_heads][head_dim] (fp16
 * bits), block_tables[num_seqs][max_blocks_per_seq] and seq_lens[num_seqs].
 *
 * Query head h reads KV head h / (num_heads/num_kv_heads) (consecutive heads
 * share a KV head, "deep-dive-into-vllm-05" §3.2).  Position j of sequence i
 * is slot j % block_size of physical block block_tables[i][j / block_size].
 *
 * If `pairs` is non-NULL only the num_pairs (sequence, head) pairs listed in
 * it (pairs[2k], pairs[2k+1]) are computed and written; other outputs are
 * left untouched.  Returns ORC_OK, ORC_ERR_ARG for a bad shape, ORC_ERR_RANGE
 * for a block id outside [0, num_blocks) or a sequence longer than its block
 * table, ORC_ERR_NOMEM if a gather buffer cannot be allocated.
 */
int oracle_decode_attention(double *out, const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *block_tables,
                            const int32_t *seq_lens, double scale, int64_t num_seqs,
                            int64_t num_heads, int64_t num_kv_heads, int64_t head_dim,
                            int64_t block_size, int64_t max_blocks_per_seq, int64_t num_blocks,
                            const int32_t *pairs, int64_t num_pairs)
{
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks_per_seq < 0 || num_seqs < 0)
        return ORC_ERR_ARG;
    int64_t group = num_heads / num_kv_heads;
    int status = ORC_OK;

    for (int64_t i = 0; i < num_seqs && status == ORC_OK; ++i) {
        int64_t len = seq_lens[i];
        if (len < 0 || len > max_blocks_per_seq * block_size)
            return ORC_ERR_RANGE;
        for (int64_t kvh = 0; kvh < num_kv_heads && status == ORC_OK; ++kvh) {
            /* which heads of this KV group are wanted */
            int want_any = 0;
            for (int64_t g = 0; g < group; ++g) {
                int64_t h = kvh * group + g;
                if (!pairs) {
                    want_any = 1;
                } else {
                    for (int64_t p = 0; p < num_pairs; ++p)
                        if (pairs[2 * p] == i && pairs[2 * p + 1] == h)
                            want_any = 1;
                }
            }
            if (!want_any)
                continue;

            /* gather this sequence's blocks into contiguous K, V for kvh */
            size_t n = (size_t)(len > 0 ? len : 1) * (size_t)head_dim;
            double *K = (double *)malloc(n * sizeof(double));
            double *V = (double *)malloc(n * sizeof(double));
            double *scores = (double *)malloc((size_t)(len > 0 ? len : 1) * sizeof(double));
            double *qd = (double *)malloc((size_t)head_dim * sizeof(double));
            if (!K || !V || !scores || !qd) {
                status = ORC_ERR_NOMEM;
            } else {
                for (int64_t j = 0; j < len && status == ORC_OK; ++j) {
                    int64_t logical = j / block_size;
                    int64_t in_block = j % block_size;
                    int64_t phys = block_tables[i * max_blocks_per_seq + logical];
                    if (phys < 0 || phys >= num_blocks) {
                        status = ORC_ERR_RANGE;
                        break;
                    }
                    for (int64_t d = 0; d < head_dim; ++d) {
                        K[j * head_dim + d] = cache_at(k_cache, phys, in_block, kvh, d, block_size,
                                                       num_kv_heads, head_dim);
                        V[j * head_dim + d] = cache_at(v_cache, phys, in_block, kvh, d, block_size,
                                                       num_kv_heads, head_dim);
                    }
                }
                for (int64_t g = 0; g < group && status == ORC_OK; ++g) {
                    int64_t h = kvh * group + g;
                    int wanted = !pairs;
                    for (int64_t p = 0; pairs && p < num_pairs; ++p)
                        if (pairs[2 * p] == i && pairs[2 * p + 1] == h)
                            wanted = 1;
                    if (!wanted)
                        continue;
                    for (int64_t d = 0; d < head_dim; ++d)
                        qd[d] = oracle_half_to_double(q[(i * num_heads + h) * head_dim + d]);
                    textbook_attention(out + (i * num_heads + h) * head_dim, qd, K, V, len,
                                       head_dim, scale, scores);
                }
            }
            free(K);
            free(V);
            free(scores);
            free(qd);
        }
    }
    return status;
}

/* Paged decode attention over an E4M3 cache: the same textbook computation as
 * oracle_decode_attention with each key/value element dequantized exactly
 * (value(code) * scale of its (token, head) row, in float64). */
int oracle_decode_attention_fp8(double *out, const uint16_t *q, const uint8_t *k_cache,
                                const uint8_t *v_cache, const float *k_scale,
                                const float *v_scale, const int32_t *block_tables,
                                const int32_t *seq_lens, double scale, int64_t num_seqs,
                                int64_t num_heads, int64_t num_kv_heads, int64_t head_dim,
                                int64_t block_size, int64_t max_blocks_per_seq,
                                int64_t num_blocks, const int32_t *pairs, int64_t num_pairs)
{
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks_per_seq < 0 || num_seqs < 0)
        return ORC_ERR_ARG;
    int64_t group = num_heads / num_kv_heads;
    int status = ORC_OK;
    for (int64_t i = 0; i < num_seqs && status == ORC_OK; ++i) {
        int64_t len = seq_lens[i];
        if (len < 0 || len > max_blocks_per_seq * block_size)
            return ORC_ERR_RANGE;
        for (int64_t kvh = 0; kvh < num_kv_heads && status == ORC_OK; ++kvh) {
            int want_any = !pairs;
            for (int64_t p = 0; pairs && p < num_pairs; ++p)
                if (pairs[2 * p] == i && pairs[2 * p + 1] / group == kvh)
                    want_any = 1;
            if (!want_any)
                continue;
            size_t n = (size_t)(len > 0 ? len : 1) * (size_t)head_dim;
            double *K = (double *)malloc(n * sizeof(double));
            double *V = (double *)malloc(n * sizeof(double));
            double *scores = (double *)malloc((size_t)(len > 0 ? len : 1) * sizeof(double));
            double *qd = (double *)malloc((size_t)head_dim * sizeof(double));
            if (!K || !V || !scores || !qd) {
                status = ORC_ERR_NOMEM;
            } else {
                for (int64_t j = 0; j < len && status == ORC_OK; ++j) {
                    int64_t phys = block_tables[i * max_blocks_per_seq + j / block_size];
                    if (phys < 0 || phys >= num_blocks) {
                        status = ORC_ERR_RANGE;
                        break;
                    }
                    int64_t row = (phys * block_size + j % block_size) * num_kv_heads + kvh;
                    for (int64_t d = 0; d < head_dim; ++d) {
                        K[j * head_dim + d] =
                            oracle_e4m3_value(k_cache[row * head_dim + d]) * (double)k_scale[row];
                        V[j * head_dim + d] =
                            oracle_e4m3_value(v_cache[row * head_dim + d]) * (double)v_scale[row];
                    }
                }
                for (int64_t g = 0; g < group && status == ORC_OK; ++g) {
                    int64_t h = kvh * group + g;
                    int wanted = !pairs;
                    for (int64_t p = 0; pairs && p < num_pairs; ++p)
                        if (pairs[2 * p] == i && pairs[2 * p + 1] == h)
                            wanted = 1;
                    if (!wanted)
                        continue;
                    for (int64_t d = 0; d < head_dim; ++d)
                        qd[d] = oracle_half_to_double(q[(i * num_heads + h) * head_dim + d]);
                    textbook_attention(out + (i * num_heads + h) * head_dim, qd, K, V, len,
                                       head_dim, scale, scores);
                }
            }
            free(K);
            free(V);
            free(scores);
            free(qd);
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Attention of a chunk of new tokens per sequence ("vLLM 技术内幕" §3.2: V1
 * schedules prompt and output tokens alike, {request: num_tokens} per step,
 * a long prompt cut into chunks across steps beside running decodes; §7.4:
 * draft tokens are scheduled with their request and verified together).
 * Sequence i holds seq_lens[i] = L tokens in the cache after this step's
 * write; the last Q = query_start[i+1] - query_start[i] of them are new.  New
 * token j (0 <= j < Q) sits at position L - Q + j and attends to the cached
 * positions 0 .. L - Q + j (itself and everything before it).  q and out are
 * [query_start[S], H, D]; row r of q is new token r - query_start[i] of the
 * sequence i with query_start[i] <= r < query_start[i+1].  With `rows`
 * (a list of query rows) only those rows are computed; the others are left
 * untouched. */
int oracle_chunk_attention(double *out, const uint16_t *q, const uint16_t *k_cache,
                           const uint16_t *v_cache, const int32_t *block_tables,
                           const int32_t *seq_lens, const int32_t *query_start, double scale,
                           int64_t num_seqs, int64_t num_heads, int64_t num_kv_heads,
                           int64_t head_dim, int64_t block_size, int64_t max_blocks_per_seq,
                           int64_t num_blocks, const int64_t *rows, int64_t num_rows)
{
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks_per_seq < 0 || num_seqs < 0 || query_start[0] != 0)
        return ORC_ERR_ARG;
    int64_t group = num_heads / num_kv_heads;
    int status = ORC_OK;
    for (int64_t i = 0; i < num_seqs && status == ORC_OK; ++i) {
        int64_t len = seq_lens[i];
        int64_t r0 = query_start[i], r1 = query_start[i + 1];
        int64_t nq = r1 - r0;
        if (len < 0 || len > max_blocks_per_seq * block_size || nq < 0 || nq > len)
            return ORC_ERR_RANGE;
        /* any wanted row in this sequence? */
        int want_any = 0;
        for (int64_t r = r0; r < r1 && !want_any; ++r) {
            if (!rows) {
                want_any = 1;
            } else {
                for (int64_t k = 0; k < num_rows; ++k)
                    if (rows[k] == r)
                        want_any = 1;
            }
        }
        if (!want_any)
            continue;
        for (int64_t kvh = 0; kvh < num_kv_heads && status == ORC_OK; ++kvh) {
            size_t n = (size_t)(len > 0 ? len : 1) * (size_t)head_dim;
            double *K = (double *)malloc(n * sizeof(double));
            double *V = (double *)malloc(n * sizeof(double));
            double *scores = (double *)malloc((size_t)(len > 0 ? len : 1) * sizeof(double));
            double *qd = (double *)malloc((size_t)head_dim * sizeof(double));
            if (!K || !V || !scores || !qd) {
                status = ORC_ERR_NOMEM;
            } else {
                for (int64_t j = 0; j < len && status == ORC_OK; ++j) {
                    int64_t phys = block_tables[i * max_blocks_per_seq + j / block_size];
                    if (phys < 0 || phys >= num_blocks) {
                        status = ORC_ERR_RANGE;
                        break;
                    }
                    for (int64_t d = 0; d < head_dim; ++d) {
                        K[j * head_dim + d] = cache_at(k_cache, phys, j % block_size, kvh, d,
                                                       block_size, num_kv_heads, head_dim);
                        V[j * head_dim + d] = cache_at(v_cache, phys, j % block_size, kvh, d,
                                                       block_size, num_kv_heads, head_dim);
                    }
                }
                for (int64_t r = r0; r < r1 && status == ORC_OK; ++r) {
                    int wanted = !rows;
                    for (int64_t k = 0; rows && k < num_rows; ++k)
                        if (rows[k] == r)
                            wanted = 1;
                    if (!wanted)
                        continue;
                    int64_t pos = len - nq + (r - r0); /* the new token's position */
                    for (int64_t g = 0; g < group; ++g) {
                        int64_t h = kvh * group + g;
                        for (int64_t d = 0; d < head_dim; ++d)
                            qd[d] = oracle_half_to_double(q[(r * num_heads + h) * head_dim + d]);
                        /* causal: positions 0 .. pos */
                        textbook_attention(out + (r * num_heads + h) * head_dim, qd, K, V,
                                           pos + 1, head_dim, scale, scores);
                    }
                }
            }
            free(K);
            free(V);
            free(scores);
            free(qd);
        }
    }
    return status;
}
