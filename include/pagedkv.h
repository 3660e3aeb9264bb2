/*
 * pagedkv.h -- C ABI of libpagedkv, the GB300 (sm_103a) hot path of paged
 * KV-cache attention: the paged cache write and paged decode attention.
 *
 * Conventions for every entry point:
 *  - Pointers named *_cache, q, out, k, v, slot_mapping, block_tables,
 *    seq_lens and workspace are DEVICE pointers owned by the caller; the
 *    library never allocates, frees or retains them beyond the call.
 *  - Every call is asynchronous on `stream` (NULL = the legacy default
 *    stream) and never synchronises, except pkv_get_device_error.
 *  - Every call first validates its arguments on the host; an invalid call
 *    returns a negative pkv_status and launches nothing.  A failed launch
 *    returns PKV_ERR_CUDA (pkv_last_error_string() has the CUDA message).
 *  - Bad DATA found on the device (a slot or block id out of range, a
 *    sequence longer than its block table) never faults: the offending item
 *    is skipped and the first one is recorded; read it with
 *    pkv_get_device_error.
 *  - fp16 means IEEE binary16 (CUDA __half).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_NULL = -1,        /* a required pointer is NULL                        */
    PKV_ERR_INVALID = -2,     /* a size, stride or count is out of its domain      */
    PKV_ERR_UNSUPPORTED = -3, /* valid but not built: head_dim, group size, bs ... */
    PKV_ERR_ALIGNMENT = -4,   /* a pointer or stride breaks a required alignment   */
    PKV_ERR_WORKSPACE = -5,   /* split-KV needs a (larger) workspace               */
    PKV_ERR_CUDA = -6         /* a CUDA runtime call or launch failed              */
} pkv_status;

/* Kinds recorded by the device-side error word (pkv_get_device_error). */
typedef enum pkv_device_error {
    PKV_DEVERR_NONE = 0,
    PKV_DEVERR_SLOT = 1,     /* slot >= num_blocks*block_size; index = token          */
    PKV_DEVERR_BLOCK_ID = 2, /* block id outside [0, num_blocks);
                                index = seq * max_blocks_per_seq + logical block     */
    PKV_DEVERR_SEQ_LEN = 3,  /* seq_len < 0, or more tokens than the block table or
                                max_seq_len allow; index = seq                         */
    PKV_DEVERR_TIMEOUT = 4   /* a staging wait gave up (about 2 s); index = CTA id   */
} pkv_device_error;

/*
 * One cache view ("vLLM KV Cache Layout 可视化" -- 核心, KVCacheTensor): a
 * group of same-shaped layers inside one byte allocation.  The byte address
 * of slot `s` of layer `layer` is
 *     offset + layer*layer_stride + (s / block_size)*block_stride
 *            + (s % block_size)*row_width.
 * Layer-outer layouts (LBHNC, LBNHC) have block_stride = page and
 * layer_stride = page*num_blocks; block-outer layouts (BLHNC, BLNHC, BHLNC)
 * have layer_stride = page and block_stride = the bytes of one whole block
 * (page = block_size*row_width) ("layout 是什么").
 */
typedef struct pkv_view {
    int64_t offset;       /* bytes from the cache pointer to layer 0, block 0   */
    int64_t layer_stride; /* bytes between the same block of adjacent layers    */
    int64_t block_stride; /* bytes between adjacent physical blocks of a layer  */
    int64_t row_width;    /* bytes of one token row (one slot)                  */
    int32_t layer;        /* the layer this call writes                         */
} pkv_view;

/*
 * Paged KV-cache write ("vLLM KV Cache Layout 可视化" -- 查一个 token and
 * kernel 那一侧; "deep-dive-into-vllm-05" §2: prefill writes many slots,
 * decode appends one per sequence).
 *
 * For every token t in [0, num_tokens): slot = slot_mapping[t] is split back
 * into block = slot / block_size and position = slot % block_size, and the
 * row_width bytes at k + t*row_width are copied to
 *     k_cache + offset + layer*layer_stride + block*block_stride
 *             + position*row_width
 * (and likewise v -> v_cache, at the same address, when v != NULL).
 *
 *  k, v          device, num_tokens rows of view.row_width bytes, contiguous.
 *                v may be NULL (single-cache write); then v_cache must be NULL.
 *  slot_mapping  device int64 [num_tokens].  A negative slot is padding and is
 *                skipped.  slot >= num_blocks*block_size is skipped and
 *                recorded (PKV_DEVERR_SLOT).  Two tokens with the same slot
 *                in one call: which row lands is unspecified.
 *  k_cache, v_cache  device byte allocations holding the view; the caller
 *                guarantees every slot in [0, num_blocks*block_size) of the
 *                view lies inside them.  Bytes no token addresses are not
 *                touched.
 *  Rows are copied byte for byte (no conversion); 16-byte vectors are used
 *  when every address and stride allows, else 8, 4, 2 or 1 byte.
 *  Returns PKV_OK (num_tokens == 0 launches nothing), PKV_ERR_NULL,
 *  PKV_ERR_INVALID (block_size <= 0, num_blocks <= 0, row_width <= 0 or
 *  > 2^30, block_stride <= 0, offset/layer/layer_stride < 0), PKV_ERR_CUDA.
 */
int pkv_cache_write(const void *k, const void *v, const int64_t *slot_mapping,
                    int64_t num_tokens, void *k_cache, void *v_cache, pkv_view view,
                    int32_t block_size, int64_t num_blocks, pkv_stream_t stream);

/* One (source rows, cache, view) triple of pkv_cache_write_multi. */
typedef struct pkv_write_desc {
    const void *src; /* device: num_tokens rows of view.row_width bytes      */
    void *cache;     /* device byte allocation holding the view              */
    pkv_view view;   /* includes the layer written                           */
} pkv_write_desc;

#define PKV_MAX_WRITE_DESCS 32

/*
 * Several cache writes that share one slot_mapping, in one launch: for every
 * token t and descriptor d, the row at d.src + t*d.view.row_width goes to the
 * address of slot_mapping[t] in d's view, exactly as pkv_cache_write does.
 * This is how every layer and cache of one block table is written at once:
 * the two caches (MLA and indexer) of "vLLM KV Cache Layout 可视化" --
 * 两种 cache 共用一张 block table share one slot number per token (查一个
 * token).
 *  descs       HOST array of num_descs (0..PKV_MAX_WRITE_DESCS) descriptors;
 *              read during the call only.  Rows of different descriptors must
 *              not overlap in memory (which lands is then unspecified).
 *  Other arguments, slot rules and errors as pkv_cache_write.
 */
int pkv_cache_write_multi(const pkv_write_desc *descs, int32_t num_descs,
                          const int64_t *slot_mapping, int64_t num_tokens, int32_t block_size,
                          int64_t num_blocks, pkv_stream_t stream);

/*
 * Copy whole physical blocks within one cache view ("vLLM 技术内幕" §2.2,
 * copy on write: a sequence about to write into a block whose ref_cnt is
 * above one gets a new block holding a copy of the old one).
 * For each pair p in [0, num_pairs), with src = block_mapping[2p] and dst =
 * block_mapping[2p+1], and each layer l in [view.layer, view.layer +
 * num_layers): the page of block_size*row_width bytes at
 *     offset + l*layer_stride + src*block_stride
 * is copied to the same place of block dst.
 *  cache          device byte allocation holding the view.
 *  block_mapping  device int64 [num_pairs][2].  A pair with an id outside
 *                 [0, num_blocks) is skipped and recorded (PKV_DEVERR_BLOCK_ID,
 *                 index = pair); src == dst is a no-op.  A block must not be
 *                 both a source and a destination, nor a destination twice
 *                 (the result is then unspecified).
 *  Returns PKV_OK (nothing to copy launches nothing), PKV_ERR_NULL,
 *  PKV_ERR_INVALID, PKV_ERR_ALIGNMENT, PKV_ERR_CUDA.
 */
int pkv_copy_blocks(void *cache, pkv_view view, int32_t num_layers, int32_t block_size,
                    const int64_t *block_mapping, int64_t num_pairs, int64_t num_blocks,
                    pkv_stream_t stream);

/*
 * Paged decode attention ("deep-dive-into-vllm-05" §2 read loop and §3.2
 * GQA; "vLLM 技术内幕" §2.1: the query is dotted with the keys of each
 * physical block in turn and values are accumulated block by block).
 *
 * For sequence i (length L = seq_lens[i]) and query head h, with G =
 * num_heads/num_kv_heads and kv = h / G (consecutive heads share a KV head):
 *     s_j  = scale * q[i,h,:] . K_j,   K_j = k_cache[bt[i, j/bs], j%bs, kv, :]
 *     out[i,h,:] = sum_j exp(s_j - max s) V_j / sum_j exp(s_j - max s),
 * j in [0, L).  Computed block by block with an online (running max / sum)
 * softmax in fp32; a sequence whose blocks are spread over several CTAs
 * leaves partial (max, sum, weighted values) that are merged with a
 * log-sum-exp rescale inside the same launch.  L == 0 gives zeros.
 *
 * Two schedules (pkv_decode_options.schedule):
 *  - balanced (default): one wave of persistent CTAs, each owning an equal
 *    share of all (KV head group, sequence, block) triples -- a CTA serves up
 *    to 8 KV heads of one group, so more KV heads make more groups; needs a
 *    workspace of pkv_decode_workspace_bytes(...) bytes;
 *  - grid: one CTA per (kv head, sequence, partition of 512 tokens); needs a
 *    workspace only when max_seq_len > 512.
 * With AUTO the balanced schedule runs when the shape and the workspace
 * allow it, else the grid schedule.
 *
 *  out           device fp16 [num_seqs, num_heads, head_dim] (written).
 *  q             device fp16 [num_seqs, num_heads, head_dim].
 *  k_cache, v_cache  device fp16 [num_blocks, block_size, num_kv_heads,
 *                head_dim] ("deep-dive-into-vllm-05" §1.2), 16-byte aligned.
 *  block_tables  device int32 [num_seqs, max_blocks_per_seq]; entries past a
 *                sequence's ceil(L/block_size) blocks are ignored.  An id
 *                outside [0, num_blocks) is skipped and recorded.
 *  seq_lens      device int32 [num_seqs].  A length beyond the block table
 *                (or, on the grid schedule, beyond max_seq_len) is truncated
 *                and recorded (PKV_DEVERR_SEQ_LEN).
 *  max_seq_len   host hint: an upper bound of seq_lens (sizes the grid
 *                schedule's partitions).
 *  workspace     device scratch, 16-byte aligned, of at least
 *                pkv_decode_workspace_bytes(...) bytes (or NULL, see above).
 *                It must be zero-filled before its first use (e.g. by
 *                pkv_decode_workspace_init); every call that records no
 *                PKV_DEVERR_TIMEOUT leaves it zero-filled again.  Calls that
 *                share a workspace must not overlap on the GPU.
 *  Ordering: the launch may overlap the previous kernel in the stream when
 *  that kernel signals programmatic launch completion (pkv_cache_write does).
 *  Before that kernel's completion the call reads only q, block_tables and
 *  seq_lens; it reads the caches and writes out/workspace only after.  So a
 *  preceding kernel that signals early must not write q, block_tables or
 *  seq_lens (kernels that never signal are waited for in full, as usual).
 *  Supported: head_dim in {64, 128}; G in {1, 2, 4, 8}; block_size == 16;
 *  num_seqs <= 65535.
 *  Returns PKV_OK (num_seqs == 0 launches nothing), PKV_ERR_NULL,
 *  PKV_ERR_INVALID, PKV_ERR_UNSUPPORTED, PKV_ERR_ALIGNMENT,
 *  PKV_ERR_WORKSPACE, PKV_ERR_CUDA.
 */
int pkv_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *seq_lens, float scale,
                         int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int32_t num_seqs, int32_t max_blocks_per_seq,
                         int32_t max_seq_len, int64_t num_blocks, void *workspace,
                         size_t workspace_bytes, pkv_stream_t stream);

/* How the per-block arithmetic of pkv_decode_attention_ex runs. */
typedef enum pkv_compute {
    PKV_COMPUTE_AUTO = 0, /* the measured-fastest path (MMA)                     */
    PKV_COMPUTE_SIMT = 1, /* fp32 FMA on CUDA cores, warp-shuffle reductions     */
    PKV_COMPUTE_MMA = 2   /* the GQA group packed into 16x8x16 fp16 MMAs, fp32
                             accumulate                                           */
} pkv_compute;

/* Which CTA schedule pkv_decode_attention_ex uses. */
typedef enum pkv_schedule {
    PKV_SCHEDULE_AUTO = 0,     /* balanced when possible, else grid           */
    PKV_SCHEDULE_GRID = 1,     /* one CTA per (kv head, sequence, partition)  */
    PKV_SCHEDULE_BALANCED = 2  /* persistent CTAs over equal block ranges     */
} pkv_schedule;

typedef struct pkv_decode_options {
    int32_t partition_size; /* grid schedule: tokens per partition, a multiple
                               of block_size in [16, 8192]; 0 = 512          */
    int32_t compute;        /* a pkv_compute value                           */
    int32_t schedule;       /* a pkv_schedule value                          */
} pkv_decode_options;

/* pkv_decode_attention with explicit options (opts may be NULL = defaults).
 * Asking for the balanced schedule when it cannot run returns
 * PKV_ERR_WORKSPACE (workspace too small) or PKV_ERR_UNSUPPORTED. */
int pkv_decode_attention_ex(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *seq_lens, float scale,
                            int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_seqs, int32_t max_blocks_per_seq,
                            int32_t max_seq_len, int64_t num_blocks, void *workspace,
                            size_t workspace_bytes, const pkv_decode_options *opts,
                            pkv_stream_t stream);

/* Workspace bytes for any schedule of pkv_decode_attention on the current
 * device (its SM count sizes the balanced schedule's partials; without a
 * device, a 256-SM bound is used).  0 for invalid arguments. */
size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_seq_len);

/* Same, for a grid-schedule partition size (0 = 512). */
size_t pkv_decode_workspace_bytes_ex(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t max_seq_len,
                                     int32_t partition_size);

/*
 * FP8 KV cache ("deep-dive-into-vllm-05" §3.4: quantize on write -- the KV is
 * stored at low precision when written -- and dequantize on read inside the
 * attention kernel; the scales stay with the blocks).  Format: E4M3 (OCP
 * FP8: 4 exponent bits, bias 7, 3 mantissa bits, largest finite 448), one
 * fp32 scale per (token, KV head) row -- the pages' indexer rows carry one
 * FP32 scale per 128 FP8 values ("vLLM KV Cache Layout 可视化").
 *
 * Caches: k_cache, v_cache uint8 [num_blocks, block_size, num_kv_heads,
 * head_dim]; k_scale, v_scale fp32 [num_blocks, block_size, num_kv_heads].
 *
 * pkv_cache_write_fp8 quantizes fp16 rows k, v [num_tokens, num_kv_heads,
 * head_dim] into their slots, in fp32: amax = max |x| of the row,
 * s = amax / 448, code = round-to-nearest-even(x / s) saturated to +-448
 * (s == 0 gives zero codes).  Slot rules and errors as pkv_cache_write;
 * head_dim in {64, 128}; v, v_cache, v_scale all NULL or all set.
 */
int pkv_cache_write_fp8(const void *k, const void *v, const int64_t *slot_mapping,
                        int64_t num_tokens, void *k_cache, void *v_cache, float *k_scale,
                        float *v_scale, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int64_t num_blocks, pkv_stream_t stream);

/*
 * pkv_decode_attention over FP8 caches (balanced schedule, MMA policy): keys
 * and values are dequantized as value(code) * scale of their row; the result
 * is the attention of pkv_decode_attention on those values.  Needs
 * 16-byte aligned caches and scales and a workspace of
 * pkv_decode_workspace_bytes(...) bytes (zero-filled before first use, left
 * zero-filled).  Other arguments and errors as pkv_decode_attention.
 */
int pkv_decode_attention_fp8(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const float *k_scale, const float *v_scale,
                             const int32_t *block_tables, const int32_t *seq_lens, float scale,
                             int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int32_t num_seqs, int32_t max_blocks_per_seq,
                             int32_t max_seq_len, int64_t num_blocks, void *workspace,
                             size_t workspace_bytes, pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * Attention of a chunk of new tokens per sequence ("vLLM 技术内幕" §3.2: V1
 * schedules prompt and output tokens alike -- {request: num_tokens} per step
 * -- and cuts a long prompt into chunks that run beside the decodes; §7.4:
 * draft tokens are scheduled with their request and verified together).
 *
 * Sequence i holds seq_lens[i] = L tokens in the cache, this step's new
 * tokens included (write them first, e.g. with pkv_cache_write); its last
 * Q = query_start[i+1] - query_start[i] tokens are the new ones.  New token
 * j (0 <= j < Q) sits at position L - Q + j and attends causally to the
 * cache positions 0 .. L - Q + j.  A chunk of one token is a decode.
 *   out, q          fp16 [num_query_tokens, num_heads, head_dim]; query row r
 *                   is new token r - query_start[i] of the sequence i with
 *                   query_start[i] <= r < query_start[i+1]
 *   k_cache, v_cache, block_tables, seq_lens, scale, num_heads,
 *   num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks:
 *                   as for pkv_decode_attention
 *   query_start     int32 [num_seqs + 1], device: query_start[0] = 0,
 *                   non-decreasing, query_start[num_seqs] = num_query_tokens
 *   max_query_len   host bound on every Q (sizes the launch)
 *   max_seq_len     host bound on every L (sizes the launch and workspace)
 *   workspace       pkv_chunk_workspace_bytes(...) bytes, zeroed once
 *                   (pkv_decode_workspace_init); every call leaves it zeroed
 * Ordering: as for pkv_decode_attention, the launch may overlap a previous
 * kernel that signals programmatic launch completion (pkv_cache_write does);
 * before that kernel's completion the call reads only seq_lens, query_start,
 * q and block_tables, so such a kernel must not write those.
 * Supported: head_dim 64 or 128, block_size 16, group size 1, 2, 4 or 8.
 * Rows of a sequence whose Q exceeds max_query_len or L, or whose L exceeds
 * its block table or max_seq_len, are skipped and recorded as
 * PKV_DEVERR_SEQ_LEN; a bad block id is skipped and recorded.
 * Returns PKV_ERR_WORKSPACE when the workspace is missing or too small. */
int pkv_chunk_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_tables, const int32_t *seq_lens,
                        const int32_t *query_start, float scale, int32_t num_heads,
                        int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                        int32_t num_seqs, int32_t max_blocks_per_seq, int32_t num_query_tokens,
                        int32_t max_query_len, int32_t max_seq_len, int64_t num_blocks,
                        void *workspace, size_t workspace_bytes, pkv_stream_t stream);

/* Workspace bytes pkv_chunk_attention needs for these bounds (0 for an
 * invalid shape): the short chunks' scratch, the work list, tickets, and,
 * when max_seq_len exceeds one 4096-token KV partition, fp32 partial states
 * of every query row for each partition. */
size_t pkv_chunk_workspace_bytes(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t num_query_tokens,
                                 int32_t max_query_len, int32_t max_seq_len);

/* Bytes of the built-in scratch of pkv_decode_attention_noalloc (16 MiB). */
#define PKV_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * pkv_decode_attention without a workspace, for callers that cannot allocate
 * device memory: a plugin inside a host runtime that owns the device-memory
 * budget and passes in only inputs and outputs, or a latency-critical loop
 * that must never call cudaMalloc (which can synchronise the device).  The
 * pages have no counterpart; it computes exactly what pkv_decode_attention
 * computes, with the same arguments minus the workspace.
 *
 * Its scratch is a device array of PKV_NOALLOC_SCRATCH_BYTES built into the
 * library: every device that loads the library holds it until the process
 * exits.  The call allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine).
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress); make that first call
 *    before any stream capture.
 *  - Every call clears the array's ticket counters on `stream` before the
 *    kernel (the array keeps the previous call's contents otherwise).
 *  - All calls share the one array: calls that overlap on the GPU (other
 *    streams, other threads) race and corrupt each other's results.
 *  - A shape whose scratch need exceeds PKV_NOALLOC_SCRATCH_BYTES is refused
 *    with PKV_ERR_WORKSPACE before anything runs (pkv_last_error_string()
 *    gives the bytes needed); use pkv_decode_attention for it.
 */
int pkv_decode_attention_noalloc(void *out, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_tables,
                                 const int32_t *seq_lens, float scale, int32_t num_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int32_t num_seqs, int32_t max_blocks_per_seq,
                                 int32_t max_seq_len, int64_t num_blocks, pkv_stream_t stream);

/* Zero-fill a workspace on `stream` (cudaMemsetAsync). */
int pkv_decode_workspace_init(void *workspace, size_t workspace_bytes, pkv_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the device-side error record of
 * the current device: *kind receives a pkv_device_error value (0 = none) and
 * *index its index (-1 when none).  Either pointer may be NULL.
 */
int pkv_get_device_error(int32_t *kind, int64_t *index, pkv_stream_t stream);

/* Static text for a pkv_status value. */
const char *pkv_status_string(int status);

/* Text of the last CUDA error a call of this thread returned PKV_ERR_CUDA for. */
const char *pkv_last_error_string(void);

/* ABI version of this header (major*10000 + minor*100 + patch). */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
