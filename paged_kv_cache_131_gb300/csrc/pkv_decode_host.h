// pkv_decode_host.h -- launch parameters shared by the two decode schedules
// (grid: one CTA per kv_head x partition x sequence; balanced: persistent
// CTAs over equal ranges of the (sequence, block) space).
#pragma once

#include <cuda.h>  // CUtensorMap (a 128-byte descriptor; no driver call here)
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

struct ErrorRecord;

namespace dec {

constexpr int kGridWarps = 4;
constexpr int kGridStages = 2;
constexpr int kMaxPartitionTokens = 8192;
constexpr int kDefaultPartitionTokens = 512;
constexpr int kMaxBalancedKvHeads = 8;   // KV heads (consumer warps) per CTA (+1 producer)
constexpr int kSmemPerSM = 227 * 1024;   // opt-in dynamic shared memory per CTA
constexpr int kTileAlign = 1024;         // staged tiles start 1024-byte aligned (swizzle)

// Bytes of a staged row's swizzle chunk: 128 when the row is a multiple of
// 128 bytes, else 64 (rows are always a multiple of 64).
__host__ __device__ constexpr int chunk_bytes_for_row(int row_bytes) {
    return row_bytes % 128 == 0 ? 128 : 64;
}

// Tensor map over a token-major cache [num_blocks * 16 rows][row_bytes]
// viewed as {chunk bytes, token rows, chunks} (the chunk stride is smaller
// than the row stride), with a box of {chunk, 16 tokens, box_chunks} and the
// chunk's swizzle.  A box lands in shared memory as 16 * box_chunks * chunk
// bytes, chunk-major.  Returns a PKV status.
int make_kv_tensor_map(CUtensorMap *map, const void *cache, int64_t num_blocks, int row_bytes,
                       int box_chunks);

// Tensor map over query rows fp16 [num_tokens][num_heads][head_dim] viewed
// as {head_dim * 2 bytes, heads, tokens}, with a box of {128 bytes, group
// heads, 128 / group tokens} and the 128-byte swizzle: a box at (128 c,
// kv_head * group, token t) lands as 128 rows (token-major, head-minor) of
// the bytes 128 c .. 128 c + 127 of each head.  Returns a PKV status.
int make_q_tensor_map(CUtensorMap *map, const void *q, int64_t num_tokens, int num_heads,
                      int head_dim, int group);

// Grid schedule.
struct GridParams {
    CUtensorMap tm_k;  // per-head boxes of the key / value caches
    CUtensorMap tm_v;
    __half *out;
    const __half *q;
    const __half *k_cache;
    const __half *v_cache;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    float scale_log2;  // scale * log2(e): scores live in the log2 domain
    int num_heads;
    int num_kv_heads;
    int max_blocks_per_seq;
    int num_partitions;    // P, grid.z
    int partition_blocks;  // partition_size / 16
    int64_t num_blocks;
    int *counters;    // [S * Hk] tickets, zero between calls
    float2 *part_ml;  // [S, H, P] (m, l)
    float *part_o;    // [S, H, P, D]
    ErrorRecord *err;
};

// Bytes of the grid schedule's staging rings (reused by its combine).
int grid_ring_bytes(int D);
int grid_smem_bytes(int D, int G, int partition_blocks);
int64_t grid_workspace_bytes(int64_t S, int64_t H, int64_t D, int64_t P);
int launch_grid(const GridParams &p, int D, int G, bool simt, int num_seqs,
                cudaStream_t stream);

// Balanced schedule.
struct BalancedParams {
    CUtensorMap tm_k;  // whole-row boxes of the key / value caches
    CUtensorMap tm_v;
    __half *out;
    const __half *q;
    const __half *k_cache;
    const __half *v_cache;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    float scale_log2;
    int num_seqs;
    int num_heads;
    int num_kv_heads;
    int max_blocks_per_seq;
    int num_stages;  // staging ring depth (blocks in flight per CTA)
    int row_bytes;   // staged row: one head group of one token, heads_per_cta*D*elem bytes
    // the KV heads are taken in groups of heads_per_cta (<= 8, one consumer
    // warp each); the work list is (group, sequence, block), groups outermost
    int heads_per_cta;
    int groups;      // num_kv_heads / heads_per_cta
    const float *k_scale;  // FP8 caches: [NB, 16, Hk] per-row scales (else null)
    const float *v_scale;
    // several new tokens per sequence (MmaColsPolicy): sequence i's query
    // rows are query_start[i] .. query_start[i+1]-1; sequences whose
    // (new tokens x group) exceeds max_cols are left to the chunk kernel.
    // Null for decode (one new token per sequence, query row = sequence).
    const int32_t *query_start;
    int max_cols;
    int num_query_tokens;
    // 1: nothing this kernel reads was written by the kernel launched just
    // before it (launched with programmatic serialisation), so it waits for
    // that kernel only before exiting; 0: it waits before touching the caches
    int defer_wait;
    // if non-null and > 0 there: the work is split over that many CTAs (the
    // first ones) instead of the whole grid; written by an earlier kernel
    const int *active_ctas;
    int64_t num_blocks;
    int *counters;    // [S * Hk] tickets, zero between calls
    float2 *part_ml;  // [2 * grid][heads_per_cta][rows]
    float *part_o;    // [2 * grid][heads_per_cta][rows][D]
    ErrorRecord *err;
};

struct BalancedShape {
    bool ok;          // the schedule supports this shape
    int stages;       // ring depth
    int heads;        // KV heads per CTA (a divisor of num_kv_heads, <= 8)
    int groups;       // num_kv_heads / heads
    int row_bytes;    // staged row bytes (one head group)
    int smem;         // dynamic shared memory per CTA
    int ctas_per_sm;  // resident CTAs per SM
    int grid;         // CTAs launched
    int64_t workspace;  // bytes of scratch it needs
};

// Shape of the balanced launch for fp16 or FP8 caches; rows = partial-state
// rows per (sequence, kv head): G for decode, 8 * col_tiles for chunks.
BalancedShape balanced_shape(int num_seqs, int num_kv_heads, int G, int D, int num_sms,
                             bool fp8, int rows = 0);
// Sets the fields of p that follow from the shape -- ring depth, staged row,
// head groups, the scratch layout inside `workspace` (counters, partial
// states for `rows` rows per (sequence, kv head)) and the tensor maps of the
// two caches (p.num_seqs, p.num_kv_heads and p.num_blocks must be set).
// Returns a PKV status.
int setup_balanced(BalancedParams &p, const BalancedShape &shape, int rows, void *workspace,
                   const void *k_cache, const void *v_cache);
// col_tiles: 0 for decode, else the column n-tiles (1 or 2) of MmaColsPolicy.
int launch_balanced(const BalancedParams &p, const BalancedShape &shape, int D, int G, bool simt,
                    bool fp8, cudaStream_t stream, int col_tiles = 0);

inline int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// The argument checks every fp16 decode entry point makes before it touches
// a stream: pointers, sizes, supported shape (G in {1,2,4,8}, head_dim 64 or
// 128, block_size 16) and alignment.  Returns a PKV status (PKV_OK also for
// num_seqs == 0, which launches nothing).
int check_decode_args(const void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, const int32_t *seq_lens, float scale,
                      int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t num_seqs, int32_t max_blocks_per_seq,
                      int32_t max_seq_len, int64_t num_blocks);

}  // namespace dec
}  // namespace pkv
