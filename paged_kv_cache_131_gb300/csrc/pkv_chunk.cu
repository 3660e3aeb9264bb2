// pkv_chunk.cu -- attention of a chunk of new tokens per sequence over the
// paged cache, causal within the new tokens ("vLLM 技术内幕" §3.2: chunked
// prefill, prompt and output tokens scheduled alike; §7.4: draft tokens
// verified together).  Sequence i holds L tokens, the last Q of them new;
// new token j (position L - Q + j) attends to positions 0 .. L - Q + j.
//
// Sequences whose new tokens times the group size fit the balanced decode
// schedule's query columns (8 or 16: MmaColsPolicy) run there -- the same
// streaming of whole token rows as a decode; the others run here, on the
// fifth-generation tensor cores (tcgen05) with accumulators in tensor memory.
//
// The work is a list of items (query tile of 128 rows, KV head, KV
// partition of 4096 tokens, sequence), built on the device by a one-CTA plan
// kernel for the sequences this kernel takes (partitions past a tile's
// causal range are not items).  Persistent CTAs (one per SM) pull items in
// list order from an atomic counter, so tiles with more keys and tiles with
// fewer balance out.  A row is (new token j, query head g of the KV head's
// group): row = j*G + g, so a tile covers 128/G consecutive new tokens.
// When both kernels have work, the plan kernel also estimates each one's
// share and picks how many SMs the balanced schedule gets; this kernel's
// last that-many CTAs leave at once and the balanced grid uses only its
// first that-many, so the two run side by side on disjoint SMs.
//
// Per CTA, warp-specialised, all hand-offs through mbarriers:
//  * warp 0 takes the items (the next one when the current one's last step
//    is staged; the longest items are handed out first), stages the tile's
//    query rows into shared memory and the partition's
//    keys, 8 blocks (128 keys) per step, one tensor copy per block and
//    64-dimension chunk, into a 4-step ring laid out [chunk][key][128 B] so
//    the 128 keys form one MMA operand;
//  * warp 1 stages the values, one tensor copy per block, into a 2-step ring;
//  * warp 2 (one thread) copies the query tile into tensor memory (two
//    tiles in flight) and issues per step S = Q K^T (M = 128 rows, N = 128
//    keys, one MMA per 16-dimension k step, A read from tensor memory) into
//    a 128-column score buffer; warp 11 (one thread) issues O += P V
//    (N = head_dim, 16 keys per MMA) with the weights P read from tensor
//    memory (two buffers).  An MMA that depends on the previous one holds
//    its issuer back, so each chain has its own issuing warp;
//  * warps 3-10 run the softmax, two threads of one warp per query row,
//    each with half of each step's keys (tensor-memory loads of two 16-lane
//    halves): they read the row's scores, mask keys past the row's position
//    (and past the sequence or in a bad block), combine the two half-row
//    maxima with one shuffle, keep the row's running maximum m and the sums
//    l in the log2 domain and write the fp16 weights P = 2^(s - m) back to
//    tensor memory.  The reference m moves only when the maximum grows by
//    more than 2^8 (the weights stay <= 256): then each thread rescales its
//    half of the row's O in tensor memory first.  The result O / l does not
//    depend on which reference was used.
// A tile whose causal range fits one partition writes fp16 out; otherwise
// every partition leaves fp32 partial states (m, l, O) and, per softmax warp,
// the last CTA of the tile to take a ticket merges them with a log-sum-exp
// rescale.  No CTA waits for another.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "../../include/pagedkv.h"
#include "pkv_decode_common.cuh"
#include "pkv_decode_host.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace chunk {
namespace {

using dec::kBS;
using dec::kNegInf;

constexpr int kRows = 128;                     // query rows per tile: the MMA's M
constexpr int kStepBlocks = 8;                 // blocks per step
constexpr int kStepKeys = kStepBlocks * kBS;   // 128 keys: the score MMA's N
constexpr int kKStages = 4;                    // key ring depth (steps)
constexpr int kVStages = 2;                    // value ring depth (steps)
constexpr int kPartTokens = 4096;              // KV partition
constexpr int kClaimLead = 1;                  // steps staged after the next item is claimed
constexpr int kPartBlocks = kPartTokens / kBS;
// softmax: eight warps; warp 3 + 4 wh + q takes the rows (tensor-memory
// lanes) 32 q + 16 wh .. + 15, two threads per row: lanes 16 h + i take keys
// 64 h .. 64 h + 63 of a step and the head dimensions (D/2) h .. of O
constexpr int kSoftmaxWarps = 8;
constexpr int kGroupKeys = kStepKeys / 2;
constexpr int kPVWarp = 3 + kSoftmaxWarps;  // issues the P V MMAs (warp 2 the score MMAs)
constexpr int kThreads = (4 + kSoftmaxWarps) * 32;
// tensor memory: O in columns [0, head_dim), the scores in [128, 256), the
// weights (fp16 pairs) in two buffers of 64 columns, the query tile (fp16
// pairs, copied from shared memory) in two buffers of 64 columns
constexpr int kTmemCols = 512;
constexpr int kTmemO = 0;
constexpr int kTmemS = 128;
constexpr int kTmemP = 256;
constexpr int kTmemQ = 384;
constexpr float kRescaleLog2 = 8.f;            // move the reference past 2^8
// rates of the split between the call's two kernels (see the plan kernel)
// (single precision: this GPU's double-precision rate is low)
constexpr float kHbmBytesPerUs = 6.0e6f;        // decode stream, whole GPU
constexpr float kSmBytesPerUs = 58.0e3f;        // decode stream per SM
constexpr float kTileStepUs = 1.3f;             // one 128-key step of a tile

struct ChunkParams {
    CUtensorMap tm_k;  // keys: one 128-byte chunk of 16 rows per copy
    CUtensorMap tm_v;  // values: a head's chunks of 16 rows per copy
    CUtensorMap tm_q;  // query rows: 128 bytes of each row of a 128-row tile
    __half *out;
    const __half *q;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    const int32_t *query_start;
    float scale_log2;
    int num_heads;
    int num_kv_heads;
    int max_blocks_per_seq;
    int max_query_len;
    int max_seq_len;
    int num_tiles;  // tiles per (sequence, kv head) the tickets are sized for
    int num_parts;  // KV partitions the partial states are sized for
    int num_query_tokens;
    int min_rows;   // sequences with fewer rows (new tokens x group) are not ours
    int num_seqs;
    int head_dim;
    int num_ctas;    // CTAs the tile kernel is launched with
    int max_cols;    // rows the balanced schedule takes per (sequence, kv head); 0: none
    // work list: the sequences taken here (big_seq[k]) and the exclusive
    // prefix of their item counts (big_cum[k], big_cum[n_big] = total items);
    // *work is the next item to hand out
    int *big_seq;
    int *big_cum;
    int *n_big;
    int *work;
    // SMs left to the balanced schedule's share of the call (written by the
    // plan kernel; that many tile CTAs exit at once)
    int *split;
    int64_t num_blocks;
    int *counters;    // [S][Hk][num_tiles][8] tickets (one per softmax warp), zero between calls
    // partial states, row index R = kv_head * Tq * G + query_start * G + tile
    // row (the rows of a half-warp are consecutive): (m, l) [2 halves][parts][R]
    // (each half-warp keeps a copy), O [parts][D][R]
    float2 *part_ml;
    float *part_o;
    ErrorRecord *err;
};

// An item as the producer hands it to the other warps (64 bytes).
struct ItemInfo {
    int seq, part, kvh, tile;
    int nsteps, nblk, L, Q;
    int q0, nparts, done, pad;
    uint32_t valid[kPartBlocks / 32];  // one bit per block of the partition: id in range
};

// Shared memory (from a 1024-aligned base): the query tile being staged,
// the key ring, the value ring, the mbarriers, two item records and a few
// words.
template <int D>
struct Geo {
    static constexpr int kChunks = D / 64;                   // 128-byte chunks of a head row
    static constexpr int kQ = kChunks * kRows * 128;         // [chunk][row][128 B]
    static constexpr int kK = kChunks * kStepKeys * 128;     // [chunk][key][128 B]
    static constexpr int kVBlock = kChunks * kBS * 128;      // [chunk][token][128 B]
    static constexpr int kV = kStepBlocks * kVBlock;
    static constexpr int kOffK = kQ;
    static constexpr int kOffV = kOffK + kKStages * kK;
    static constexpr int kOffBar = kOffV + kVStages * kV;
    static constexpr int kBars = 2 + 2 + 1 + 1 + 2 * kKStages + 2 * kVStages + 1 + 1 + 2 + 2 + 1;
    static constexpr int kOffInfo = kOffBar + kBars * 8;
    static constexpr int kOffMisc = kOffInfo + 2 * static_cast<int>(sizeof(ItemInfo));
    static constexpr int kBytes = kOffMisc + 16;
};

int smem_bytes(int D) {
    return dec::kTileAlign + (D == 128 ? Geo<128>::kBytes : Geo<64>::kBytes);
}

// mbarrier addresses (shared space) by role
struct Bars {
    uint32_t b;
    // item records: published / read by every role
    __device__ uint32_t q_full(int s) const { return b + 8 * s; }
    __device__ uint32_t q_empty(int s) const { return b + 8 * (2 + s); }
    // the query tile in shared memory: landed / copied to tensor memory
    __device__ uint32_t qs_full() const { return b + 8 * 4; }
    __device__ uint32_t qs_empty() const { return b + 8 * 5; }
    __device__ uint32_t k_full(int s) const { return b + 8 * (6 + s); }
    __device__ uint32_t k_empty(int s) const { return b + 8 * (6 + kKStages + s); }
    __device__ uint32_t v_full(int s) const { return b + 8 * (6 + 2 * kKStages + s); }
    __device__ uint32_t v_empty(int s) const { return b + 8 * (6 + 2 * kKStages + kVStages + s); }
    static constexpr int kS = 6 + 2 * kKStages + 2 * kVStages;
    __device__ uint32_t s_full() const { return b + 8 * kS; }
    __device__ uint32_t s_free() const { return b + 8 * (kS + 1); }
    __device__ uint32_t p_full(int s) const { return b + 8 * (kS + 2 + s); }
    __device__ uint32_t pv_done(int s) const { return b + 8 * (kS + 4 + s); }
    __device__ uint32_t o_free() const { return b + 8 * (kS + 6); }
};

// arrivals that free an item record: the value producer, the two MMA warps
// and every softmax warp, once each has read it
constexpr int kQEmptyArrivals = 3 + kSoftmaxWarps;

// Every lane waits (bounded); false if any lane gave up.
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity));
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (the f32x2 forms of sm_100 and later: one instruction for
// two lanes' worth of fma or add) and the three-input maximum.

__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 f32x2_split(uint64_t r) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}

// a * b + c per lane, round to nearest
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Geometry of sequence s for this kernel; false if the sequence is not
// ours (too few rows) or invalid (recorded when `report`).
struct SeqGeo {
    int L, Q, q0, rows, tiles, parts;
};

__device__ __forceinline__ bool seq_geo(const ChunkParams &p, int s, int G, bool report,
                                        SeqGeo &sg) {
    const int L = __ldg(p.seq_lens + s);
    const int q0 = __ldg(p.query_start + s), q1 = __ldg(p.query_start + s + 1);
    const int Q = q1 - q0;
    if (L < 0 || L > p.max_blocks_per_seq * kBS || L > p.max_seq_len || Q < 0 || Q > L ||
        Q > p.max_query_len || q0 < 0 || q1 > p.num_query_tokens) {
        if (report) record_error(p.err, PKV_DEVERR_SEQ_LEN, s);
        return false;
    }
    sg.L = L;
    sg.Q = Q;
    sg.q0 = q0;
    sg.rows = Q * G;
    if (sg.rows < p.min_rows || sg.rows == 0) return false;
    sg.tiles = (sg.rows + kRows - 1) / kRows;
    sg.parts = (L + kPartTokens - 1) / kPartTokens;
    return true;
}

// First query tile that needs KV partition `part` (its last token reaches
// the partition): tile t's last token j_last(t) = (min(rows, 128(t+1)) - 1)/G
// sees keys up to L - Q + j_last(t).
__device__ __forceinline__ int first_tile(const SeqGeo &sg, int part, int G) {
    const int x = part * kPartTokens - (sg.L - sg.Q);  // j_last must reach x
    if (x <= 0) return 0;
    const int t = (x * G + 1 + kRows - 1) / kRows - 1;
    return min(sg.tiles - 1, max(0, t));
}

__device__ __forceinline__ int seq_items(const SeqGeo &sg, int G, int Hk) {
    int n = 0;
    for (int pt = 0; pt < sg.parts; ++pt) n += sg.tiles - first_tile(sg, pt, G);
    return n * Hk;
}

// One CTA: the list of the sequences this kernel takes and their item counts.
__global__ void __launch_bounds__(1024) chunk_plan_kernel(const __grid_constant__ ChunkParams p,
                                                          int G) {
    __shared__ int wsum[32];
    __shared__ int run[2];  // sequences listed, items listed
    // work of the two kernels of the call: key/value blocks the balanced
    // schedule streams, and 128-key steps of the tile kernel's items
    __shared__ unsigned long long dec_blocks;
    __shared__ float tile_steps;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        run[0] = run[1] = 0;
        dec_blocks = 0ull;
        tile_steps = 0.f;
    }
    __syncthreads();
    for (int s0 = 0; s0 < p.num_seqs; s0 += blockDim.x) {
        const int s = s0 + threadIdx.x;
        SeqGeo sg;
        const bool mine = s < p.num_seqs && seq_geo(p, s, G, true, sg);
        const int cnt = mine ? seq_items(sg, G, p.num_kv_heads) : 0;
        float my_steps = 0.f;
        unsigned long long my_dec = 0;
        if (mine) {
            // 128-key steps of the sequence's items, estimated in closed form:
            // tile t (128/G new tokens each, the last one clipped) sees
            // L - Q + min(Q, (t + 1) 128/G) keys, plus on average half a step
            // of rounding per (tile, partition) item
            const float R = static_cast<float>(kRows / G), nt = static_cast<float>(sg.tiles);
            const float keys = nt * static_cast<float>(sg.L - sg.Q) +
                               R * nt * (nt - 1.f) * 0.5f + static_cast<float>(sg.Q);
            my_steps = keys * (1.f / kStepKeys) * static_cast<float>(p.num_kv_heads) +
                       0.5f * static_cast<float>(cnt);
        } else if (s < p.num_seqs && p.max_cols > 0) {
            const int L = __ldg(p.seq_lens + s);
            const int Q = __ldg(p.query_start + s + 1) - __ldg(p.query_start + s);
            if (Q > 0 && Q <= L && Q * G <= p.max_cols && L <= p.max_blocks_per_seq * kBS)
                my_dec = static_cast<unsigned long long>((L + kBS - 1) / kBS);
        }
        // one shared atomic per warp and counter
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            my_steps += __shfl_xor_sync(0xffffffffu, my_steps, o);
            my_dec += __shfl_xor_sync(0xffffffffu, my_dec, o);
        }
        if (lane == 0 && my_steps > 0.f) atomicAdd(&tile_steps, my_steps);
        if (lane == 0 && my_dec) atomicAdd(&dec_blocks, my_dec);
        // two exclusive scans at once: (is listed, items) packed in one int2
        int a = mine ? 1 : 0, c = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ya = __shfl_up_sync(0xffffffffu, a, o);
            const int yc = __shfl_up_sync(0xffffffffu, c, o);
            if (lane >= o) {
                a += ya;
                c += yc;
            }
        }
        __shared__ int wa[32];
        if (lane == 31) {
            wa[warp] = a;
            wsum[warp] = c;
        }
        __syncthreads();
        if (warp == 0) {
            const int nw = blockDim.x >> 5;
            int va = lane < nw ? wa[lane] : 0, vc = lane < nw ? wsum[lane] : 0;
            int ia = va, ic = vc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int ya = __shfl_up_sync(0xffffffffu, ia, o);
                const int yc = __shfl_up_sync(0xffffffffu, ic, o);
                if (lane >= o) {
                    ia += ya;
                    ic += yc;
                }
            }
            if (lane < nw) {
                wa[lane] = ia - va;
                wsum[lane] = ic - vc;
            }
        }
        __syncthreads();
        const int ea = run[0] + wa[warp] + a - (mine ? 1 : 0);
        const int ec = run[1] + wsum[warp] + c - cnt;
        // launched as a programmatic dependent: the lengths and offsets above
        // may be read while the previous kernel (the cache write) finishes,
        // but nothing is written before it has completed -- which also makes
        // this kernel's completion imply that kernel's for the ones after it
        if (s0 == 0) grid_dependency_wait();
        if (mine) {
            p.big_seq[ea] = s;
            p.big_cum[ea] = ec;
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) {
            run[0] = ea + (mine ? 1 : 0);
            run[1] = ec + cnt;
        }
        __syncthreads();
    }
    grid_dependency_wait();  // (returns at once if the loop waited already)
    if (threadIdx.x == 0) {
        p.big_cum[run[0]] = run[1];
        *p.n_big = run[0];
        *p.work = 0;
    }
    // SMs for the balanced schedule: the split that evens the two kernels'
    // estimated times when they run side by side.  Decode: its bytes at
    // min(HBM rate, SMs x per-SM rate); tile: its steps at a per-step cost
    // over the remaining SMs, plus half an average item for the last wave.
    // Rates measured on this GPU (chunked prefill beside decodes: the decode
    // kernel streams ~58 GB/s per SM when it shares the GPU; a tile step
    // costs ~1-1.5 us beside it, 1.2-1.3 gave the shortest calls, 1.1 far
    // longer ones).  Thread i tries 2 + 2i SMs; the smallest estimate wins
    // (ties: fewer SMs).
    __shared__ unsigned long long best_w[32];
    unsigned long long key = ~0ull;
    if (dec_blocks > 0) {
        const int b = 2 + 2 * static_cast<int>(threadIdx.x);
        if (b < p.num_ctas) {
            const float dec_bytes = static_cast<float>(dec_blocks) * kBS * p.num_kv_heads *
                                    p.head_dim * 2 * 2;
            const float steps = tile_steps;
            const float items = fmaxf(1.f, static_cast<float>(run[1]));
            const float tail = 0.5f * __fdividef(steps, items) * kTileStepUs;
            const float t_dec = __fdividef(dec_bytes, fminf(kHbmBytesPerUs, b * kSmBytesPerUs));
            const float t_tile =
                __fdividef(steps * kTileStepUs, static_cast<float>(p.num_ctas - b)) + tail;
            // (non-negative floats order as their bits)
            key = (static_cast<unsigned long long>(__float_as_uint(fmaxf(t_dec, t_tile))) << 32) |
                  static_cast<unsigned>(b);
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, key, o);
        key = y < key ? y : key;
    }
    if (lane == 0) best_w[warp] = key;
    __syncthreads();
    if (warp == 0) {
        unsigned long long k = lane < static_cast<int>(blockDim.x >> 5) ? best_w[lane] : ~0ull;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const unsigned long long y = __shfl_xor_sync(0xffffffffu, k, o);
            k = y < k ? y : k;
        }
        if (lane == 0) *p.split = k == ~0ull ? 0 : static_cast<int>(k & 0xffffffffu);
    }
}

// Block ids of an item's partition: lane l holds blocks l, 32 + l, 64 + l and
// 96 + l of it; -1 past the item or out of range (recorded when `report`).
__device__ __forceinline__ void load_ids(const ChunkParams &p, int seq, int blo, int nblk,
                                         int lane, bool report, int (&ids)[kPartBlocks / 32]) {
#pragma unroll
    for (int w = 0; w < kPartBlocks / 32; ++w) {
        const int b = w * 32 + lane;
        int id = -1;
        if (b < nblk) {
            const int64_t at = static_cast<int64_t>(seq) * p.max_blocks_per_seq + blo + b;
            id = __ldg(p.block_tables + at);
            if (id < 0 || static_cast<int64_t>(id) >= p.num_blocks) {
                if (report) record_error(p.err, PKV_DEVERR_BLOCK_ID, at);
                id = -1;
            }
        }
        ids[w] = id;
    }
}

// Block b's id (every lane calls).
__device__ __forceinline__ int id_of(const int (&ids)[kPartBlocks / 32], int b) {
    int v = -1;
#pragma unroll
    for (int w = 0; w < kPartBlocks / 32; ++w) {
        const int x = __shfl_sync(0xffffffffu, ids[w], b & 31);
        if ((b >> 5) == w) v = x;
    }
    return v;
}

// The (partition, kv head, tile) of item `local` of a sequence: partition-
// major, then tile (the last first), then kv head.
__device__ __forceinline__ int3 decode_item(const SeqGeo &sg, int local, int G, int Hk) {
    for (int pt = 0; pt < sg.parts; ++pt) {
        const int t0 = first_tile(sg, pt, G);
        const int nt = sg.tiles - t0;
        // a partition's tiles longest first (a later tile sees more keys),
        // every KV head of a tile together, so the CTAs that finish first
        // take the short ones at the end
        if (local < nt * Hk) return make_int3(pt, local % Hk, sg.tiles - 1 - local / Hk);
        local -= nt * Hk;
    }
    return make_int3(-1, -1, -1);
}

// An item as the key producer takes it from the list (every lane holds the
// scalars; block ids are spread over the lanes).
struct Fetched {
    int done, seq, part, kvh, tile, nsteps, nblk, L, Q, q0, nparts;
    int ids[kPartBlocks / 32];
    uint32_t valid[kPartBlocks / 32];
};

__device__ __forceinline__ void fetch_item(const ChunkParams &p, int n_big, int total, int G,
                                           int logG, int lane, Fetched &f) {
    int item = 0;
    if (lane == 0) item = atomicAdd(p.work, 1);
    item = __shfl_sync(0xffffffffu, item, 0);
    f.done = item >= total;
    if (f.done) return;
    // the listed sequence holding the item (every lane searches alike)
    int lo = 0, hi = n_big - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldcg(p.big_cum + mid) <= item) lo = mid;
        else hi = mid - 1;
    }
    const int seq = __ldcg(p.big_seq + lo);
    SeqGeo sg;
    seq_geo(p, seq, G, false, sg);  // (the plan listed it: valid)
    const int3 d = decode_item(sg, item - __ldcg(p.big_cum + lo), G, p.num_kv_heads);
    const int j_last = (min(sg.rows, (d.z + 1) * kRows) - 1) >> logG;
    const int kv_end = sg.L - sg.Q + j_last + 1;  // keys [0, kv_end) for the tile
    const int k1 = min(kv_end, (d.x + 1) * kPartTokens);
    const int blo = d.x * kPartBlocks;
    f.seq = seq;
    f.part = d.x;
    f.kvh = d.y;
    f.tile = d.z;
    f.nblk = (k1 + kBS - 1) / kBS - blo;  // >= 1
    f.nsteps = (f.nblk + kStepBlocks - 1) / kStepBlocks;
    f.L = sg.L;
    f.Q = sg.Q;
    f.q0 = sg.q0;
    f.nparts = (kv_end + kPartTokens - 1) / kPartTokens;
    load_ids(p, seq, blo, f.nblk, lane, true, f.ids);
#pragma unroll
    for (int w = 0; w < kPartBlocks / 32; ++w) f.valid[w] = __ballot_sync(0xffffffffu, f.ids[w] >= 0);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_attention_kernel(const __grid_constant__ ChunkParams p) {
    using Gm = Geo<D>;
    constexpr int CH = Gm::kChunks;
    constexpr int DH = D / 2;  // the head dimensions (of O) each softmax thread owns
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((dec::kTileAlign - (smem_u32(smem_raw) & (dec::kTileAlign - 1))) &
                                (dec::kTileAlign - 1));
    const uint32_t sb = smem_u32(smem);
    const Bars br{sb + Gm::kOffBar};
    ItemInfo *info = reinterpret_cast<ItemInfo *>(smem + Gm::kOffInfo);
    // misc: [0] tensor-memory base
    volatile int *misc = reinterpret_cast<volatile int *>(smem + Gm::kOffMisc);

    const int Hk = p.num_kv_heads, H = p.num_heads;
    const int G = H / Hk, logG = __ffs(G) - 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(br.q_full(s), 1);
            mbar_init(br.q_empty(s), kQEmptyArrivals);
            mbar_init(br.p_full(s), kSoftmaxWarps);
            mbar_init(br.pv_done(s), 1);
        }
        mbar_init(br.qs_full(), 1);
        mbar_init(br.qs_empty(), 1);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(br.k_full(s), 1);
            mbar_init(br.k_empty(s), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(br.v_full(s), 1);
            mbar_init(br.v_empty(s), 1);
        }
        mbar_init(br.s_full(), 1);
        mbar_init(br.s_free(), kSoftmaxWarps);
        mbar_init(br.o_free(), kSoftmaxWarps);
        fence_mbarrier_init();
    }
    // the work list, the caches and the outputs are written by earlier
    // kernels of the stream
    grid_dependency_wait();
    // the last `split` CTAs leave their SMs to the balanced schedule
    if (static_cast<int>(blockIdx.x) >= static_cast<int>(gridDim.x) - __ldcg(p.split)) return;
    // the kernel launched next (the decode schedule's share of the call)
    // needs nothing from this one: let its CTAs take the SMs this grid leaves
    grid_launch_dependents();
    if (warp == 2) {
        tc::tmem_alloc(sb + Gm::kOffMisc, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = static_cast<uint32_t>(misc[0]);

    if (warp == 0) {
        // ===================== items, query tiles and keys =====================
        const int n_big = __ldcg(p.n_big);
        const int total = __ldcg(p.big_cum + n_big);
        int gs = 0;  // steps staged
        bool ok = true;
        Fetched cur;
        fetch_item(p, n_big, total, G, logG, lane, cur);
        for (int it = 0; ok; ++it) {
            const int slot = it & 1;
            if (it >= 2 && !wait_all(br.q_empty(slot), ((it >> 1) - 1) & 1)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                ItemInfo &in = info[slot];
                in.done = cur.done;
                if (!cur.done) {
                    in.seq = cur.seq;
                    in.part = cur.part;
                    in.kvh = cur.kvh;
                    in.tile = cur.tile;
                    in.nsteps = cur.nsteps;
                    in.nblk = cur.nblk;
                    in.L = cur.L;
                    in.Q = cur.Q;
                    in.q0 = cur.q0;
                    in.nparts = cur.nparts;
#pragma unroll
                    for (int w = 0; w < kPartBlocks / 32; ++w) in.valid[w] = cur.valid[w];
                }
                mbar_arrive(br.q_full(slot));
            }
            if (cur.done) break;
            // the query tile, into the staging buffer once the previous tile
            // has been copied to tensor memory
            if (it >= 1 && !wait_all(br.qs_empty(), (it - 1) & 1)) {
                ok = false;
                break;
            }
            if (lane == 0) mbar_arrive_expect_tx(br.qs_full(), Gm::kQ);
            __syncwarp();
            if (lane < CH)
                tensor_g2s_3d(sb + lane * (kRows * 128), &p.tm_q, 128 * lane, cur.kvh * G,
                              cur.q0 + cur.tile * (kRows >> logG), br.qs_full());
            // the next item is taken when this one's last steps are staged,
            // a ring's depth before its softmax ends: the CTAs that finish
            // first take the next items (its lookups overlap those steps)
            Fetched nxt;
            nxt.done = 1;
            const int fetch_at = max(cur.nsteps - kClaimLead, 0);
            for (int n = 0; n < cur.nsteps; ++n, ++gs) {
                const int ks = gs % kKStages;
                if (gs >= kKStages && !wait_all(br.k_empty(ks), ((gs / kKStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                const int nb = min(kStepBlocks, cur.nblk - n * kStepBlocks);
                if (lane == 0) mbar_arrive_expect_tx(br.k_full(ks), nb * CH * kBS * 128);
                __syncwarp();
                // lane l: block l / CH of the step, chunk l % CH (a bad block
                // reads rows before the cache: zeros)
                const int b = min(lane / CH, kStepBlocks - 1), c = lane % CH;
                const int id = id_of(cur.ids, n * kStepBlocks + b);
                if (lane < nb * CH)
                    tensor_g2s_3d(sb + Gm::kOffK + ks * Gm::kK + c * (kStepKeys * 128) +
                                      b * (kBS * 128),
                                  &p.tm_k, 0, id >= 0 ? id * kBS : -kBS, cur.kvh * CH + c,
                                  br.k_full(ks));
                if (n == fetch_at) fetch_item(p, n_big, total, G, logG, lane, nxt);
            }
            cur = nxt;
        }
        if (!ok) {
            if (lane == 0) record_error(p.err, PKV_DEVERR_TIMEOUT, blockIdx.x);
            // let the last copies land before the CTA can exit
            for (int s = 0; s < kKStages && s < gs; ++s) {
                const int last = gs - 1 - ((gs - 1 - s) % kKStages);
                mbar_wait_bounded(br.k_full(s), (last / kKStages) & 1);
            }
        }
    } else if (warp == 1) {
        // ================================ values ================================
        int gs = 0;
        bool ok = true;
        for (int it = 0; ok; ++it) {
            const int slot = it & 1;
            if (!wait_all(br.q_full(slot), (it >> 1) & 1)) {
                ok = false;
                break;
            }
            const ItemInfo &in = info[slot];
            const int done = in.done, seq = in.seq, part = in.part, kvh = in.kvh;
            const int nsteps = in.nsteps, nblk = in.nblk;
            __syncwarp();
            if (lane == 0) mbar_arrive(br.q_empty(slot));
            if (done) break;
            int ids[kPartBlocks / 32];
            load_ids(p, seq, part * kPartBlocks, nblk, lane, false, ids);
            for (int n = 0; n < nsteps; ++n, ++gs) {
                const int vs = gs % kVStages;
                if (gs >= kVStages && !wait_all(br.v_empty(vs), ((gs / kVStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                const int nb = min(kStepBlocks, nblk - n * kStepBlocks);
                if (lane == 0) mbar_arrive_expect_tx(br.v_full(vs), nb * Gm::kVBlock);
                __syncwarp();
                const int id = id_of(ids, n * kStepBlocks + min(lane, kStepBlocks - 1));
                if (lane < nb)
                    tensor_g2s_3d(sb + Gm::kOffV + vs * Gm::kV + lane * Gm::kVBlock, &p.tm_v, 0,
                                  id >= 0 ? id * kBS : -kBS, kvh * CH, br.v_full(vs));
            }
        }
        if (!ok) {
            if (lane == 0) record_error(p.err, PKV_DEVERR_TIMEOUT, blockIdx.x);
            for (int s = 0; s < kVStages && s < gs; ++s) {
                const int last = gs - 1 - ((gs - 1 - s) % kVStages);
                mbar_wait_bounded(br.v_full(s), (last / kVStages) & 1);
            }
        }
    } else if (warp == 2) {
        // ============================ score MMAs ============================
        // (one issuing thread; inside this kernel each MMA held its issuer
        // back ~110-140 cycles, so the scores and the P V products have one
        // issuing warp each and their chains overlap in the tensor pipe)
        int gs = 0;
        bool ok = true;
        for (int it = 0; ok; ++it) {
            const int slot = it & 1;
            if (!wait_all(br.q_full(slot), (it >> 1) & 1)) {
                ok = false;
                break;
            }
            const ItemInfo &in = info[slot];
            const int done = in.done, nsteps = in.nsteps, nblk = in.nblk;
            __syncwarp();
            if (lane == 0) mbar_arrive(br.q_empty(slot));
            if (done) break;
            // the query tile into tensor memory (the MMAs read A from there);
            // copies and MMAs of this thread run in issue order
            const uint32_t q_t = tmem + kTmemQ + 64 * slot;
            ok = wait_all(br.qs_full(), it & 1);
            if (!ok) break;
            tc::fence_after_sync();
            if (lane == 0) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc::cp_128x256b(q_t + 8 * kk,
                                    tc::smem_desc(sb + (kk >> 2) * (kRows * 128) + (kk & 3) * 32,
                                                  16, 1024, tc::kSwizzle128B));
                tc::commit(br.qs_empty());
            }
            __syncwarp();
            for (int n = 0; n < nsteps && ok; ++n) {
                const int g = gs + n, ks = g % kKStages;
                ok = wait_all(br.k_full(ks), (g / kKStages) & 1);
                // the softmax has read the previous step's scores
                if (ok && g >= 1) ok = wait_all(br.s_free(), (g - 1) & 1);
                if (!ok) break;
                tc::fence_after_sync();
                if (lane == 0) {
                    // one MMA per k step over the step's keys (an MMA of
                    // N 64 or less costs the issuing thread about as much as
                    // one of N 128, so fewer and wider ones are faster)
                    const int nb = min(kStepBlocks, nblk - n * kStepBlocks);
                    const uint32_t idesc = tc::idesc_f16_f32(kRows, nb * kBS, false, false);
                    const uint32_t k_s = sb + Gm::kOffK + ks * Gm::kK;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        tc::mma_ts(tmem + kTmemS, q_t + 8 * kk,
                                   tc::smem_desc(k_s + (kk >> 2) * (kStepKeys * 128) + (kk & 3) * 32,
                                                 16, 1024, tc::kSwizzle128B),
                                   idesc, kk > 0);
                    tc::commit(br.s_full());
                    tc::commit(br.k_empty(ks));
                }
                __syncwarp();
            }
            gs += nsteps;
        }
        if (!ok && lane == 0) record_error(p.err, PKV_DEVERR_TIMEOUT, blockIdx.x);
    } else if (warp == kPVWarp) {
        // ============================= P V MMAs =============================
        constexpr uint32_t kIdescPV = tc::idesc_f16_f32(kRows, D, false, true);
        int gs = 0;
        bool ok = true;
        for (int it = 0; ok; ++it) {
            const int slot = it & 1;
            if (!wait_all(br.q_full(slot), (it >> 1) & 1)) {
                ok = false;
                break;
            }
            const ItemInfo &in = info[slot];
            const int done = in.done, nsteps = in.nsteps, nblk = in.nblk, L = in.L;
            const int blo = in.part * kPartBlocks;
            __syncwarp();
            if (lane == 0) mbar_arrive(br.q_empty(slot));
            if (done) break;
            for (int m = 0; m < nsteps && ok; ++m) {
                const int g = gs + m, vs = g % kVStages;
                const int nb = min(kStepBlocks, nblk - m * kStepBlocks);
                ok = wait_all(br.v_full(vs), (g / kVStages) & 1);
                if (!ok) break;
                const uint32_t v_s = sb + Gm::kOffV + vs * Gm::kV;
                if (m == nsteps - 1) {
                    // value rows at and past the sequence end hold anything
                    // (their weights are 0, but 0 * NaN is not): zero them
                    const int t0 = L - (blo + m * kStepBlocks + nb - 1) * kBS;
                    if (t0 < kBS) {
                        const int units = (kBS - t0) * 8;  // 16-byte units per chunk
                        uint8_t *vb = smem + Gm::kOffV + vs * Gm::kV + (nb - 1) * Gm::kVBlock;
                        for (int i = lane; i < units * CH; i += 32) {
                            const int c = i / units, r = i % units;
                            *reinterpret_cast<uint4 *>(vb + c * (kBS * 128) +
                                                       (t0 + (r >> 3)) * 128 + (r & 7) * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                }
                ok = wait_all(br.p_full(g & 1), (g >> 1) & 1);
                // the previous item's O has been read out
                if (ok && m == 0 && it > 0) ok = wait_all(br.o_free(), (it - 1) & 1);
                if (!ok) break;
                tc::fence_after_sync();
                if (lane == 0) {
                    for (int b = 0; b < nb; ++b)
                        tc::mma_ts(tmem + kTmemO, tmem + kTmemP + 64 * (g & 1) + 8 * b,
                                   tc::smem_desc(v_s + b * Gm::kVBlock, kBS * 128, 1024,
                                                 tc::kSwizzle128B),
                                   kIdescPV, (m > 0 || b > 0) ? 1u : 0u);
                    tc::commit(br.pv_done(g & 1));
                    tc::commit(br.v_empty(vs));
                }
                __syncwarp();
            }
            gs += nsteps;
        }
        if (!ok && lane == 0) record_error(p.err, PKV_DEVERR_TIMEOUT, blockIdx.x);
    } else {
        // =============================== softmax ===============================
        // two threads per row: lane 16 h + i of warp 3 + 4 wh + q holds row
        // 32 q + 16 wh + i, keys 64 h .. of each step and head dimensions
        // DH h .. of O; a warp reaches tensor-memory lanes 32 * (warp % 4) ..
        const int wh = (warp - 3) >> 2;
        const int quarter = warp & 3;
        const int h = lane >> 4;
        const int r = quarter * 32 + wh * 16 + (lane & 15);
        const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32 + wh * 16) << 16);
        const int64_t Tq = p.num_query_tokens;
        const float sl2 = p.scale_log2;
        int gs = 0;
        bool ok = true;
        for (int it = 0; ok; ++it) {
            const int slot = it & 1;
            if (!wait_all(br.q_full(slot), (it >> 1) & 1)) {
                ok = false;
                break;
            }
            const ItemInfo &in = info[slot];
            const int done = in.done, seq = in.seq, part = in.part, kvh = in.kvh, tile = in.tile;
            const int nsteps = in.nsteps, nblk = in.nblk, L = in.L, Q = in.Q, q0 = in.q0;
            const int nparts = in.nparts;
            uint32_t valid[kPartBlocks / 32];
#pragma unroll
            for (int w = 0; w < kPartBlocks / 32; ++w) valid[w] = in.valid[w];
            // every block of the item in range (the usual case): the steps
            // need no look-up in the array above
            bool all_valid = true;
#pragma unroll
            for (int w = 0; w < kPartBlocks / 32; ++w) {
                const int nbw = min(max(nblk - 32 * w, 0), 32);
                const uint32_t need = nbw == 32 ? 0xffffffffu : ((1u << nbw) - 1u);
                all_valid = all_valid && (valid[w] & need) == need;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(br.q_empty(slot));
            if (done) break;
            const int rows = Q * G;
            const int rr = tile * kRows + r;
            const bool row_ok = rr < rows;
            const int j = rr >> logG;
            const int lim = row_ok ? L - Q + j : -1;  // last key position this row sees
            const int64_t orow = static_cast<int64_t>(q0 + j) * H + kvh * G + (rr & (G - 1));
            float m_used = kNegInf, l = 0.f;  // l: this thread's keys only

            for (int n = 0; n < nsteps; ++n) {
                const int g = gs + n;
                if (!wait_all(br.s_full(), g & 1)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                uint32_t sx[kGroupKeys];  // this row's scores of this thread's keys (fp32 bits)
#pragma unroll
                for (int c = 0; c < kGroupKeys / 32; ++c)
                    tc::ld32_halves<kGroupKeys>(tl + kTmemS + 32 * c,
                                                *reinterpret_cast<uint32_t(*)[32]>(sx + 32 * c));
                tc::wait_ld();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(br.s_free());
                const int nb = min(kStepBlocks, nblk - n * kStepBlocks);
                const int nbg = min(max(nb - 4 * h, 0), 4);  // this thread's blocks
                const int kbase = part * kPartTokens + n * kStepKeys + kGroupKeys * h;
                const int b0 = n * kStepBlocks + 4 * h;
                uint32_t vmask = 0xFu;
                if (!all_valid) vmask = (valid[b0 >> 5] >> (b0 & 31)) & 0xFu;
                // the maximum of the raw scores first (independent of the
                // masks, so the two overlap); it stands, scaled once, when
                // every key of the warp is visible and the scale is not
                // negative, else the scores are scaled and masked and their
                // maximum taken again
                const bool fast = __all_sync(0xffffffffu, nbg == 4 && vmask == 0xFu &&
                                                              kbase + kGroupKeys - 1 <= lim &&
                                                              sl2 >= 0.f);
                float mr[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mr[i] = kNegInf;
#pragma unroll
                for (int e = 0; e < kGroupKeys / 2; ++e)
                    mr[e & 7] = fmax3(mr[e & 7], __uint_as_float(sx[2 * e]),
                                      __uint_as_float(sx[2 * e + 1]));
                float mx = fmax3(fmax3(mr[0], mr[1], mr[2]), fmax3(mr[3], mr[4], mr[5]),
                                 fmaxf(mr[6], mr[7]));
                if (!fast) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) mr[i] = kNegInf;
#pragma unroll
                    for (int e = 0; e < kGroupKeys; ++e) {
                        const bool vis = e < nbg * kBS && ((vmask >> (e >> 4)) & 1u) && kbase + e <= lim;
                        const float t = vis ? __uint_as_float(sx[e]) * sl2 : kNegInf;
                        sx[e] = __float_as_uint(t);
                        mr[e & 7] = fmaxf(mr[e & 7], t);
                    }
                    mx = fmax3(fmax3(mr[0], mr[1], mr[2]), fmax3(mr[3], mr[4], mr[5]),
                               fmaxf(mr[6], mr[7]));
                } else {
                    mx *= sl2;
                }
                // the row's other half: the thread 16 lanes away
                const float mo = __shfl_xor_sync(0xffffffffu, mx, 16);
                const float m_new = fmaxf(m_used, fmaxf(mx, mo));
                const bool raise = m_new > m_used + kRescaleLog2;
                // O holds this item's earlier steps relative to m_used: rescale
                // this thread's columns before the reference moves (the
                // previous P V done first)
                const bool resc = raise && n > 0 && m_used != kNegInf;
                if (__any_sync(0xffffffffu, resc)) {
                    if (!wait_all(br.pv_done((g - 1) & 1), ((g - 1) >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const float alpha = resc ? ex2(m_used - m_new) : 1.f;
#pragma unroll
                    for (int c = 0; c < DH / 32; ++c) {
                        uint32_t x[32];
                        tc::ld32_halves<DH>(tl + kTmemO + 32 * c, x);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            x[e] = __float_as_uint(__uint_as_float(x[e]) * alpha);
                        tc::st32_halves<DH>(tl + kTmemO + 32 * c, x);
                    }
                    tc::wait_st();
                    l *= alpha;
                }
                if (raise) m_used = m_new;
                const float ms = m_used == kNegInf ? 0.f : m_used;
                // weights 2^(s * scale - m) (2^(t - m) for the masked scores),
                // fp16 pairs: column 32 h + i of the buffer holds keys
                // 64 h + 2i, 2i+1; the P V of two steps back must be done
                // with this buffer
                const float a = fast ? sl2 : 1.f;
                const int pb = g & 1;
                if (g >= 2) {
                    if (!wait_all(br.pv_done(pb), ((g - 2) >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                }
                // key pairs in packed fp32 lanes: one fma and one add per pair
                const uint64_t a2 = f32x2(a, a), nms2 = f32x2(-ms, -ms);
                uint64_t l2[4] = {0ull, 0ull, 0ull, 0ull};
                uint32_t x[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float2 t = f32x2_split(fma_f32x2(
                        f32x2(__uint_as_float(sx[2 * e]), __uint_as_float(sx[2 * e + 1])), a2, nms2));
                    const float p0 = ex2(t.x), p1 = ex2(t.y);
                    l2[e & 3] = add_f32x2(l2[e & 3], f32x2(p0, p1));
                    x[e] = pack_half2(p0, p1);
                }
                tc::st32_halves<32>(tl + kTmemP + 64 * pb, x);
                const float2 la = f32x2_split(add_f32x2(add_f32x2(l2[0], l2[1]), add_f32x2(l2[2], l2[3])));
                l += la.x + la.y;
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(br.p_full(pb));
            }
            if (!ok) break;
            gs += nsteps;

            // ---- the item's output: O / l, or the partial state (m, l, O),
            // this thread's head dimensions
            if (!wait_all(br.pv_done((gs - 1) & 1), ((gs - 1) >> 1) & 1)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            float o[DH];
            {
                uint32_t ob[DH];
#pragma unroll
                for (int c = 0; c < DH / 32; ++c)
                    tc::ld32_halves<DH>(tl + kTmemO + 32 * c,
                                        *reinterpret_cast<uint32_t(*)[32]>(ob + 32 * c));
                tc::wait_ld();
#pragma unroll
                for (int d = 0; d < DH; ++d) o[d] = __uint_as_float(ob[d]);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(br.o_free());
            l += __shfl_xor_sync(0xffffffffu, l, 16);  // the row's sum over both halves' keys
            if (nparts == 1) {
                if (row_ok) {
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * D + DH * h);
#pragma unroll
                    for (int c = 0; c < DH / 8; ++c)
                        dst[c] = make_uint4(pack_half2(o[8 * c] * inv, o[8 * c + 1] * inv),
                                            pack_half2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                            pack_half2(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                            pack_half2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
                }
                continue;
            }
            // partial state, dimension-major so the rows of a half-warp are
            // consecutive words; each half keeps its own copy of (m, l)
            const int64_t NR = Tq * H;
            const int64_t R = static_cast<int64_t>(kvh) * Tq * G + static_cast<int64_t>(q0) * G + rr;
            const int64_t parts_total = p.num_parts;
            float2 *ml = p.part_ml + h * parts_total * NR;
            if (row_ok) {
                ml[part * NR + R] = make_float2(m_used, l);
                float *dst = p.part_o + (static_cast<int64_t>(part) * D + DH * h) * NR + R;
#pragma unroll
                for (int d = 0; d < DH; ++d) dst[d * NR] = o[d];
            }
            // a ticket per (sequence, kv head, tile, softmax warp): the warp
            // that brings the last partition of its rows merges them.  The
            // warp barrier orders every lane's partial before lane 0's
            // releasing ticket; the last taker acquires the other
            // partitions' partials.
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                int *ticket = p.counters +
                              ((static_cast<int64_t>(seq) * Hk + kvh) * p.num_tiles + tile) *
                                  kSoftmaxWarps +
                              (warp - 3);
                last = atom_add_acq_rel_gpu(ticket, 1) == nparts - 1;
                // every partition has taken its ticket: leave the workspace zeroed
                if (last) st_relaxed_gpu(ticket, 0);
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            __syncwarp();  // memory order: lane 0's acquire before every lane's loads
            if (!last || !row_ok) continue;
            // the tile's last partition: merge every partition's partial row
            float M = kNegInf;
            for (int pp = 0; pp < nparts; ++pp) M = fmaxf(M, __ldcg(ml + pp * NR + R).x);
            float den = 0.f;
#pragma unroll
            for (int d = 0; d < DH; ++d) o[d] = 0.f;
            for (int pp = 0; pp < nparts; ++pp) {
                const float2 v = __ldcg(ml + pp * NR + R);
                const float w = v.x == kNegInf ? 0.f : ex2(v.x - M);
                den = fmaf(v.y, w, den);
                const float *src = p.part_o + (static_cast<int64_t>(pp) * D + DH * h) * NR + R;
#pragma unroll
                for (int d = 0; d < DH; ++d) o[d] = fmaf(__ldcg(src + d * NR), w, o[d]);
            }
            const float inv = den > 0.f ? 1.f / den : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * D + DH * h);
#pragma unroll
            for (int c = 0; c < DH / 8; ++c)
                dst[c] = make_uint4(pack_half2(o[8 * c] * inv, o[8 * c + 1] * inv),
                                    pack_half2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                    pack_half2(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                    pack_half2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
        }
        if (!ok && lane == 0) record_error(p.err, PKV_DEVERR_TIMEOUT, blockIdx.x);
    }

    // every role is done: hand the tensor memory back
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

using ChunkFn = void (*)(const ChunkParams);

ChunkFn select(int D) {
    if (D == 128) return chunk_attention_kernel<128>;
    if (D == 64) return chunk_attention_kernel<64>;
    return nullptr;
}

struct Sizes {
    int64_t tiles, parts, counters_bytes, ml_bytes, o_bytes, list_bytes;
    int col_tiles;          // balanced schedule's column n-tiles (0: not used)
    dec::BalancedShape bal;  // its shape (workspace first in the scratch)
    int64_t bal_bytes;
};

Sizes sizes(int64_t S, int64_t H, int64_t Hk, int64_t D, int64_t Tq, int64_t max_q,
            int64_t max_len) {
    Sizes z{};
    const int64_t G = H / Hk;
    z.tiles = std::max<int64_t>(1, (max_q * G + kRows - 1) / kRows);
    z.parts = std::max<int64_t>(1, (max_len + kPartTokens - 1) / kPartTokens);
    z.counters_bytes = dec::align256(S * Hk * z.tiles * kSoftmaxWarps * 4);  // per softmax warp
    z.list_bytes = dec::align256((2 * S + 4) * 4);  // big_seq, big_cum, n_big, work, split
    z.ml_bytes = z.parts > 1 ? dec::align256(2 * z.parts * Tq * H * 8) : 0;  // per group
    z.o_bytes = z.parts > 1 ? z.parts * Tq * H * D * 4 : 0;
    // the balanced schedule takes the chunks of up to 8 query rows, or of up
    // to 16 when no chunk needs the tile kernel (one column tile is the
    // cheaper policy, so it is used whenever the tile kernel runs anyway)
    z.col_tiles = (max_q * G <= 8 || max_q * G > 16) ? 1 : 2;
    z.bal = dec::balanced_shape(static_cast<int>(S), static_cast<int>(Hk), static_cast<int>(G),
                                static_cast<int>(D), sm_count(), false, 8 * z.col_tiles);
    if (!z.bal.ok) z.col_tiles = 0;
    z.bal_bytes = z.bal.ok ? dec::align256(z.bal.workspace) : 0;
    return z;
}

}  // namespace
}  // namespace chunk
}  // namespace pkv

extern "C" size_t pkv_chunk_workspace_bytes(int32_t num_seqs, int32_t num_heads,
                                            int32_t num_kv_heads, int32_t head_dim,
                                            int32_t num_query_tokens, int32_t max_query_len,
                                            int32_t max_seq_len) {
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        num_heads % num_kv_heads != 0 || num_query_tokens < 0 || max_query_len <= 0 ||
        max_seq_len <= 0)
        return 0;
    const auto z = pkv::chunk::sizes(num_seqs, num_heads, num_kv_heads, head_dim,
                                     num_query_tokens, max_query_len, max_seq_len);
    return static_cast<size_t>(z.bal_bytes + z.list_bytes + z.counters_bytes + z.ml_bytes +
                               z.o_bytes);
}

extern "C" int pkv_chunk_attention(void *out, const void *q, const void *k_cache,
                                   const void *v_cache, const int32_t *block_tables,
                                   const int32_t *seq_lens, const int32_t *query_start,
                                   float scale, int32_t num_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size, int32_t num_seqs,
                                   int32_t max_blocks_per_seq, int32_t num_query_tokens,
                                   int32_t max_query_len, int32_t max_seq_len,
                                   int64_t num_blocks, void *workspace, size_t workspace_bytes,
                                   pkv_stream_t stream) {
    using namespace pkv;
    using namespace pkv::chunk;
    if (num_seqs < 0 || num_query_tokens < 0) return PKV_ERR_INVALID;
    if (num_seqs == 0 || num_query_tokens == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start)
        return PKV_ERR_NULL;
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || max_query_len <= 0 ||
        max_seq_len <= 0 || !std::isfinite(scale))
        return PKV_ERR_INVALID;
    const int G = num_heads / num_kv_heads;
    if (!(G == 1 || G == 2 || G == 4 || G == 8)) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != kBS) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(query_start, 4) ||
        (workspace != nullptr && !aligned(workspace, 16)))
        return PKV_ERR_ALIGNMENT;
    const auto z = sizes(num_seqs, num_heads, num_kv_heads, head_dim, num_query_tokens,
                         max_query_len, max_seq_len);
    // work items (and their prefix sums) are 32-bit: at most
    // (sum of tiles <= Tq*G/64 + S) * partitions * Hk of them
    const int64_t tiles_sum = (static_cast<int64_t>(num_query_tokens) * G + kRows - 1) / kRows +
                              num_seqs;
    if (tiles_sum * z.parts * num_kv_heads > INT32_MAX || z.tiles > INT32_MAX)
        return PKV_ERR_UNSUPPORTED;
    const int64_t need = z.bal_bytes + z.list_bytes + z.counters_bytes + z.ml_bytes + z.o_bytes;
    if (workspace == nullptr || static_cast<int64_t>(workspace_bytes) < need)
        return PKV_ERR_WORKSPACE;
    ChunkFn fn = select(head_dim);
    if (fn == nullptr) return PKV_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const float scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    const int row_bytes = num_kv_heads * head_dim * 2;

    // ---- chunks of up to 8 * col_tiles query rows: the balanced schedule,
    // launched after the tile kernel (below) when there are long chunks too
    int min_rows = 1;
    bool use_bal = false;
    dec::BalancedParams b{};
    // (the balanced schedule indexes the flattened block list in 32 bits)
    if (z.col_tiles > 0 && static_cast<int64_t>(num_seqs) * max_blocks_per_seq <= INT32_MAX) {
        b.out = static_cast<__half *>(out);
        b.q = static_cast<const __half *>(q);
        b.k_cache = static_cast<const __half *>(k_cache);
        b.v_cache = static_cast<const __half *>(v_cache);
        b.block_tables = block_tables;
        b.seq_lens = seq_lens;
        b.scale_log2 = scale_log2;
        b.num_seqs = num_seqs;
        b.num_heads = num_heads;
        b.num_kv_heads = num_kv_heads;
        b.max_blocks_per_seq = max_blocks_per_seq;
        b.num_blocks = num_blocks;
        b.query_start = query_start;
        b.max_cols = 8 * z.col_tiles;
        b.num_query_tokens = num_query_tokens;
        const int st = dec::setup_balanced(b, z.bal, b.max_cols, ws, k_cache, v_cache);
        if (st != PKV_OK) return st;
        b.err = device_error_record();
        if (b.err == nullptr) return PKV_ERR_CUDA;
        min_rows = b.max_cols + 1;
        if (static_cast<int64_t>(max_query_len) * G < min_rows)  // no long chunks
            return dec::launch_balanced(b, z.bal, head_dim, G, false, false, s, z.col_tiles);
        use_bal = true;
    }

    // ---- the larger chunks: query tiles of 128 rows
    ChunkParams p{};
    p.out = static_cast<__half *>(out);
    p.q = static_cast<const __half *>(q);
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.query_start = query_start;
    p.scale_log2 = scale_log2;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_query_len = max_query_len;
    p.max_seq_len = max_seq_len;
    p.num_tiles = static_cast<int>(z.tiles);
    p.num_parts = static_cast<int>(z.parts);
    p.num_query_tokens = num_query_tokens;
    p.min_rows = min_rows;
    p.num_blocks = num_blocks;
    uint8_t *cws = ws + z.bal_bytes;
    p.num_seqs = num_seqs;
    p.big_seq = reinterpret_cast<int *>(cws);
    p.big_cum = p.big_seq + num_seqs;
    p.n_big = p.big_cum + num_seqs + 1;
    p.work = p.n_big + 1;
    p.split = p.work + 1;
    p.head_dim = head_dim;
    p.max_cols = use_bal ? b.max_cols : 0;
    cws += z.list_bytes;
    p.counters = reinterpret_cast<int *>(cws);
    p.part_ml = reinterpret_cast<float2 *>(cws + z.counters_bytes);
    p.part_o = reinterpret_cast<float *>(cws + z.counters_bytes + z.ml_bytes);
    {
        // keys: one 128-byte chunk per copy; values: the head's chunks (a
        // head's head_dim * 2 bytes are whole 128-byte chunks); query rows
        const int chunks = head_dim * 2 / 128;
        int st = dec::make_kv_tensor_map(&p.tm_k, k_cache, num_blocks, row_bytes, 1);
        if (st == PKV_OK)
            st = dec::make_kv_tensor_map(&p.tm_v, v_cache, num_blocks, row_bytes, chunks);
        if (st == PKV_OK)
            st = dec::make_q_tensor_map(&p.tm_q, q, num_query_tokens, num_heads, head_dim, G);
        if (st != PKV_OK) return st;
    }
    p.err = device_error_record();
    if (p.err == nullptr) return PKV_ERR_CUDA;

    // the work list (one CTA), then persistent CTAs that pull from it
    const int smem = smem_bytes(head_dim);
    int per_sm = 0;
    {
        const int st = prepare_kernel(reinterpret_cast<const void *>(fn), kThreads, smem, &per_sm);
        if (st != PKV_OK) return st;
    }
    p.num_ctas = std::max(1, sm_count() * std::max(1, per_sm));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t pcfg = {};
    pcfg.gridDim = dim3(1);
    pcfg.blockDim = dim3(1024);
    pcfg.stream = s;
    pcfg.attrs = attr;
    pcfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&pcfg, chunk_plan_kernel, p, G);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_failure(e, "chunk plan launch");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.num_ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fn, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_failure(e, "chunk attention launch");
    if (!use_bal) return PKV_OK;
    // the short chunks: their CTAs start as the tile kernel's leave (it
    // allows dependents at its start); the caches were written before the
    // plan kernel completed (it waits for the previous kernel), and the two
    // kernels write disjoint rows and scratch, so this grid waits for the
    // tile kernel only before it exits
    b.defer_wait = 1;
    b.active_ctas = p.split;  // its ranges over the SMs the plan left it
    return dec::launch_balanced(b, z.bal, head_dim, G, false, false, s, z.col_tiles);
}
