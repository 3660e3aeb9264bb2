// pkv_chunk.cu -- attention of a chunk of new tokens per sequence over the
// paged cache, causal within the new tokens ("vLLM 技术内幕" §3.2: chunked
// prefill, prompt and output tokens scheduled alike; §7.4: draft tokens
// verified together).  Sequence i holds L tokens, the last Q of them new;
// new token j (position L - Q + j) attends to positions 0 .. L - Q + j.
//
// Sequences whose new tokens times the group size fit the balanced decode
// schedule's query columns (8 or 16: MmaColsPolicy) run there -- the same
// streaming of whole token rows as a decode; the others run here.
//
// The work is a list of items (query tile of 64 rows, KV head, KV
// partition of 2048 tokens, sequence), built on the device by a one-CTA plan
// kernel for the sequences this kernel takes (partitions past a tile's
// causal range are not items).  Persistent CTAs (two per SM) pull items in
// list order from an atomic counter, so tiles with more keys and tiles with
// fewer balance out.  A row is (new token j, query head g of the KV head's
// group): row = j*G + g, so a tile covers 64/G consecutive new tokens.  Four
// consumer warps own 16 rows each; a producer warp stages the partition's
// blocks -- two per stage, each block one tensor copy (TMA) of the head's
// 16 key rows and one of its 16 value rows -- into a 4-deep ring.  Per stage
// (32 keys) a warp computes S = Q K^T (m16n8k16: rows = query rows, columns
// = tokens), masks the keys past each row's position, folds the 32 keys into
// each row's online softmax (log2 domain) and accumulates O += P V, the
// weights taken straight from the score fragments.  A tile whose causal range fits one
// partition writes fp16 out; otherwise every partition leaves fp32 partial
// states and the last CTA of the tile to take a ticket merges them with a
// log-sum-exp rescale.  No CTA waits for another.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "/root/repo/include/pagedkv.h"
#include "pkv_decode_common.cuh"
#include "pkv_decode_host.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace chunk {
namespace {

using dec::kBS;
using dec::kNegInf;
using dec::SwizzledTile;

constexpr int kRows = 64;                 // query rows per CTA
constexpr int kWarps = 4;                 // consumer warps, 16 rows each
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kStages = 4;
constexpr int kBlocksPerStage = 2;
constexpr int kPartTokens = 2048;         // KV partition
constexpr int kPartBlocks = kPartTokens / kBS;

struct ChunkParams {
    CUtensorMap tm_k;  // per-head boxes of the key / value caches
    CUtensorMap tm_v;
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
    int num_tiles;  // grid.x
    int num_query_tokens;
    int min_rows;   // sequences with fewer rows (new tokens x group) are not ours
    int num_seqs;
    // work list: the sequences taken here (big_seq[k]) and the exclusive
    // prefix of their item counts (big_cum[k], big_cum[n_big] = total items);
    // *work is the next item to hand out
    int *big_seq;
    int *big_cum;
    int *n_big;
    int *work;
    int64_t num_blocks;
    int *counters;    // [S][Hk][num_tiles] tickets, zero between calls
    float2 *part_ml;  // [parts][Tq][H] (m, l)
    float *part_o;    // [parts][Tq][H][D]
    ErrorRecord *err;
};

template <int D>
struct Geo {
    static constexpr int kTile = kBS * D * 2;  // one block's K (or V) slice of one head
    static constexpr int kStage = 2 * kBlocksPerStage * kTile;
    static constexpr int kRing = kStages * kStage;
};

constexpr int kMisc = 8;  // ints of CTA-wide scratch

int smem_bytes(int D) {
    const int tile = kBS * D * 2;
    return dec::kTileAlign + kStages * 2 * kBlocksPerStage * tile + 2 * kStages * 8 +
           kPartBlocks * 4 + kMisc * 4;
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
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
// the partition): tile t's last token j_last(t) = (min(rows, 64(t+1)) - 1)/G
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
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) run[0] = run[1] = 0;
    __syncthreads();
    for (int s0 = 0; s0 < p.num_seqs; s0 += blockDim.x) {
        const int s = s0 + threadIdx.x;
        SeqGeo sg;
        const bool mine = s < p.num_seqs && seq_geo(p, s, G, true, sg);
        const int cnt = mine ? seq_items(sg, G, p.num_kv_heads) : 0;
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
    if (threadIdx.x == 0) {
        p.big_cum[run[0]] = run[1];
        *p.n_big = run[0];
        *p.work = 0;
    }
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 2)
    chunk_attention_kernel(const __grid_constant__ ChunkParams p) {
    using Gm = Geo<D>;
    constexpr int KS = D / 16;  // k-steps of S = Q K^T
    constexpr int NT = D / 8;   // n-tiles of O
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((dec::kTileAlign - (smem_u32(smem_raw) & (dec::kTileAlign - 1))) &
                                (dec::kTileAlign - 1));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Gm::kRing);
    uint64_t *empty = full + kStages;
    int *bt_s = reinterpret_cast<int *>(empty + kStages);
    // misc: [0] last-contributor flag, [1] failure flag, [2..7] current item
    // (sequence, partition, kv head, tile, valid)
    int *misc = bt_s + kPartBlocks;

    const int Hk = p.num_kv_heads, H = p.num_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kWarps);
        }
        fence_mbarrier_init();
        misc[1] = 0;
    }
    // the work list, the caches and the outputs are all written by earlier
    // kernels of the stream
    grid_dependency_wait();
    __syncthreads();
    const int n_big = __ldcg(p.n_big);
    const int total = __ldcg(p.big_cum + n_big);
    const uint32_t ring_s = smem_u32(smem);
    const uint32_t full_s = smem_u32(full), empty_s = smem_u32(empty);
    const SwizzledTile tl{7u};
    int gstep = 0;  // ring steps run by this CTA so far (stage and phase of the next)

    for (;;) {
        if (threadIdx.x == 0) {
            const int item = atomicAdd(p.work, 1);
            int valid = item < total && !misc[1];
            if (valid) {
                // the listed sequence holding the item, then its (partition,
                // kv head, tile): partition-major, then kv head, then tile
                int lo = 0, hi = n_big - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (__ldcg(p.big_cum + mid) <= item) lo = mid;
                    else hi = mid - 1;
                }
                const int s = __ldcg(p.big_seq + lo);
                int local = item - __ldcg(p.big_cum + lo);
                SeqGeo sg;
                valid = seq_geo(p, s, G, false, sg);
                int part = 0, kv = 0, tile = 0;
                for (int pt = 0; valid && pt < sg.parts; ++pt) {
                    const int t0 = first_tile(sg, pt, G);
                    const int nt = sg.tiles - t0;
                    if (local < nt * Hk) {
                        part = pt;
                        kv = local / nt;
                        tile = t0 + local % nt;
                        break;
                    }
                    local -= nt * Hk;
                }
                misc[2] = s;
                misc[3] = part;
                misc[4] = kv;
                misc[5] = tile;
            }
            misc[6] = valid;
        }
        __syncthreads();
        if (!misc[6]) break;
        const int seq = misc[2], part = misc[3], kvh = misc[4], tile = misc[5];
        SeqGeo sg;
        seq_geo(p, seq, G, false, sg);
        const int L = sg.L, Q = sg.Q, q0 = sg.q0, rows = sg.rows;
        const int j_last = (min(rows, (tile + 1) * kRows) - 1) / G;
        const int kv_end = L - Q + j_last + 1;  // keys [0, kv_end) for this tile
        const int nparts = (kv_end + kPartTokens - 1) / kPartTokens;
        const int k0 = part * kPartTokens;
        const int k1 = min(kv_end, k0 + kPartTokens);
        const int blo = k0 / kBS;
        const int nblk = (k1 + kBS - 1) / kBS - blo;  // >= 1
        const int nsteps = (nblk + kBlocksPerStage - 1) / kBlocksPerStage;
        const int head_chunk = kvh * (D * 2 / 128);

        // the partition's block ids, checked
        for (int b = threadIdx.x; b < nblk; b += kThreads) {
            int id = __ldg(p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq + blo + b);
            if (id < 0 || static_cast<int64_t>(id) >= p.num_blocks) {
                record_error(p.err, PKV_DEVERR_BLOCK_ID,
                             static_cast<int64_t>(seq) * p.max_blocks_per_seq + blo + b);
                id = -1;
            }
            bt_s[b] = id;
        }
        __syncthreads();

        if (warp == kWarps) {
            // ============================== producer ==============================
            for (int i = 0; i < nsteps; ++i) {
                const int gi = gstep + i;
                const int st = gi % kStages;
                if (gi >= kStages) {
                    const bool free_ =
                        mbar_wait_bounded(empty_s + st * 8, ((gi / kStages) - 1) & 1);
                    if (!__all_sync(0xffffffffu, free_)) {
                        if (lane == 0) {
                            record_error(p.err, PKV_DEVERR_TIMEOUT, blockIdx.x);
                            atomicOr(&misc[1], 1);
                        }
                        break;
                    }
                }
                const int nb = min(kBlocksPerStage, nblk - i * kBlocksPerStage);
                int ncopy = 0;
                for (int k = 0; k < nb; ++k) ncopy += bt_s[i * kBlocksPerStage + k] >= 0 ? 1 : 0;
                if (lane == 0)
                    mbar_arrive_expect_tx(full_s + st * 8,
                                          static_cast<uint32_t>(ncopy) * 2u * Gm::kTile);
                __syncwarp();
                // lanes 0, 1: key tiles of the stage's blocks; lanes 2, 3: value tiles
                const int k = lane % kBlocksPerStage;
                const bool value = lane >= kBlocksPerStage;
                if (lane < 2 * kBlocksPerStage && k < nb) {
                    const int id = bt_s[i * kBlocksPerStage + k];
                    if (id >= 0)
                        tensor_g2s_3d(ring_s + st * Gm::kStage +
                                          (value ? kBlocksPerStage + k : k) * Gm::kTile,
                                      value ? &p.tm_v : &p.tm_k, 0, id * kBS, head_chunk,
                                      full_s + st * 8);
                }
            }
        } else {
            // ============================== consumers ==============================
            const int g = lane >> 2, t = lane & 3;
            int lim[2];
            int64_t orow[2];  // (query row * H + head) of each of the lane's two rows, or -1
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int rr = tile * kRows + warp * 16 + g + 8 * r;
                if (rr < rows) {
                    const int j = rr / G;
                    lim[r] = L - Q + j;  // last key position it sees
                    orow[r] = static_cast<int64_t>(q0 + j) * H + kvh * G + rr % G;
                } else {
                    lim[r] = -1;
                    orow[r] = -1;
                }
            }
            int wlim = max(lim[0], lim[1]);  // the largest key position this warp sees
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                wlim = max(wlim, __shfl_xor_sync(0xffffffffu, wlim, o));
            uint32_t qa[KS][4];
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (orow[r] >= 0) {
                        const uint32_t *src =
                            reinterpret_cast<const uint32_t *>(p.q + orow[r] * D + kk * 16);
                        qa[kk][r] = __ldg(src + t);
                        qa[kk][2 + r] = __ldg(src + 4 + t);
                    } else {
                        qa[kk][r] = qa[kk][2 + r] = 0u;
                    }
                }
            }
            float o[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
            float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};
            const int ktok = (lane & 7) + (lane >> 4) * 8;
            const uint32_t kcol = ((lane >> 3) & 1) * 16;
            const int vtok = (lane & 7) + ((lane >> 3) & 1) * 8;
            const uint32_t vcol = (lane >> 4) * 16;

            bool ok = true;
            for (int i = 0; i < nsteps; ++i) {
                const int gi = gstep + i;
                const int st = gi % kStages;
                const bool landed = mbar_wait_bounded(full_s + st * 8, (gi / kStages) & 1);
                if (!__all_sync(0xffffffffu, landed)) {
                    ok = false;
                    break;
                }
                const int nb = min(kBlocksPerStage, nblk - i * kBlocksPerStage);
                // the stage's blocks in one softmax step (2 x 16 keys): which
                // of them this warp needs (warp-uniform), and where they start
                bool use[kBlocksPerStage];
                int kps[kBlocksPerStage];
                bool any = false;
#pragma unroll
                for (int k = 0; k < kBlocksPerStage; ++k) {
                    kps[k] = (blo + i * kBlocksPerStage + k) * kBS;
                    use[k] = k < nb && bt_s[i * kBlocksPerStage + k] >= 0 && kps[k] <= wlim;
                    any = any || use[k];
                }
                if (any) {
                    const uint32_t stage = ring_s + st * Gm::kStage;
                    // S = Q K^T for both blocks: n-tiles (block k, tokens 0-7 / 8-15)
                    float sc[kBlocksPerStage][2][4];
#pragma unroll
                    for (int k = 0; k < kBlocksPerStage; ++k)
#pragma unroll
                        for (int n = 0; n < 2; ++n)
#pragma unroll
                            for (int e = 0; e < 4; ++e) sc[k][n][e] = 0.f;
#pragma unroll
                    for (int k = 0; k < kBlocksPerStage; ++k) {
                        if (!use[k]) continue;
                        const uint32_t kb = stage + k * Gm::kTile;
#pragma unroll
                        for (int kk = 0; kk < KS; ++kk) {
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4(b0, b1, b2, b3, kb + tl.at(ktok, kcol + kk * 32));
                            mma_16816(sc[k][0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                            mma_16816(sc[k][1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
                        }
                    }
                    // element e of n-tile n of block k: row g (e < 2) or g+8,
                    // key position kps[k] + 8n + 2t + (e & 1)
                    float mx[2] = {kNegInf, kNegInf};
#pragma unroll
                    for (int k = 0; k < kBlocksPerStage; ++k)
#pragma unroll
                        for (int n = 0; n < 2; ++n)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int r = e >> 1;
                                const int pos = kps[k] + 8 * n + 2 * t + (e & 1);
                                sc[k][n][e] = use[k] && pos <= lim[r] ? sc[k][n][e] * p.scale_log2
                                                                      : kNegInf;
                                mx[r] = fmaxf(mx[r], sc[k][n][e]);
                            }
                    float alpha[2], msafe[2];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                        const float mnew = fmaxf(m[r], mx[r]);
                        // a row with no visible key yet keeps m = -inf, l = 0, o = 0
                        msafe[r] = mnew == kNegInf ? 0.f : mnew;
                        alpha[r] = exp2f(m[r] - msafe[r]);
                        m[r] = mnew;
                    }
                    // weights, rounded to fp16 as the MMA applies them: the A
                    // fragments of P V, one k-step per block
                    uint32_t pa[kBlocksPerStage][4];
                    float lsum[2] = {0.f, 0.f};
#pragma unroll
                    for (int k = 0; k < kBlocksPerStage; ++k)
#pragma unroll
                        for (int n = 0; n < 2; ++n)
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const uint32_t h2 =
                                    pack_half2(exp2f(sc[k][n][2 * r] - msafe[r]),
                                               exp2f(sc[k][n][2 * r + 1] - msafe[r]));
                                pa[k][2 * n + r] = h2;
                                const float2 u = unpack_half2(h2);
                                lsum[r] += u.x + u.y;
                            }
#pragma unroll
                    for (int r = 0; r < 2; ++r) l[r] = l[r] * alpha[r] + lsum[r];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        o[nt][0] *= alpha[0];
                        o[nt][1] *= alpha[0];
                        o[nt][2] *= alpha[1];
                        o[nt][3] *= alpha[1];
                    }
#pragma unroll
                    for (int k = 0; k < kBlocksPerStage; ++k) {
                        if (!use[k]) continue;
                        const uint32_t vb = stage + (kBlocksPerStage + k) * Gm::kTile;
                        // value rows past the sequence end hold anything (their
                        // weights are 0, but 0 * NaN is not): every warp zeroes
                        // them before use (the same zeros, so the writes agree)
                        if (kps[k] + kBS > L) dec::zero_tail_rows<D>(vb, tl, 0u, L - kps[k], lane);
                        // O += P V; per transposed ldmatrix: tokens 0-7 / 8-15
                        // of dims 0-7, then of dims 8-15
#pragma unroll
                        for (int nd = 0; nd < D / 16; ++nd) {
                            uint32_t v0, v1, v2, v3;
                            ldsm_x4_trans(v0, v1, v2, v3, vb + tl.at(vtok, vcol + nd * 32));
                            mma_16816(o[2 * nd], pa[k][0], pa[k][1], pa[k][2], pa[k][3], v0, v1);
                            mma_16816(o[2 * nd + 1], pa[k][0], pa[k][1], pa[k][2], pa[k][3], v2,
                                      v3);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_s + st * 8);
            }
            if (!ok && lane == 0) {
                record_error(p.err, PKV_DEVERR_TIMEOUT, blockIdx.x);
                atomicOr(&misc[1], 1);
            }

            // normaliser of each row (its four lanes hold parts of it)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
                l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
            }
            if (nparts == 1) {
                if (ok) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        if (orow[r] < 0) continue;
                        const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
                        __half *dst = p.out + orow[r] * D + 2 * t;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            *reinterpret_cast<__half2 *>(dst + 8 * nt) =
                                __floats2half2_rn(o[nt][2 * r] * inv, o[nt][2 * r + 1] * inv);
                    }
                }
            } else {
                // partial state of this partition, then the ticket
                const int64_t Tq = p.num_query_tokens;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (orow[r] < 0) continue;
                    const int64_t idx = static_cast<int64_t>(part) * Tq * H + orow[r];
                    if (t == 0) p.part_ml[idx] = make_float2(m[r], l[r]);
                    float *dst = p.part_o + idx * D + 2 * t;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        *reinterpret_cast<float2 *>(dst + 8 * nt) =
                            make_float2(o[nt][2 * r], o[nt][2 * r + 1]);
                }
                __threadfence();
                named_barrier(1, kWarps * 32);
                if (threadIdx.x == 0) {
                    int *ticket =
                        p.counters + (static_cast<int64_t>(seq) * Hk + kvh) * p.num_tiles + tile;
                    __threadfence();
                    const int prev = atomicAdd(ticket, 1);
                    const int last = prev == nparts - 1;
                    if (last) {
                        atomicExch(ticket, 0);  // leave the workspace zeroed
                        __threadfence();
                    }
                    misc[0] = last;
                }
                named_barrier(1, kWarps * 32);
                if (misc[0]) {
                    // last partition of the tile: merge every partition's
                    // partial rows (this warp's 16 rows; lanes over head dims)
                    constexpr int DPL = D / 32;
                    for (int rr = 0; rr < 16; ++rr) {
                        const int rw = tile * kRows + warp * 16 + rr;
                        if (rw >= rows) break;
                        const int64_t orw = static_cast<int64_t>(q0 + rw / G) * H + kvh * G + rw % G;
                        float M = kNegInf;
                        for (int pp = 0; pp < nparts; ++pp)
                            M = fmaxf(M, __ldcg(p.part_ml + static_cast<int64_t>(pp) * Tq * H + orw).x);
                        float den = 0.f, acc[DPL];
#pragma unroll
                        for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
                        for (int pp = 0; pp < nparts; ++pp) {
                            const int64_t idx = static_cast<int64_t>(pp) * Tq * H + orw;
                            const float2 ml = __ldcg(p.part_ml + idx);
                            const float w = ml.x == kNegInf ? 0.f : exp2f(ml.x - M);
                            den = fmaf(ml.y, w, den);
                            const float *src = p.part_o + idx * D + lane * DPL;
                            if constexpr (DPL == 4) {
                                const float4 v = __ldcg(reinterpret_cast<const float4 *>(src));
                                acc[0] = fmaf(v.x, w, acc[0]);
                                acc[1] = fmaf(v.y, w, acc[1]);
                                acc[2] = fmaf(v.z, w, acc[2]);
                                acc[3] = fmaf(v.w, w, acc[3]);
                            } else {
                                const float2 v = __ldcg(reinterpret_cast<const float2 *>(src));
                                acc[0] = fmaf(v.x, w, acc[0]);
                                acc[1] = fmaf(v.y, w, acc[1]);
                            }
                        }
                        const float inv = den > 0.f ? 1.f / den : 0.f;
                        __half *dst = p.out + orw * D + lane * DPL;
#pragma unroll
                        for (int i = 0; i < DPL; i += 2)
                            *reinterpret_cast<__half2 *>(dst + i) =
                                __floats2half2_rn(acc[i] * inv, acc[i + 1] * inv);
                    }
                }
            }
        }
        gstep += nsteps;
        __syncthreads();  // the item is done: bt_s and misc are free again
    }
    // (every issued copy was waited for by the consumers, unless a wait gave
    // up; then let the copies of the last ring turn land before exiting)
    if (warp == kWarps && misc[1]) {
        for (int st = 0; st < kStages && st < gstep; ++st) {
            const int last_use = gstep - 1 - ((gstep - 1 - st) % kStages);
            mbar_wait_bounded(full_s + st * 8, (last_use / kStages) & 1);
        }
    }
}

using ChunkFn = void (*)(const ChunkParams);

ChunkFn select(int D, int G) {
#define PKV_CASE(d, g) \
    if (D == d && G == g) return chunk_attention_kernel<d, g>;
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
#undef PKV_CASE
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
    z.counters_bytes = dec::align256(S * Hk * z.tiles * 4);
    z.list_bytes = dec::align256((2 * S + 3) * 4);  // big_seq, big_cum, n_big, work
    z.ml_bytes = z.parts > 1 ? dec::align256(z.parts * Tq * H * 8) : 0;
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
    ChunkFn fn = select(head_dim, G);
    if (fn == nullptr) return PKV_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const float scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    const int row_bytes = num_kv_heads * head_dim * 2;

    // ---- chunks of up to 8 * col_tiles query rows: the balanced schedule
    int min_rows = 1;
    // (the balanced schedule indexes the flattened block list in 32 bits)
    if (z.col_tiles > 0 && static_cast<int64_t>(num_seqs) * max_blocks_per_seq <= INT32_MAX) {
        dec::BalancedParams b{};
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
        b.num_stages = z.bal.stages;
        b.row_bytes = z.bal.row_bytes;
        b.num_blocks = num_blocks;
        b.query_start = query_start;
        b.max_cols = 8 * z.col_tiles;
        b.num_query_tokens = num_query_tokens;
        const int64_t c_bytes = dec::align256(static_cast<int64_t>(num_seqs) * num_kv_heads * 4);
        const int64_t slots = 2 * static_cast<int64_t>(z.bal.grid) * num_kv_heads * b.max_cols;
        b.counters = reinterpret_cast<int *>(ws);
        b.part_ml = reinterpret_cast<float2 *>(ws + c_bytes);
        b.part_o = reinterpret_cast<float *>(ws + c_bytes + dec::align256(slots * 8));
        const int box = row_bytes / dec::chunk_bytes_for_row(row_bytes);
        int st = dec::make_kv_tensor_map(&b.tm_k, k_cache, num_blocks, row_bytes, box);
        if (st == PKV_OK) st = dec::make_kv_tensor_map(&b.tm_v, v_cache, num_blocks, row_bytes, box);
        if (st != PKV_OK) return st;
        b.err = device_error_record();
        if (b.err == nullptr) return PKV_ERR_CUDA;
        st = dec::launch_balanced(b, z.bal, head_dim, G, false, false, s, z.col_tiles);
        if (st != PKV_OK) return st;
        min_rows = b.max_cols + 1;
        if (static_cast<int64_t>(max_query_len) * G < min_rows) return PKV_OK;  // all done
    }

    // ---- the larger chunks: query tiles of 64 rows
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
    p.num_query_tokens = num_query_tokens;
    p.min_rows = min_rows;
    p.num_blocks = num_blocks;
    uint8_t *cws = ws + z.bal_bytes;
    p.num_seqs = num_seqs;
    p.big_seq = reinterpret_cast<int *>(cws);
    p.big_cum = p.big_seq + num_seqs;
    p.n_big = p.big_cum + num_seqs + 1;
    p.work = p.n_big + 1;
    cws += z.list_bytes;
    p.counters = reinterpret_cast<int *>(cws);
    p.part_ml = reinterpret_cast<float2 *>(cws + z.counters_bytes);
    p.part_o = reinterpret_cast<float *>(cws + z.counters_bytes + z.ml_bytes);
    {
        // per-head boxes: kv_head's head_dim*2 bytes are whole 128-byte chunks
        const int box = head_dim * 2 / dec::chunk_bytes_for_row(row_bytes);
        int st = dec::make_kv_tensor_map(&p.tm_k, k_cache, num_blocks, row_bytes, box);
        if (st == PKV_OK) st = dec::make_kv_tensor_map(&p.tm_v, v_cache, num_blocks, row_bytes, box);
        if (st != PKV_OK) return st;
    }
    p.err = device_error_record();
    if (p.err == nullptr) return PKV_ERR_CUDA;

    // the work list (one CTA), then persistent CTAs that pull from it
    chunk_plan_kernel<<<1, 1024, 0, s>>>(p, G);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_failure(e, "chunk plan launch");
    const int smem = smem_bytes(head_dim);
    int per_sm = 0;
    const int st = prepare_kernel(reinterpret_cast<const void *>(fn), kThreads, smem, &per_sm);
    if (st != PKV_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(std::max(1, sm_count() * std::max(1, per_sm))));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fn, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_failure(e, "chunk attention launch");
}
