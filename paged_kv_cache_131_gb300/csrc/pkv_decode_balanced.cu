// pkv_decode_balanced.cu -- paged decode attention, balanced schedule.
//
// The KV heads are taken in groups of up to 8 (heads_per_cta, a divisor of
// num_kv_heads).  The work is the flattened list of (head group, sequence,
// logical block) triples, groups outermost: T = groups * sum_i ceil(L_i / 16)
// blocks, each carrying one head group of 16 tokens.  The launch is one wave
// of persistent CTAs; CTA c owns the contiguous range [c*T/N, (c+1)*T/N) of
// that list, so every CTA reads the same number of bytes whatever the length
// mix, and no CTA is empty.  A (head group, sequence) pair is a "virtual
// sequence": a contiguous interval of the list, numbered group * S + seq.
//
// A CTA has one producer warp and one consumer warp per KV head of a group.
//  - The producer walks its range.  For each block it takes the next stage
//    of a `num_stages`-deep ring (waiting on the stage's "empty" mbarrier),
//    publishes the block's (virtual sequence, valid tokens, block id), and
//    issues one tiled tensor copy (TMA) for the block's 16 key rows and one
//    for its 16 value rows (a staged row = the group's KV heads of one token,
//    heads_per_cta*head_dim*elem contiguous bytes; FP8 adds two bulk copies
//    of the block's scales, all heads), completing on the stage's "full"
//    mbarrier.  One copy per tile
//    keeps the producer's issue cost per block small: issuing a copy takes
//    the warp about as long whatever its size, and per-row copies made the
//    producer the bottleneck.  Block-table entries are loaded a 32-block
//    window ahead.
//  - Consumer warp h waits on "full", folds head h of the group (KV head
//    group*heads_per_cta + h) 16 keys/values into its
//    online-softmax state (compute policy of pkv_decode_common.cuh) and
//    arrives on "empty".  When the sequence changes it finishes the previous
//    one: a sequence wholly inside the range is normalised and written as
//    fp16; a sequence cut by a range boundary leaves a partial (m, l, o) in
//    the workspace, and the last of its contributors to take a ticket merges
//    the partials with a log-sum-exp rescale.  No warp ever waits for
//    another CTA.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>

#include "../../include/pagedkv.h"
#include "pkv_decode_common.cuh"
#include "pkv_decode_host.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace dec {
namespace {

constexpr int kMaxStages = 4;
constexpr int kMaxStagesFp8 = 6;  // FP8 stages are half the size: keep as many bytes in flight
constexpr int kMaxThreads = (kMaxBalancedKvHeads + 1) * 32;
// Dynamic shared memory:
//   ring   stages * (key tile, value tile[, key scales, value scales]),
//          each stage 1024-byte aligned; a tile is 16 rows, chunk-major and
//          swizzled (SwizzledTile)
//   full   stages mbarriers (1 arrival + transaction bytes)
//   empty  stages mbarriers (one arrival per consumer warp)
//   meta   stages int4 {sequence, valid tokens, block id (-1 = skip), 0}
//   cum    S + 1 int32: exclusive prefix sum of the sequences' block counts
//   lens   S int32: sequence lengths (clamped to the block table)
//   misc   4 int32
//   pbuf   heads_per_cta * 16 * G fp32 (SIMT policy: one block's softmax weights)
// (plus kTileAlign bytes to align the dynamic shared memory base)
int smem_bytes(int stages, int stage_bytes, int S, int Hk, int G) {
    return kTileAlign + stages * stage_bytes + stages * 16 + stages * 16 + (2 * S + 1) * 4 + 16 +
           Hk * kBS * G * 4;
}

// Bytes of one stage: key and value tiles (+ FP8 scales), 1024-aligned.
__host__ __device__ int stage_bytes_for(int row_bytes, int Hk, bool fp8) {
    const int raw = 2 * kBS * row_bytes + (fp8 ? 2 * kBS * Hk * 4 : 0);
    return (raw + kTileAlign - 1) / kTileAlign * kTileAlign;
}

// Largest s in [0, S) with cum[s] <= f (cum non-decreasing, cum[0] = 0).
__device__ __forceinline__ int find_seq(const int *cum, int S, int64_t f) {
    int lo = 0, hi = S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cum[mid] <= f) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// CTA whose range holds flattened block f (ranges [c*T/N, (c+1)*T/N)).
__device__ __forceinline__ int cta_of(int64_t f, int64_t T, int64_t N) {
    return static_cast<int>(((f + 1) * N + T - 1) / T - 1);
}

// Merge the partials of (seq, kvh) left by CTAs c_a..c_b and write fp16 out.
// One warp.  The contributors' (m, l) are loaded together (lane j holds
// contributor j of each 32-wide chunk) and reduced with shuffles; the
// partial outputs are then accumulated U contributors at a time (32 floats
// in flight per lane), so their loads overlap instead of forming a chain of
// L2 round trips.
// R partial rows per (sequence, kv head); row r is query row
// (row0 + r / Gq) * H + kvh * Gq + r % Gq, rows >= ncols unused.  Rows are
// merged eight at a time (bounded registers).
// kvh is the KV head, hl its index within its head group (the partial rows
// are laid out per group member).
template <int D, int R>
__device__ void combine_partials(const BalancedParams &p, int kvh, int hl, int c_a, int c_b,
                                 int64_t f_s, int64_t T, int64_t N, int lane, int64_t row0,
                                 int ncols, int Gq) {
    constexpr int G = R < 8 ? R : 8;  // rows per pass
    constexpr int DPL = D / 32;
    constexpr int U = (32 / (G * DPL)) < 1 ? 1 : ((32 / (G * DPL)) > 4 ? 4 : 32 / (G * DPL));
    const int Hc = p.heads_per_cta;
    const int nc = c_b - c_a + 1;
    // first partial row of contributor c_a + j
    auto row_of = [&](int j) -> int64_t {
        const int c = c_a + j;
        const int64_t fc = static_cast<int64_t>(c) * T / N;
        const int64_t slot = 2 * static_cast<int64_t>(c) + ((j == 0 && fc < f_s) ? 1 : 0);
        return (slot * Hc + hl) * R;
    };
    for (int r0 = 0; r0 < R && r0 < ncols; r0 += G) {
        // pass 1: the running maximum of every row over all contributors
        float M[G];
#pragma unroll
        for (int g = 0; g < G; ++g) M[g] = kNegInf;
        for (int j0 = 0; j0 < nc; j0 += 32) {
            if (j0 + lane < nc) {
                const int64_t r = row_of(j0 + lane) + r0;
#pragma unroll
                for (int g = 0; g < G; ++g) M[g] = fmaxf(M[g], __ldcg(p.part_ml + r + g).x);
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                M[g] = fmaxf(M[g], __shfl_xor_sync(0xffffffffu, M[g], o));
        // pass 2: per chunk, each lane's contributor weight 2^(m - M) (0 for
        // a contributor whose blocks were all skipped or masked), the
        // normaliser, and the weighted partial outputs
        float den[G], acc[G][DPL];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            den[g] = 0.f;
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[g][i] = 0.f;
        }
        for (int j0 = 0; j0 < nc; j0 += 32) {
            float w[G];
            int64_t r = 0;
            if (j0 + lane < nc) {
                r = row_of(j0 + lane) + r0;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float2 ml = __ldcg(p.part_ml + r + g);
                    w[g] = ml.x == kNegInf ? 0.f : exp2f(ml.x - M[g]);
                    den[g] = fmaf(ml.y, w[g], den[g]);
                }
            } else {
#pragma unroll
                for (int g = 0; g < G; ++g) w[g] = 0.f;
            }
            const int cnt = min(32, nc - j0);
            for (int k0 = 0; k0 < cnt; k0 += U) {
                float o[U][G][DPL];
                float wk[U][G];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = min(k0 + u, cnt - 1);  // a repeated contributor gets weight 0
                    const int64_t rk = __shfl_sync(0xffffffffu, r, k);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float wg = __shfl_sync(0xffffffffu, w[g], k);
                        wk[u][g] = k0 + u < cnt ? wg : 0.f;
                        const float *po = p.part_o + (rk + g) * D + lane * DPL;
                        if constexpr (DPL == 4) {
                            const float4 v = __ldcg(reinterpret_cast<const float4 *>(po));
                            o[u][g][0] = v.x; o[u][g][1] = v.y; o[u][g][2] = v.z; o[u][g][3] = v.w;
                        } else {
                            const float2 v = __ldcg(reinterpret_cast<const float2 *>(po));
                            o[u][g][0] = v.x; o[u][g][1] = v.y;
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int i = 0; i < DPL; ++i)
                            acc[g][i] = fmaf(o[u][g][i], wk[u][g], acc[g][i]);
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) den[g] += __shfl_xor_sync(0xffffffffu, den[g], o);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int rr = r0 + g;
            if (rr >= ncols) break;
            const float inv = den[g] > 0.f ? 1.f / den[g] : 0.f;
            __half *out =
                p.out + ((row0 + rr / Gq) * p.num_heads + kvh * Gq + rr % Gq) * D + lane * DPL;
#pragma unroll
            for (int i = 0; i < DPL; i += 2)
                *reinterpret_cast<__half2 *>(out + i) =
                    __floats2half2_rn(acc[g][i] * inv, acc[g][i + 1] * inv);
        }
    }
}

template <int D, int G, class Policy, bool kFp8>
__device__ __forceinline__ void balanced_body(const BalancedParams &p, uint8_t *smem_raw) {
    uint8_t *smem = smem_raw + ((kTileAlign - (smem_u32(smem_raw) & (kTileAlign - 1))) &
                                (kTileAlign - 1));
    const int Hk = p.num_kv_heads, Hc = p.heads_per_cta, S = p.num_seqs, NS = p.num_stages;
    const int H = p.num_heads;
    const SwizzledTile tile{chunk_bytes_for_row(p.row_bytes) == 128 ? 7u : 6u};
    const int tile_bytes = kBS * p.row_bytes;
    // tensor-copy boxes: the group's chunks of a row; group g starts at chunk g * box
    const int box_chunks = p.row_bytes / chunk_bytes_for_row(p.row_bytes);
    // FP8: a stage also holds the block's key and value scales ([16][Hk] fp32 each)
    const int scale_bytes = kFp8 ? kBS * Hk * 4 : 0;
    const int stage_bytes = stage_bytes_for(p.row_bytes, Hk, kFp8);
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * stage_bytes);
    uint64_t *empty = full + NS;
    int4 *meta = reinterpret_cast<int4 *>(empty + NS);
    int *cum = reinterpret_cast<int *>(meta + NS);
    int *lens = cum + S + 1;
    int *misc = lens + S;
    float *pbuf_all = reinterpret_cast<float *>(misc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nthreads = blockDim.x, nwarps = nthreads >> 5;

    // CTAs taking part: the whole grid, or the first *active_ctas of it.  The
    // others leave before doing anything: they may be scheduled only when an
    // SM frees up at the end of the call, and must not add to it.
    int grid = static_cast<int>(gridDim.x);
    if (p.active_ctas != nullptr) {
        const int a = __ldcg(p.active_ctas);
        if (a > 0 && a < grid) grid = a;
    }
    if (static_cast<int>(blockIdx.x) >= grid) return;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), Hc);
        }
        fence_mbarrier_init();
    }

    // Launched with programmatic stream serialization, so this grid may start
    // while the previous kernel in the stream -- typically the cache write,
    // which writes nothing but the caches -- is still running.  Lengths, block
    // tables and queries are read before grid_dependency_wait(); the caches
    // and the outputs are touched only after it.

    // While the lengths below make their round trip: the copies' tensor maps,
    // and this CTA's share of the block table into L2 (a small table only),
    // so the block-table window it reads next is an L2 hit.
    if (threadIdx.x == 0) {
        prefetch_tensormap(&p.tm_k);
        prefetch_tensormap(&p.tm_v);
    }
    if (static_cast<int64_t>(S) * p.max_blocks_per_seq <= (int64_t(4) << 20)) {  // <= 16 MB
        const int lines = (S * p.max_blocks_per_seq * 4 + 127) >> 7;
        const int per = (lines + grid - 1) / grid, end = min(lines, (blockIdx.x + 1) * per);
        const char *tb = reinterpret_cast<const char *>(p.block_tables);
        for (int i = blockIdx.x * per + threadIdx.x; i < end; i += nthreads)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(tb + static_cast<size_t>(i) * 128));
    }

    // ---- lengths (clamped to the block table) and their block-count prefix sum
    const int cap = p.max_blocks_per_seq * kBS;
    const int chunk = (S + nthreads - 1) / nthreads;
    const int s_begin = min(S, threadIdx.x * chunk), s_end = min(S, s_begin + chunk);
    int local = 0;
    for (int s = s_begin; s < s_end; ++s) {
        int L = __ldg(p.seq_lens + s);
        if (L < 0 || L > cap) {
            if (blockIdx.x == 0) record_error(p.err, PKV_DEVERR_SEQ_LEN, s);
            L = L < 0 ? 0 : cap;
        }
        if constexpr (Policy::kColumns) {
            // -1: not this kernel's (no new token, or more columns than it holds)
            const int nq = __ldg(p.query_start + s + 1) - __ldg(p.query_start + s);
            if (nq > L || nq < 0) {
                if (blockIdx.x == 0) record_error(p.err, PKV_DEVERR_SEQ_LEN, s);
                L = -1;
            } else if (nq == 0 || nq * G > p.max_cols) {
                L = -1;
            }
        }
        lens[s] = L;
        local += L > 0 ? (L + kBS - 1) / kBS : 0;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    int *wsum = reinterpret_cast<int *>(ring);  // scratch, before the ring is used
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int v = lane < nwarps ? wsum[lane] : 0;
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane < nwarps) wsum[lane] = inc - v;
        if (lane == nwarps - 1) wsum[32] = inc;
    }
    __syncthreads();
    {
        int run = wsum[warp] + incl - local;
        for (int s = s_begin; s < s_end; ++s) {
            cum[s] = run;
            run += lens[s] > 0 ? (lens[s] + kBS - 1) / kBS : 0;
        }
        if (threadIdx.x == 0) cum[S] = wsum[32];
    }
    fence_proxy_async_smem();  // scratch writes before the first bulk copy into the ring
    __syncthreads();

    // ---- empty sequences get zeros (no block of theirs is in any range)
    const int64_t Tb = cum[S];                 // blocks of one head group
    const int64_t T = Tb * p.groups;           // the whole (group, sequence, block) list
    const int64_t N = min(static_cast<int64_t>(grid), T);
    bool zeros_due = false;
    for (int s = blockIdx.x; s < S && !zeros_due; s += grid) zeros_due = lens[s] == 0;
    if (zeros_due && (blockIdx.x >= N || warp < Hc)) {
        // the consumers (or every warp of a CTA without a range) write them
        if (!p.defer_wait) grid_dependency_wait();
        const int nz = blockIdx.x >= N ? nthreads : Hc * 32;
        for (int s = blockIdx.x; s < S; s += grid) {
            if (lens[s] == 0) {
                uint4 *o = reinterpret_cast<uint4 *>(p.out + static_cast<int64_t>(s) * H * D);
                for (int e = threadIdx.x; e < H * D / 8; e += nz) o[e] = make_uint4(0, 0, 0, 0);
            }
        }
    }
    if (blockIdx.x >= N) return;
    const int64_t f0 = static_cast<int64_t>(blockIdx.x) * T / N;
    const int64_t f1 = (static_cast<int64_t>(blockIdx.x) + 1) * T / N;
    const int n = static_cast<int>(f1 - f0);  // >= 1

    const uint32_t ring_s = smem_u32(ring);
    const uint32_t full_s = smem_u32(full), empty_s = smem_u32(empty);

    // (head group, sequence, block in the sequence) of flattened block f
    const bool grouped = p.groups > 1;
    auto locate = [&](int64_t f, int &hg, int &seq, int &blk) {
        hg = grouped ? static_cast<int>(f / Tb) : 0;
        const int64_t fl = f - static_cast<int64_t>(hg) * Tb;
        seq = find_seq(cum, S, fl);
        blk = static_cast<int>(fl - cum[seq]);
    };

    if (warp == Hc) {
        // ================================ producer ================================
        // window of 32 blocks: lane j describes block base + j (vseq: its
        // virtual sequence group * S + seq; blk: its index in the sequence;
        // z: the first chunk of its group's box)
        auto fetch = [&](int base, int &raw, int &vseq, int &nv, int &blk, int &z) {
            const int i = base + lane;
            raw = -1;
            vseq = -1;
            nv = 0;
            blk = 0;
            z = 0;
            if (i < n) {
                int hg, seq;
                locate(f0 + i, hg, seq, blk);
                vseq = hg * S + seq;
                z = hg * box_chunks;
                nv = min(kBS, lens[seq] - blk * kBS);
                // checked when its window becomes current, so the load's latency
                // hides behind the 32 blocks before it
                raw = __ldg(p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq + blk);
            }
        };
        auto check = [&](int base, int raw, int vseq, int blk) -> int {
            const int i = base + lane;
            if (i >= n) return -1;
            if (raw < 0 || static_cast<int64_t>(raw) >= p.num_blocks) {
                const int seq = vseq % S;
                record_error(p.err, PKV_DEVERR_BLOCK_ID,
                             static_cast<int64_t>(seq) * p.max_blocks_per_seq + blk);
                return -1;
            }
            return raw;
        };
        int c_raw, c_seq, c_nv, c_blk, c_z, n_raw, n_seq, n_nv, n_blk, n_z;
        fetch(0, c_raw, c_seq, c_nv, c_blk, c_z);
        int c_bid = check(0, c_raw, c_seq, c_blk);
        fetch(32, n_raw, n_seq, n_nv, n_blk, n_z);
        if (!p.defer_wait) grid_dependency_wait();  // the caches may have just been written
        int issued = 0;
        bool ok = true;
        for (int i = 0; i < n; ++i) {
            const int st = i % NS;
            if (i >= NS) {
                const bool free_ = mbar_wait_bounded(empty_s + st * 8, ((i / NS) - 1) & 1);
                if (!__all_sync(0xffffffffu, free_)) {
                    ok = false;
                    break;
                }
            }
            if (i > 0 && (i & 31) == 0) {
                c_bid = check(i, n_raw, n_seq, n_blk);
                c_seq = n_seq;
                c_nv = n_nv;
                c_blk = n_blk;
                c_z = n_z;
                fetch(i + 32, n_raw, n_seq, n_nv, n_blk, n_z);
            }
            const int bid = __shfl_sync(0xffffffffu, c_bid, i & 31);
            const int vseq = __shfl_sync(0xffffffffu, c_seq, i & 31);
            const int nv = __shfl_sync(0xffffffffu, c_nv, i & 31);
            const int blk = __shfl_sync(0xffffffffu, c_blk, i & 31);
            const int z = grouped ? __shfl_sync(0xffffffffu, c_z, i & 31) : 0;
            // the whole 16-row tiles (rows past the last valid token still
            // belong to the physical block)
            const bool copy = bid >= 0 && nv > 0;
            const uint32_t stage = ring_s + st * stage_bytes;
            if (lane == 0) {
                // .w: the block's index in its sequence
                meta[st] = make_int4(vseq, nv, bid, blk);
                mbar_arrive_expect_tx(full_s + st * 8,
                                      copy ? 2u * tile_bytes + (kFp8 ? 2u * scale_bytes : 0u)
                                           : 0u);
            }
            __syncwarp();
            if (copy && lane < 2)
                tensor_g2s_3d(stage + lane * tile_bytes, lane == 0 ? &p.tm_k : &p.tm_v, 0,
                              bid * kBS, z, full_s + st * 8);
            if (kFp8 && copy && (lane == 2 || lane == 3)) {
                // the block's scales: 16 tokens x Hk heads, contiguous
                const float *src = (lane == 2 ? p.k_scale : p.v_scale) +
                                   static_cast<int64_t>(bid) * kBS * Hk;
                bulk_g2s(stage + 2 * tile_bytes + (lane - 2) * scale_bytes, src, scale_bytes,
                         full_s + st * 8);
            }
            issued = i + 1;
        }
        if (!ok && lane == 0) record_error(p.err, PKV_DEVERR_TIMEOUT, blockIdx.x);
        // every copy issued must land before the CTA may exit
        for (int st = 0; st < NS && st < issued; ++st) {
            const int uses = (issued - 1 - st) / NS + 1;
            mbar_wait_bounded(full_s + st * 8, (uses - 1) & 1);
        }
        return;
    }
    if (warp > Hc) return;

    // ================================ consumers ================================
    const int hl = warp;  // head within the group: its bytes in the staged rows
    int kvh = warp;       // KV head of the current virtual sequence
    Policy st;
    float *pbuf = pbuf_all + hl * kBS * G;
    int cur = -1;
    {
        // warm L2 with the query rows of the (up to 8) virtual sequences this
        // range touches, so a sequence switch does not stall on a cold load
        int hg0, s0, b0, hg1, s1, b1;
        locate(f0, hg0, s0, b0);
        locate(f1 - 1, hg1, s1, b1);
        const int v_first = hg0 * S + s0, v_last = hg1 * S + s1;
        const int bytes = G * D * 2;
        for (int v = v_first; v <= v_last && v < v_first + 8; ++v) {
            const int s = v % S, h = (v / S) * Hc + hl;
            const char *row = reinterpret_cast<const char *>(
                p.q + (static_cast<int64_t>(s) * H + h * G) * D);
            for (int off = lane * 128; off < bytes; off += 32 * 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(row + off));
        }
    }
    if (!p.defer_wait) grid_dependency_wait();  // outputs and partials are written below

    QueryRows qr{p.q, p.out, 0, H, kvh, G, 0};  // the current sequence's query rows
    auto finish = [&](int vseq) {
        const int hg = grouped ? vseq / S : 0, seq = vseq - hg * S;
        const int64_t fg = static_cast<int64_t>(hg) * Tb;
        const int64_t f_s = fg + cum[seq], f_e = fg + cum[seq + 1];
        const int64_t qrow = static_cast<int64_t>(seq) * H + kvh * G;
        if (f_s >= f0 && f_e <= f1) {
            if constexpr (Policy::kColumns) st.write_output(qr, lane);
            else st.write_output(p.out + qrow * D, lane);
            return;
        }
        const int64_t slot = 2 * static_cast<int64_t>(blockIdx.x) + (f_s <= f0 ? 0 : 1);
        const int64_t base = (slot * Hc + hl) * Policy::kRows;
        if constexpr (Policy::kColumns)
            st.write_partial(p.part_ml + base, p.part_o + base * D, qr.ncols, lane);
        else
            st.write_partial(p.part_ml + base, p.part_o + base * D, lane);
        // The warp barrier orders every lane's partial stores before lane 0's
        // releasing ticket; the last taker acquires all contributors' stores,
        // and the shuffle below passes that on to the other lanes.
        __syncwarp();
        const int c_a = cta_of(f_s, T, N), c_b = cta_of(f_e - 1, T, N);
        int last = 0;
        if (lane == 0) {
            int *ticket = p.counters + static_cast<int64_t>(seq) * Hk + kvh;
            const int prev = atom_add_acq_rel_gpu(ticket, 1);
            last = prev == c_b - c_a;
            // every contributor has taken its ticket: leave the workspace zeroed
            if (last) st_relaxed_gpu(ticket, 0);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __syncwarp();  // memory order: lane 0's acquire before every lane's loads
            if constexpr (Policy::kColumns)
                combine_partials<D, Policy::kRows>(p, kvh, hl, c_a, c_b, f_s, T, N, lane,
                                                   qr.row0, qr.ncols, G);
            else
                combine_partials<D, G>(p, kvh, hl, c_a, c_b, f_s, T, N, lane, seq, G, G);
        }
    };

    // FP8 scales of this lane's tokens in a staged block
    using Fp8 = MmaFp8Policy<D, G>;
    constexpr int kLT = Fp8::kLaneTokens;
    auto load_scales = [&](int s, float (&ks)[kLT], float (&vs)[kLT]) {
        const float *sc = reinterpret_cast<const float *>(ring + s * stage_bytes + 2 * tile_bytes);
#pragma unroll
        for (int t = 0; t < kLT; ++t) {
            const int tok = Fp8::token_of(lane, t);
            ks[t] = sc[tok * Hk + kvh];
            vs[t] = sc[kBS * Hk + tok * Hk + kvh];
        }
    };

    bool ok = true;
    for (int i = 0; i < n;) {
        const int s = i % NS;
        const bool landed = mbar_wait_bounded(full_s + s * 8, (i / NS) & 1);
        if (!__all_sync(0xffffffffu, landed)) {
            ok = false;
            break;
        }
        const int4 mt = meta[s];
        if (mt.x != cur) {
            if (cur >= 0) finish(cur);
            cur = mt.x;
            const int hg = grouped ? cur / S : 0, seq = cur - hg * S;
            kvh = hg * Hc + hl;
            if constexpr (Policy::kColumns) {
                const int qs0 = __ldg(p.query_start + seq), qs1 = __ldg(p.query_start + seq + 1);
                qr.row0 = qs0;
                qr.kvh = kvh;
                qr.ncols = (qs1 - qs0) * G;
                qr.lim0 = lens[seq] - (qs1 - qs0);
                st.init(qr, lane);
            } else {
                st.init(p.q + (static_cast<int64_t>(seq) * H + kvh * G) * D, p.scale_log2, lane);
            }
        }
        int used = 1;
        int s2 = 0;
        if constexpr (kFp8) {
            // A full block takes its successor along when that one is of the
            // same sequence: one softmax step over 32 tokens.  (Waiting for
            // the successor while holding this stage cannot stall the
            // producer: the successor's stage was released before.)
            int4 mt2 = make_int4(-1, 0, -1, 0);
            if (mt.z >= 0 && mt.y == kBS && i + 1 < n) {
                s2 = (i + 1) % NS;
                const bool landed2 = mbar_wait_bounded(full_s + s2 * 8, ((i + 1) / NS) & 1);
                if (!__all_sync(0xffffffffu, landed2)) {
                    ok = false;
                    break;
                }
                mt2 = meta[s2];
            }
            const uint32_t kb8 = ring_s + s * stage_bytes;
            const uint32_t head = hl * D;
            if (mt2.x == mt.x && mt2.z >= 0 && mt2.y > 0) {
                const uint32_t kb8b = ring_s + s2 * stage_bytes;
                if (mt2.y < kBS) zero_tail_bytes<D>(kb8b + tile_bytes, tile, head, mt2.y, lane);
                float ks[2][kLT], vs[2][kLT];
                load_scales(s, ks[0], vs[0]);
                load_scales(s2, ks[1], vs[1]);
                const uint32_t kbs[2] = {kb8, kb8b};
                const uint32_t vbs[2] = {kb8 + tile_bytes, kb8b + tile_bytes};
                const int nvs[2] = {mt.y, mt2.y};
                st.template step<2>(kbs, vbs, tile, head, nvs, p.scale_log2, lane, ks, vs);
                used = 2;
            } else if (mt.z >= 0 && mt.y > 0) {
                if (mt.y < kBS) zero_tail_bytes<D>(kb8 + tile_bytes, tile, head, mt.y, lane);
                float ks[1][kLT], vs[1][kLT];
                load_scales(s, ks[0], vs[0]);
                const uint32_t kbs[1] = {kb8};
                const uint32_t vbs[1] = {kb8 + tile_bytes};
                const int nvs[1] = {mt.y};
                st.template step<1>(kbs, vbs, tile, head, nvs, p.scale_log2, lane, ks, vs);
            }
        } else {
            if (mt.z >= 0 && mt.y > 0) {
                const uint32_t kb = ring_s + s * stage_bytes;
                const uint32_t vb = kb + tile_bytes;
                const uint32_t head = hl * D * 2;
                if (Policy::kZeroTailRows && mt.y < kBS)
                    zero_tail_rows<D>(vb, tile, head, mt.y, lane);
                if constexpr (Policy::kColumns)
                    st.block(kb, vb, tile, head, mt.y, mt.w * kBS, p.scale_log2, lane);
                else
                    st.block(kb, vb, tile, head, mt.y, p.scale_log2, lane, pbuf);
            }
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(empty_s + s * 8);
            if (used == 2) mbar_arrive(empty_s + s2 * 8);
        }
        i += used;
    }
    if (!ok) {
        if (lane == 0) record_error(p.err, PKV_DEVERR_TIMEOUT, blockIdx.x);
        return;
    }
    if (cur >= 0) finish(cur);
}

template <int D, int G, class Policy, bool kFp8>
__global__ void __launch_bounds__(kMaxThreads, 1)
    decode_balanced_kernel(const __grid_constant__ BalancedParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    balanced_body<D, G, Policy, kFp8>(p, smem_raw);
    // deferred: this grid read nothing the previous one wrote, but must not
    // complete before it (later work in the stream relies on both); CTAs
    // outside the active set did nothing, the first CTA always takes part
    if (p.defer_wait) {
        const int a = p.active_ctas != nullptr ? __ldcg(p.active_ctas) : 0;
        if (a <= 0 || static_cast<int>(blockIdx.x) < a) grid_dependency_wait();
    }
}

using BalancedFn = void (*)(const BalancedParams);

template <int D, int G>
BalancedFn pick(bool simt, bool fp8, int col_tiles) {
    if (col_tiles == 1) return decode_balanced_kernel<D, G, MmaColsPolicy<D, G, 1>, false>;
    if (col_tiles == 2) return decode_balanced_kernel<D, G, MmaColsPolicy<D, G, 2>, false>;
    if (fp8) return decode_balanced_kernel<D, G, MmaFp8Policy<D, G>, true>;
    if (simt) return decode_balanced_kernel<D, G, SimtPolicy<D, G>, false>;
    return decode_balanced_kernel<D, G, MmaPolicy<D, G>, false>;
}

BalancedFn select(int D, int G, bool simt, bool fp8, int col_tiles) {
#define PKV_CASE(d, g) \
    if (D == d && G == g) return pick<d, g>(simt, fp8, col_tiles);
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
#undef PKV_CASE
    return nullptr;
}

}  // namespace

BalancedShape balanced_shape(int num_seqs, int num_kv_heads, int G, int D, int num_sms,
                             bool fp8, int rows) {
    if (rows <= 0) rows = G;
    BalancedShape r{};
    r.ok = num_kv_heads >= 1 && num_seqs >= 1 && (D == 64 || D == 128) &&
           (G == 1 || G == 2 || G == 4 || G == 8);
    if (!r.ok) return r;
    // heads per CTA: the largest divisor of num_kv_heads up to 8 whose staged
    // row has the swizzle chunk of the whole row (the tensor maps span whole
    // rows; a group's box starts at a chunk boundary)
    const int elem = fp8 ? 1 : 2;
    const int chunk = chunk_bytes_for_row(num_kv_heads * D * elem);
    int hc = 0;
    for (int h = std::min(num_kv_heads, kMaxBalancedKvHeads); h >= 1 && hc == 0; --h)
        if (num_kv_heads % h == 0 && chunk_bytes_for_row(h * D * elem) == chunk) hc = h;
    // (virtual sequence numbers group * S + seq stay 32-bit)
    if (hc == 0 || static_cast<int64_t>(num_seqs) * (num_kv_heads / hc) > INT32_MAX) {
        r.ok = false;
        return r;
    }
    const int row_bytes = hc * D * elem;
    const int stage_bytes = stage_bytes_for(row_bytes, num_kv_heads, fp8);
    int stages = fp8 ? kMaxStagesFp8 : kMaxStages;
    while (stages >= 2 && smem_bytes(stages, stage_bytes, num_seqs, hc, G) > kSmemPerSM) --stages;
    if (stages < 2) {
        r.ok = false;
        return r;
    }
    r.stages = stages;
    r.heads = hc;
    r.groups = num_kv_heads / hc;
    r.row_bytes = row_bytes;
    r.smem = smem_bytes(stages, stage_bytes, num_seqs, hc, G);
    const int threads = (hc + 1) * 32;
    r.ctas_per_sm = std::max(1, std::min({(228 * 1024) / (r.smem + 1024), 2048 / threads, 32}));
    r.grid = std::max(1, num_sms) * r.ctas_per_sm;
    const int64_t slots = 2 * static_cast<int64_t>(r.grid) * hc * rows;
    r.workspace = align256(static_cast<int64_t>(num_seqs) * num_kv_heads * 4) +
                  align256(slots * 8) + slots * D * 4;
    return r;
}

int setup_balanced(BalancedParams &p, const BalancedShape &shape, int rows, void *workspace,
                   const void *k_cache, const void *v_cache) {
    p.num_stages = shape.stages;
    p.row_bytes = shape.row_bytes;
    p.heads_per_cta = shape.heads;
    p.groups = shape.groups;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int64_t c_bytes = align256(static_cast<int64_t>(p.num_seqs) * p.num_kv_heads * 4);
    const int64_t slots = 2 * static_cast<int64_t>(shape.grid) * shape.heads * rows;
    p.counters = reinterpret_cast<int *>(ws);
    p.part_ml = reinterpret_cast<float2 *>(ws + c_bytes);
    p.part_o = reinterpret_cast<float *>(ws + c_bytes + align256(slots * 8));
    // maps over whole rows (all heads); a box covers one head group
    const int full_row = shape.row_bytes * shape.groups;
    const int box = shape.row_bytes / chunk_bytes_for_row(shape.row_bytes);
    int st = make_kv_tensor_map(&p.tm_k, k_cache, p.num_blocks, full_row, box);
    if (st == PKV_OK) st = make_kv_tensor_map(&p.tm_v, v_cache, p.num_blocks, full_row, box);
    return st;
}

int launch_balanced(const BalancedParams &p, const BalancedShape &shape, int D, int G, bool simt,
                    bool fp8, cudaStream_t stream, int col_tiles) {
    BalancedFn fn = select(D, G, simt, fp8, col_tiles);
    if (fn == nullptr) return PKV_ERR_UNSUPPORTED;
    const int threads = (p.heads_per_cta + 1) * 32;
    int per_sm = 0;
    const int st = prepare_kernel(reinterpret_cast<const void *>(fn), threads, shape.smem, &per_sm);
    if (st != PKV_OK) return st;
    per_sm = std::max(1, std::min(per_sm, shape.ctas_per_sm));
    const int grid = std::min(shape.grid, per_sm * std::max(1, shape.grid / shape.ctas_per_sm));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = shape.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, fn, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_failure(e, "decode balanced launch");
}

}  // namespace dec
}  // namespace pkv
