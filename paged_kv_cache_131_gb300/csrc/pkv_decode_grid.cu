// pkv_decode_grid.cu -- paged decode attention, grid schedule: one CTA of 4
// warps per (kv_head, sequence, partition of `partition_size` tokens), so
// the G query heads of a GQA group share every K/V byte the CTA reads.
//
// The CTA
//   1. loads its sequence length and the partition's slice of the block
//      table together (the slice is inside the table row whatever the
//      length), then keeps the ids of the partition's blocks, checking each
//      against [0, num_blocks);
//   2. gives each warp every 4th block of the partition and a private
//      2-stage ring: one tiled tensor copy (TMA) brings kv_head's slice
//      (head_dim*2 bytes) of the block's 16 key rows and one its value rows,
//      completing on the stage's mbarrier;
//   3. folds each block into the warp's online-softmax state (compute
//      policy of pkv_decode_common.cuh);
//   4. merges the 4 warps in shared memory; a one-partition sequence writes
//      fp16 out, otherwise the CTA stores its partial (m, l, o) and the last
//      CTA of the (sequence, kv_head) to take a ticket merges all partitions
//      with a log-sum-exp rescale.  No CTA ever waits for another.
// Partitions are the slowest grid dimension, so the empty partitions of
// short sequences are scheduled last.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/pagedkv.h"
#include "pkv_decode_common.cuh"
#include "pkv_decode_host.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace dec {
namespace {

constexpr int kWarps = kGridWarps;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = kGridStages;
constexpr int kMaxBtPerThread = (kMaxPartitionTokens / kBS + kThreads - 1) / kThreads;

template <int D>
struct Geo {
    static constexpr int kRowBytes = D * 2;  // one head's row of a token
    static constexpr int kTileBytes = kBS * kRowBytes;  // one K (or V) block tile
    static constexpr int kStageBytes = 2 * kTileBytes;  // K + V
    static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
};

// Shared-memory layout (dynamic, from a 1024-byte aligned base):
//   ring    kWarps * kStages * (K tile + V tile) -- reused after the main loop
//           by the warp merge and the partition combine
//   bars    kWarps * kStages mbarriers
//   bt      partition_blocks int32 (block ids, -1 = skipped)
//   misc    4 int32 (abort flag, last-CTA flag)
//   pbuf    kWarps * 16 * G fp32 (SIMT policy: one block's softmax weights)

template <int D, int G, class Policy>
__global__ void __launch_bounds__(kThreads)
    decode_grid_kernel(const __grid_constant__ GridParams p) {
    using Gm = Geo<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((kTileAlign - (smem_u32(smem_raw) & (kTileAlign - 1))) &
                                (kTileAlign - 1));
    uint8_t *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Gm::kRingBytes);
    int *bt_s = reinterpret_cast<int *>(bars + kWarps * kStages);
    int *misc = bt_s + p.partition_blocks;
    float *pbuf_all = reinterpret_cast<float *>(misc + 4);

    const int kvh = blockIdx.x, seq = blockIdx.y, part = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.num_heads;
    const int P = p.num_partitions;

    if (threadIdx.x == 0) misc[0] = 0;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&bars[warp * kStages + s]), 1);
        fence_mbarrier_init();
    }

    // Launched with programmatic stream serialization, so this grid may start
    // while the previous kernel in the stream -- typically the cache write,
    // which writes nothing but the caches -- is still running.  The length and
    // the block table are read before grid_dependency_wait(); the caches and
    // the outputs are touched only after it.

    // ---- sequence length and block-table slice, loaded together
    const int blk0 = part * p.partition_blocks;
    const int avail = max(0, min(p.partition_blocks, p.max_blocks_per_seq - blk0));
    const int32_t *bt_row = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq;
    int L = __ldg(p.seq_lens + seq);
    int braw[kMaxBtPerThread];
#pragma unroll
    for (int k = 0; k < kMaxBtPerThread; ++k) {
        const int j = threadIdx.x + k * kThreads;
        braw[k] = j < avail ? __ldg(bt_row + blk0 + j) : -1;
    }
    const int cap = min(p.max_blocks_per_seq, P * p.partition_blocks) * kBS;
    if (L < 0 || L > cap) {
        if (threadIdx.x == 0 && kvh == 0 && part == 0)
            record_error(p.err, PKV_DEVERR_SEQ_LEN, seq);
        L = L < 0 ? 0 : cap;
    }
    const int nblk_seq = (L + kBS - 1) / kBS;
    const int nparts = max(1, (nblk_seq + p.partition_blocks - 1) / p.partition_blocks);
    if (part >= nparts) return;  // whole CTA: nothing of this sequence here
    const int nblk = min(p.partition_blocks, nblk_seq - blk0);  // >= 0
#pragma unroll
    for (int k = 0; k < kMaxBtPerThread; ++k) {
        const int j = threadIdx.x + k * kThreads;
        if (j < nblk) {
            int b = braw[k];
            if (b < 0 || static_cast<int64_t>(b) >= p.num_blocks) {
                if (kvh == 0)
                    record_error(p.err, PKV_DEVERR_BLOCK_ID,
                                 static_cast<int64_t>(seq) * p.max_blocks_per_seq + blk0 + j);
                b = -1;
            }
            bt_s[j] = b;
        }
    }
    __syncthreads();
    grid_dependency_wait();

    // ---- per-warp pipeline over blocks warp, warp+4, warp+8, ...
    Policy st;
    const __half *qg = p.q + (static_cast<int64_t>(seq) * H + kvh * G) * D;
    st.init(qg, p.scale_log2, lane);
    float *pbuf = pbuf_all + warp * kBS * G;

    const int nw = nblk > warp ? (nblk - warp + kWarps - 1) / kWarps : 0;
    // the map's chunks are those of the whole row (all heads), a multiple of 128 bytes
    const SwizzledTile tile{7u};
    const int head_chunk = kvh * (Gm::kRowBytes / 128);
    const uint32_t ring_s = smem_u32(ring + warp * kStages * Gm::kStageBytes);
    const uint32_t bar_s = smem_u32(&bars[warp * kStages]);

    auto valid_tokens = [&](int i) -> int {
        const int j = warp + i * kWarps;
        return bt_s[j] < 0 ? 0 : min(kBS, L - (blk0 + j) * kBS);
    };
    auto issue = [&](int i) {
        const int j = warp + i * kWarps;
        const int nv = valid_tokens(i);
        const int s = i % kStages;
        const uint32_t bar = bar_s + s * 8;
        // whole 16-row tiles: rows past the last valid token still belong to
        // the physical block
        if (lane == 0)
            mbar_arrive_expect_tx(bar, nv > 0 ? 2u * Gm::kTileBytes : 0u);
        __syncwarp();
        if (nv > 0 && lane < 2)
            tensor_g2s_3d(ring_s + s * Gm::kStageBytes + lane * Gm::kTileBytes,
                          lane == 0 ? &p.tm_k : &p.tm_v, 0, bt_s[j] * kBS, head_chunk, bar);
    };

    const int npre = nw < kStages ? nw : kStages;
    for (int i = 0; i < npre; ++i) issue(i);
    int i = 0;
    bool aborted = false;
    for (; i < nw; ++i) {
        const int s = i % kStages;
        const bool landed = mbar_wait_bounded(bar_s + s * 8, (i / kStages) & 1);
        if (!__all_sync(0xffffffffu, landed)) {  // warp-uniform decision
            aborted = true;
            break;
        }
        const int nv = valid_tokens(i);
        if (nv > 0) {
            const uint32_t kb = ring_s + s * Gm::kStageBytes;
            if (Policy::kZeroTailRows && nv < kBS)
                zero_tail_rows<D>(kb + Gm::kTileBytes, tile, 0u, nv, lane);
            st.block(kb, kb + Gm::kTileBytes, tile, 0u, nv, p.scale_log2, lane, pbuf);
        }
        __syncwarp();
        if (i + kStages < nw) {
            fence_proxy_async_smem();
            issue(i + kStages);
        }
    }
    if (aborted) {
        // give up on this CTA's result, but let every copy in flight land first
        if (lane == 0)
            record_error(p.err, PKV_DEVERR_TIMEOUT,
                         (static_cast<int64_t>(part) * gridDim.y + seq) * gridDim.x + kvh);
        const int stop = (i + kStages < nw) ? i + kStages : nw;
        for (int k = i; k < stop; ++k)
            mbar_wait_bounded(bar_s + (k % kStages) * 8, (k / kStages) & 1);
        if (lane == 0) atomicOr(&misc[0], 1);
    }
    __syncthreads();  // all rings idle: reuse them for the merge

    // ---- merge the warps of this CTA
    float *mg_m = reinterpret_cast<float *>(ring);  // [kWarps][G]
    float *mg_l = mg_m + kWarps * G;                // [kWarps][G]
    float *mg_o = mg_l + kWarps * G;                // [kWarps][G][D]
    st.export_state(mg_m + warp * G, mg_l + warp * G, mg_o + warp * G * D, lane);
    __syncthreads();
    const bool bad = misc[0] != 0;
    for (int e = threadIdx.x; e < G * D; e += kThreads) {
        const int g = e / D, d = e % D;
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mg_m[w * G + g]);
        float lsum = 0.f, osum = 0.f;
        if (M != kNegInf && !bad) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float mw = mg_m[w * G + g];
                const float sc = mw == kNegInf ? 0.f : exp2f(mw - M);
                lsum = fmaf(sc, mg_l[w * G + g], lsum);
                osum = fmaf(sc, mg_o[(w * G + g) * D + d], osum);
            }
        }
        const int64_t hrow = static_cast<int64_t>(seq) * H + kvh * G + g;
        if (nparts == 1) {
            const float r = bad ? NAN : (lsum > 0.f ? osum / lsum : 0.f);
            p.out[hrow * D + d] = __float2half_rn(r);
        } else {
            p.part_o[(hrow * P + part) * D + d] = osum;
            if (d == 0) p.part_ml[hrow * P + part] = make_float2(bad ? kNegInf : M, lsum);
        }
    }
    if (nparts == 1) return;

    // ---- split-KV: the last CTA of this (sequence, kv_head) combines.  The
    // barrier orders every thread's partial before thread 0's releasing
    // ticket (a release is cumulative); the last taker acquires the other
    // CTAs' partials, and the second barrier passes that on to its threads.
    __syncthreads();
    if (threadIdx.x == 0) {
        int *ticket = p.counters + static_cast<int64_t>(seq) * p.num_kv_heads + kvh;
        const int prev = atom_add_acq_rel_gpu(ticket, 1);
        const int last = prev == nparts - 1;
        // every partition has taken its ticket: leave the workspace zeroed
        if (last) st_relaxed_gpu(ticket, 0);
        misc[1] = last;
    }
    __syncthreads();
    if (misc[1] == 0) return;

    // combine scratch, reusing the idle ring
    float *wm = reinterpret_cast<float *>(ring);  // [G][nparts] partition max, then weight
    float *wl = wm + G * nparts;                  // [G][nparts] partition sum
    float *cM = wl + G * nparts;                  // [G] max over partitions
    float *cden = cM + G;                         // [G] rescaled sum over partitions
    const int64_t hrow0 = static_cast<int64_t>(seq) * H + kvh * G;
    for (int e = threadIdx.x; e < G * nparts; e += kThreads) {
        const int g = e / nparts, pp = e % nparts;
        const float2 ml = __ldcg(p.part_ml + (hrow0 + g) * P + pp);
        wm[e] = ml.x;
        wl[e] = ml.y;
    }
    __syncthreads();
    if (threadIdx.x < G) {
        const int g = threadIdx.x;
        float M = kNegInf;
        for (int pp = 0; pp < nparts; ++pp) M = fmaxf(M, wm[g * nparts + pp]);
        float den = 0.f;
        for (int pp = 0; pp < nparts; ++pp) {
            const float mp = wm[g * nparts + pp];
            if (mp != kNegInf) den = fmaf(exp2f(mp - M), wl[g * nparts + pp], den);
        }
        cM[g] = M;
        cden[g] = den;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < G * nparts; e += kThreads) {
        const int g = e / nparts;
        const float mp = wm[e];
        wm[e] = (mp == kNegInf || !(cden[g] > 0.f)) ? 0.f : exp2f(mp - cM[g]) / cden[g];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < G * D; e += kThreads) {
        const int g = e / D, d = e % D;
        const float *po = p.part_o + (hrow0 + g) * P * D + d;
        const float *w = wm + g * nparts;
        float acc = 0.f;
        for (int pp = 0; pp < nparts; ++pp)
            acc = fmaf(w[pp], __ldcg(po + static_cast<int64_t>(pp) * D), acc);
        p.out[(hrow0 + g) * D + d] = __float2half_rn(acc);
    }
}

using GridFn = void (*)(const GridParams);

template <int D, int G>
GridFn pick(bool simt) {
    if (simt) return decode_grid_kernel<D, G, SimtPolicy<D, G>>;
    return decode_grid_kernel<D, G, MmaPolicy<D, G>>;
}

GridFn select(int D, int G, bool simt) {
#define PKV_CASE(d, g) \
    if (D == d && G == g) return pick<d, g>(simt);
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
#undef PKV_CASE
    return nullptr;
}

}  // namespace

int grid_ring_bytes(int D) { return kWarps * kStages * 2 * kBS * D * 2; }

int grid_smem_bytes(int D, int G, int partition_blocks) {
    return kTileAlign + grid_ring_bytes(D) + kWarps * kStages * 8 + partition_blocks * 4 +
           4 * 4 + kWarps * kBS * G * 4;
}

int64_t grid_workspace_bytes(int64_t S, int64_t H, int64_t D, int64_t P) {
    if (P <= 1) return 0;
    return align256(S * H * 4) + align256(S * H * P * 8) + S * H * P * D * 4;
}

int launch_grid(const GridParams &p, int D, int G, bool simt, int num_seqs,
                cudaStream_t stream) {
    GridFn fn = select(D, G, simt);
    if (fn == nullptr) return PKV_ERR_UNSUPPORTED;
    const int smem = grid_smem_bytes(D, G, p.partition_blocks);
    const int st = prepare_kernel(reinterpret_cast<const void *>(fn), kThreads, smem, nullptr);
    if (st != PKV_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_kv_heads, num_seqs, p.num_partitions);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, fn, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_failure(e, "decode grid launch");
}

}  // namespace dec
}  // namespace pkv
