// pkv_decode.cu -- paged decode attention ("deep-dive-into-vllm-05" §2 read
// loop, §3.2 GQA; "vLLM 技术内幕" §2.1: dot the query with the keys of each
// physical block in turn and accumulate the values block by block).
//
// Grid (kv_head, partition, sequence); one CTA of 4 warps owns one
// (sequence, kv_head, partition of `partition_size` tokens), so the G query
// heads of a GQA group share every K/V byte it reads.  The CTA
//   1. copies the partition's slice of the block table into shared memory,
//      checking every id against [0, num_blocks);
//   2. gives each warp every 4th physical block of the partition and a
//      private 2-stage ring: for a block, 16 lanes each issue one bulk (TMA)
//      copy of a K row (head_dim * 2 bytes of kv_head) and 16 lanes one of a
//      V row, completing on the stage's mbarrier; rows land 16 bytes apart
//      from each other's bank phase (row pitch head_dim*2 + 16) so the
//      ldmatrix reads below are conflict-free;
//   3. per block: scores of the G heads against the block's 16 keys, an
//      online-softmax update (running max m and sum l in the log2 domain)
//      and o = alpha*o + p*V, in one of two compute policies:
//        MMA  -- the G query rows packed into the 16-row A operand of
//                m16n8k16 fp16 MMAs (fp32 accumulate), S = Q K^T then
//                O += P V with P re-packed from the S fragments;
//        SIMT -- fp32 FMAs on CUDA cores, lanes split head_dim and a
//                butterfly reduce-scatter of the dot products;
//   4. merges the 4 warps' (m, l, o) in shared memory; a single-partition
//      sequence writes fp16 out directly, otherwise the CTA stores its
//      partial (m, l, o) and the last CTA of the (sequence, kv_head) to
//      finish -- an atomic ticket, no waiting -- merges all partitions with
//      a log-sum-exp rescale and writes out.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace dec {

constexpr int kBS = 16;       // tokens per physical block
constexpr int kWarps = 4;     // warps per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;    // blocks in flight per warp
constexpr int kRowPad = 16;   // bytes between staged rows beyond head_dim*2
constexpr int kMaxPartitionTokens = 8192;
constexpr int kDefaultPartitionTokens = 512;
constexpr float kNegInf = -INFINITY;

template <int D>
struct Geo {
    static constexpr int kRowBytes = D * 2 + kRowPad;
    static constexpr int kTileBytes = kBS * kRowBytes;   // one K (or V) block tile
    static constexpr int kStageBytes = 2 * kTileBytes;   // K + V
    static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
};

struct Params {
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
    int num_partitions;    // P, grid.y
    int partition_blocks;  // partition_size / 16
    int64_t num_blocks;
    int *counters;   // [S * H] tickets (only S*Hk used), zero between calls
    float2 *part_ml; // [S, H, P] (m, l)
    float *part_o;   // [S, H, P, D]
    ErrorRecord *err;
};

// ---------------------------------------------------------------------------
// MMA policy: the G (<= 8) query heads of the group are rows 0..G-1 of the A
// operand; rows 8..15 are zero and never carried.  Lane l owns head row
// g = l/4 and token/dim columns 2*(l%4) + {0,1} of each 8-wide n-tile.

template <int D, int G>
struct MmaPolicy {
    static constexpr int KS = D / 16;  // k-steps of S = Q K^T
    static constexpr int NT = D / 8;   // n-tiles of O
    static constexpr bool kZeroTailRows = true;
    uint32_t qa[KS][2];
    float o[NT][2];
    float m, l;

    __device__ __forceinline__ void init(const __half *qg, float /*scale_log2*/, int lane) {
        const int g = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            if (g < G) {
                const uint32_t *row = reinterpret_cast<const uint32_t *>(qg + g * D + kk * 16);
                qa[kk][0] = __ldg(row + tig);
                qa[kk][1] = __ldg(row + 4 + tig);
            } else {
                qa[kk][0] = qa[kk][1] = 0u;
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = 0.f;
        m = kNegInf;
        l = 0.f;
    }

    // One staged block: keys at kb, values at vb (row pitch Geo<D>::kRowBytes),
    // nv valid tokens (1..16); key rows >= nv may hold anything (their scores
    // are replaced by -inf), value rows >= nv hold zeros.
    __device__ __forceinline__ void block(uint32_t kb, uint32_t vb, int nv, float scale_log2,
                                          int lane, float * /*pbuf*/) {
        constexpr int RB = Geo<D>::kRowBytes;
        const int tig = lane & 3;
        float s0[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f};
        // S = Q K^T: B fragments straight from the row-major key tile
        const uint32_t krow = kb + ((lane >> 4) * 8 + (lane & 7)) * RB + ((lane >> 3) & 1) * 16;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(b0, b1, b2, b3, krow + kk * 32);
            mma_rows0_7(s0[0], s0[1], qa[kk][0], qa[kk][1], b0, b1);
            mma_rows0_7(s1[0], s1[1], qa[kk][0], qa[kk][1], b2, b3);
        }
        float x[4] = {s0[0], s0[1], s1[0], s1[1]};
        const int t0 = tig * 2;
        const int tok[4] = {t0, t0 + 1, t0 + 8, t0 + 9};
        float mx = kNegInf;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[i] = tok[i] < nv ? x[i] * scale_log2 : kNegInf;
            mx = fmaxf(mx, x[i]);
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mnew = fmaxf(m, mx);  // finite: nv >= 1
        const float alpha = exp2f(m - mnew);
        uint32_t pa0 = pack_half2(exp2f(x[0] - mnew), exp2f(x[1] - mnew));
        uint32_t pa2 = pack_half2(exp2f(x[2] - mnew), exp2f(x[3] - mnew));
        // the normaliser sums the same fp16-rounded weights the MMA applies
        const float2 u0 = unpack_half2(pa0), u2 = unpack_half2(pa2);
        l = l * alpha + ((u0.x + u0.y) + (u2.x + u2.y));
        m = mnew;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            o[nt][0] *= alpha;
            o[nt][1] *= alpha;
        }
        // O += P V: B fragments from the row-major value tile, transposed
        const uint32_t vrow = vb + (((lane >> 3) & 1) * 8 + (lane & 7)) * RB + (lane >> 4) * 16;
#pragma unroll
        for (int nd = 0; nd < D / 16; ++nd) {
            uint32_t v0, v1, v2, v3;
            ldsm_x4_trans(v0, v1, v2, v3, vrow + nd * 32);
            mma_rows0_7(o[2 * nd][0], o[2 * nd][1], pa0, pa2, v0, v1);
            mma_rows0_7(o[2 * nd + 1][0], o[2 * nd + 1][1], pa0, pa2, v2, v3);
        }
    }

    // Write this warp's state: m[g], l[g] and o[g][D] for g < G.
    __device__ __forceinline__ void export_state(float *mw, float *lw, float *ow, int lane) {
        const int g = lane >> 2, tig = lane & 3;
        float ls = l;
        ls += __shfl_xor_sync(0xffffffffu, ls, 1);
        ls += __shfl_xor_sync(0xffffffffu, ls, 2);
        if (g < G) {
            if (tig == 0) {
                mw[g] = m;
                lw[g] = ls;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                *reinterpret_cast<float2 *>(ow + g * D + nt * 8 + tig * 2) =
                    make_float2(o[nt][0], o[nt][1]);
            }
        }
    }
};

// ---------------------------------------------------------------------------
// SIMT policy: lane l owns dims [l*DPL, (l+1)*DPL) of every head.  A chunk of
// TC tokens gives each lane TC*G partial dot products; a butterfly
// reduce-scatter leaves lane l with the full product of index l / R
// (index = token*G + head).

// Reduce-scatter of N values per lane over xor distances H, H/2, ...:
// returns the full sum of value index lane >> (5 - log2 N).
template <int N, int H>
struct ReduceScatter {
    static __device__ __forceinline__ float run(float *v, int lane) {
        const bool up = (lane & H) != 0;
#pragma unroll
        for (int j = 0; j < N / 2; ++j) {
            const float send = up ? v[j] : v[j + N / 2];
            const float keep = up ? v[j + N / 2] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, H);
        }
        return ReduceScatter<N / 2, H / 2>::run(v, lane);
    }
};
template <int H>
struct ReduceScatter<1, H> {
    static __device__ __forceinline__ float run(float *v, int /*lane*/) {
        float x = v[0];
#pragma unroll
        for (int h = H; h >= 1; h >>= 1) x += __shfl_xor_sync(0xffffffffu, x, h);
        return x;
    }
};

template <int D, int G>
struct SimtPolicy {
    static constexpr int DPL = D / 32;                    // dims per lane: 4 or 2
    static constexpr int TC = (32 / G) < kBS ? 32 / G : kBS;  // tokens per chunk
    static constexpr int NCH = kBS / TC;                  // chunks per block
    static constexpr int NV = TC * G;                     // values per chunk per lane
    static constexpr int R = 32 / NV;                     // lanes holding the same result
    static constexpr bool kZeroTailRows = false;          // reads rows < nv only
    float q[G][DPL];  // pre-scaled by scale*log2(e)
    float o[G][DPL];
    float m_all[G];   // running max of every head (same in all lanes)
    float m_own, l_own;

    __device__ __forceinline__ static int own_head(int lane) { return (lane / R) % G; }

    __device__ __forceinline__ void init(const __half *qg, float scale_log2, int lane) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int i = 0; i < DPL; ++i) {
                q[g][i] = __half2float(qg[g * D + lane * DPL + i]) * scale_log2;
                o[g][i] = 0.f;
            }
            m_all[g] = kNegInf;
        }
        m_own = kNegInf;
        l_own = 0.f;
    }

    __device__ __forceinline__ void load_row(uint32_t addr, float (&x)[DPL]) const {
        if constexpr (DPL == 4) {
            uint32_t a, b;
            asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr));
            const float2 f0 = unpack_half2(a), f1 = unpack_half2(b);
            x[0] = f0.x; x[1] = f0.y; x[2] = f1.x; x[3] = f1.y;
        } else {
            uint32_t a;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a) : "r"(addr));
            const float2 f0 = unpack_half2(a);
            x[0] = f0.x; x[1] = f0.y;
        }
    }

    __device__ __forceinline__ void block(uint32_t kb, uint32_t vb, int nv, float /*scale*/,
                                          int lane, float *pbuf) {
        constexpr int RB = Geo<D>::kRowBytes;
        const uint32_t lane_off = lane * DPL * 2;
        const int idx = lane / R;  // result index held by this lane: token*G + head
        float s[NCH];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            float part[NV];
#pragma unroll
            for (int t = 0; t < TC; ++t) {
                float kx[DPL];
                load_row(kb + (c * TC + t) * RB + lane_off, kx);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < DPL; ++i) acc = fmaf(q[g][i], kx[i], acc);
                    part[t * G + g] = acc;
                }
            }
            const float full = ReduceScatter<NV, 16>::run(part, lane);
            s[c] = (c * TC + idx / G) < nv ? full : kNegInf;
        }
        // block max of this lane's head, over the token bits of the lane index
        float mx = s[0];
#pragma unroll
        for (int c = 1; c < NCH; ++c) mx = fmaxf(mx, s[c]);
#pragma unroll
        for (int h = R * G; h < 32; h <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, h));
        float alpha[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float mb = __shfl_sync(0xffffffffu, mx, g * R);
            const float mnew = fmaxf(m_all[g], mb);
            alpha[g] = exp2f(m_all[g] - mnew);
            m_all[g] = mnew;
        }
        const float mnew_own = fmaxf(m_own, mx);
        const float alpha_own = exp2f(m_own - mnew_own);
        m_own = mnew_own;
        float psum = 0.f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const float pc = exp2f(s[c] - mnew_own);
            psum += pc;
            if (lane % R == 0) pbuf[(c * TC + idx / G) * G + idx % G] = pc;
        }
        l_own = l_own * alpha_own + psum;
        __syncwarp();
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int i = 0; i < DPL; ++i) o[g][i] *= alpha[g];
        for (int t = 0; t < nv; ++t) {
            float vx[DPL];
            load_row(vb + t * RB + lane_off, vx);
            float pt[G];
#pragma unroll
            for (int g = 0; g < G; ++g) pt[g] = pbuf[t * G + g];
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int i = 0; i < DPL; ++i) o[g][i] = fmaf(pt[g], vx[i], o[g][i]);
        }
        __syncwarp();
    }

    __device__ __forceinline__ void export_state(float *mw, float *lw, float *ow, int lane) {
        float ls = l_own;
#pragma unroll
        for (int h = R * G; h < 32; h <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, h);
        if (lane < G * R && lane % R == 0) {
            mw[own_head(lane)] = m_own;
            lw[own_head(lane)] = ls;
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int i = 0; i < DPL; ++i) ow[g * D + lane * DPL + i] = o[g][i];
    }
};

// ---------------------------------------------------------------------------
// Shared-memory layout (dynamic):
//   ring    kWarps * kStages * (K tile + V tile)      -- aliased after the main
//           loop by the warp merge and the partition combine
//   bars    kWarps * kStages mbarriers
//   bt      partition_blocks int32 (block ids of this partition, -1 = bad)
//   misc    4 int32 (abort flag, last-CTA flag)
//   pbuf    kWarps * 16 * G fp32 (SIMT only: softmax weights of a block)

template <int D, int G>
__host__ __device__ constexpr int smem_fixed_bytes() {
    return Geo<D>::kRingBytes + kWarps * kStages * 8 + 4 * 4 + kWarps * kBS * G * 4;
}

__host__ __device__ inline int smem_bytes_for(int D, int G, int partition_blocks) {
    const int ring = kWarps * kStages * 2 * kBS * (D * 2 + kRowPad);
    return ring + kWarps * kStages * 8 + partition_blocks * 4 + 4 * 4 + kWarps * kBS * G * 4;
}

template <int D, int G, class Policy>
__global__ void __launch_bounds__(kThreads) decode_kernel(const Params p) {
    using Gm = Geo<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Gm::kRingBytes);
    int *bt_s = reinterpret_cast<int *>(bars + kWarps * kStages);
    int *misc = bt_s + p.partition_blocks;
    float *pbuf_all = reinterpret_cast<float *>(misc + 4);

    const int kvh = blockIdx.x, part = blockIdx.y, seq = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.num_heads;
    const int P = p.num_partitions;

    // Launched with programmatic stream serialization: everything above ran
    // while the previous kernel (typically the cache write) drained; no input
    // is read before that kernel's results are visible.
    grid_dependency_wait();

    // ---- sequence length and this CTA's share of it
    int L = __ldg(p.seq_lens + seq);
    const int cap = min(p.max_blocks_per_seq, P * p.partition_blocks) * kBS;
    if (L < 0 || L > cap) {
        if (threadIdx.x == 0 && kvh == 0 && part == 0)
            record_error(p.err, PKV_DEVERR_SEQ_LEN, seq);
        L = L < 0 ? 0 : cap;
    }
    const int nblk_seq = (L + kBS - 1) / kBS;
    const int nparts = max(1, (nblk_seq + p.partition_blocks - 1) / p.partition_blocks);
    if (part >= nparts) return;  // whole CTA: nothing of this sequence here
    const int blk0 = part * p.partition_blocks;
    const int nblk = min(p.partition_blocks, nblk_seq - blk0);  // >= 0

    // ---- set-up: block-table slice, mbarriers
    const int32_t *bt_row = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq;
    for (int j = threadIdx.x; j < nblk; j += kThreads) {
        int b = __ldg(bt_row + blk0 + j);
        if (b < 0 || static_cast<int64_t>(b) >= p.num_blocks) {
            record_error(p.err, PKV_DEVERR_BLOCK_ID,
                         static_cast<int64_t>(seq) * p.max_blocks_per_seq + blk0 + j);
            b = -1;
        }
        bt_s[j] = b;
    }
    if (threadIdx.x == 0) misc[0] = 0;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&bars[warp * kStages + s]), 1);
        fence_mbarrier_init();
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- per-warp pipeline over blocks warp, warp+4, warp+8, ...
    Policy st;
    const __half *qg = p.q + (static_cast<int64_t>(seq) * H + kvh * G) * D;
    st.init(qg, p.scale_log2, lane);
    float *pbuf = pbuf_all + warp * kBS * G;

    const int nw = nblk > warp ? (nblk - warp + kWarps - 1) / kWarps : 0;
    const uint32_t ring_s = smem_u32(ring + warp * kStages * Gm::kStageBytes);
    const uint32_t bar_s = smem_u32(&bars[warp * kStages]);
    const int64_t row_elems = static_cast<int64_t>(p.num_kv_heads) * D;
    const __half *kbase = p.k_cache + kvh * D;
    const __half *vbase = p.v_cache + kvh * D;

    auto valid_tokens = [&](int i) -> int {
        const int j = warp + i * kWarps;
        return bt_s[j] < 0 ? 0 : min(kBS, L - (blk0 + j) * kBS);
    };
    auto issue = [&](int i) {
        const int j = warp + i * kWarps;
        const int nv = valid_tokens(i);
        const int s = i % kStages;
        const uint32_t bar = bar_s + s * 8;
        if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nv) * D * 2 * 2);
        __syncwarp();
        const int r = lane & (kBS - 1);
        if (r < nv) {
            const int64_t row = (static_cast<int64_t>(bt_s[j]) * kBS + r) * row_elems;
            const __half *src = (lane < kBS ? kbase : vbase) + row;
            const uint32_t dst =
                ring_s + s * Gm::kStageBytes + (lane < kBS ? 0 : Gm::kTileBytes) + r * Gm::kRowBytes;
            bulk_g2s(dst, src, D * 2, bar);
        }
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
            if (Policy::kZeroTailRows && nv < kBS) {
                // value rows past a partial block meet weight 0 in the MMA and
                // must hold finite numbers: zero them (stale rows are finite)
                for (int e = lane; e < (kBS - nv) * (D / 8); e += 32) {
                    const uint32_t a = kb + Gm::kTileBytes + (nv + e / (D / 8)) * Gm::kRowBytes +
                                       (e % (D / 8)) * 16;
                    asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(a), "r"(0u)
                                 : "memory");
                }
                __syncwarp();
            }
            st.block(kb, kb + Gm::kTileBytes, nv, p.scale_log2, lane, pbuf);
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
                         (static_cast<int64_t>(seq) * gridDim.y + part) * gridDim.x + kvh);
        const int stop = (i + kStages < nw) ? i + kStages : nw;
        for (int k = i; k < stop; ++k) mbar_wait_bounded(bar_s + (k % kStages) * 8, (k / kStages) & 1);
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

    // ---- split-KV: the last CTA of this (sequence, kv_head) combines
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        int *ticket = p.counters + static_cast<int64_t>(seq) * p.num_kv_heads + kvh;
        const int prev = atomicAdd(ticket, 1);
        const int last = prev == nparts - 1;
        if (last) atomicExch(ticket, 0);  // leave the workspace zeroed
        misc[1] = last;
    }
    __syncthreads();
    if (misc[1] == 0) return;
    __threadfence();

    // combine scratch, aliasing the idle ring
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

// ---------------------------------------------------------------------------
// Host side.

using KernelFn = void (*)(const Params);

template <int D, int G>
KernelFn pick(int compute) {
    if (compute == PKV_COMPUTE_SIMT) return decode_kernel<D, G, SimtPolicy<D, G>>;
    return decode_kernel<D, G, MmaPolicy<D, G>>;
}

KernelFn select_kernel(int D, int G, int compute) {
    if (D == 128) {
        switch (G) {
            case 1: return pick<128, 1>(compute);
            case 2: return pick<128, 2>(compute);
            case 4: return pick<128, 4>(compute);
            case 8: return pick<128, 8>(compute);
        }
    } else if (D == 64) {
        switch (G) {
            case 1: return pick<64, 1>(compute);
            case 2: return pick<64, 2>(compute);
            case 4: return pick<64, 4>(compute);
            case 8: return pick<64, 8>(compute);
        }
    }
    return nullptr;
}

inline int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

int64_t workspace_bytes(int64_t S, int64_t H, int64_t D, int64_t P) {
    if (P <= 1) return 0;
    return align256(S * H * 4) + align256(S * H * P * 8) + S * H * P * D * 4;
}

int resolve_partition(const pkv_decode_options *opts) {
    return (opts && opts->partition_size) ? opts->partition_size : kDefaultPartitionTokens;
}

}  // namespace dec
}  // namespace pkv

extern "C" {

size_t pkv_decode_workspace_bytes_ex(int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                                     int32_t max_seq_len, int32_t partition_size) {
    using namespace pkv::dec;
    const int pt = partition_size ? partition_size : kDefaultPartitionTokens;
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_seq_len <= 0 || pt <= 0) return 0;
    const int64_t P = (static_cast<int64_t>(max_seq_len) + pt - 1) / pt;
    return static_cast<size_t>(workspace_bytes(num_seqs, num_heads, head_dim, P));
}

size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                                  int32_t max_seq_len) {
    return pkv_decode_workspace_bytes_ex(num_seqs, num_heads, head_dim, max_seq_len, 0);
}

int pkv_decode_workspace_init(void *workspace, size_t workspace_bytes, pkv_stream_t stream) {
    if (workspace_bytes == 0) return PKV_OK;
    if (workspace == nullptr) return PKV_ERR_NULL;
    cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes,
                                    reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : pkv::cuda_failure(e, "cudaMemsetAsync(workspace)");
}

int pkv_decode_attention_ex(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *seq_lens, float scale,
                            int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_seqs, int32_t max_blocks_per_seq,
                            int32_t max_seq_len, int64_t num_blocks, void *workspace,
                            size_t workspace_bytes_given, const pkv_decode_options *opts,
                            pkv_stream_t stream) {
    using namespace pkv;
    using namespace pkv::dec;
    if (num_seqs < 0) return PKV_ERR_INVALID;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PKV_ERR_NULL;
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || max_seq_len < 0 ||
        !std::isfinite(scale))
        return PKV_ERR_INVALID;
    const int G = num_heads / num_kv_heads;
    if (!(G == 1 || G == 2 || G == 4 || G == 8)) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != kBS) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
    const int pt = resolve_partition(opts);
    if (pt < kBS || pt > kMaxPartitionTokens || pt % kBS != 0) return PKV_ERR_INVALID;
    const int compute = opts ? opts->compute : PKV_COMPUTE_AUTO;
    if (compute < PKV_COMPUTE_AUTO || compute > PKV_COMPUTE_MMA) return PKV_ERR_INVALID;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PKV_ERR_ALIGNMENT;
    const int64_t P64 = std::max<int64_t>(1, (static_cast<int64_t>(max_seq_len) + pt - 1) / pt);
    if (P64 > 65535) return PKV_ERR_UNSUPPORTED;
    const int P = static_cast<int>(P64);
    const int partition_blocks = pt / kBS;

    Params p;
    p.out = static_cast<__half *>(out);
    p.q = static_cast<const __half *>(q);
    p.k_cache = static_cast<const __half *>(k_cache);
    p.v_cache = static_cast<const __half *>(v_cache);
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_partitions = P;
    p.partition_blocks = partition_blocks;
    p.num_blocks = num_blocks;
    p.counters = nullptr;
    p.part_ml = nullptr;
    p.part_o = nullptr;
    if (P > 1) {
        const int64_t need = workspace_bytes(num_seqs, num_heads, head_dim, P);
        if (workspace == nullptr || static_cast<int64_t>(workspace_bytes_given) < need)
            return PKV_ERR_WORKSPACE;
        if (!aligned(workspace, 16)) return PKV_ERR_ALIGNMENT;
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        const int64_t c_bytes = align256(static_cast<int64_t>(num_seqs) * num_heads * 4);
        const int64_t ml_bytes = align256(static_cast<int64_t>(num_seqs) * num_heads * P * 8);
        p.counters = reinterpret_cast<int *>(ws);
        p.part_ml = reinterpret_cast<float2 *>(ws + c_bytes);
        p.part_o = reinterpret_cast<float *>(ws + c_bytes + ml_bytes);
        // the combine's per-partition weights must fit in the (aliased) ring
        const int ring = kWarps * kStages * 2 * kBS * (head_dim * 2 + kRowPad);
        if (static_cast<int64_t>(2 * G * P + 2 * G) * 4 > ring) return PKV_ERR_UNSUPPORTED;
    }
    p.err = device_error_record();
    if (p.err == nullptr) return PKV_ERR_CUDA;

    const int comp = compute == PKV_COMPUTE_SIMT ? PKV_COMPUTE_SIMT : PKV_COMPUTE_MMA;
    KernelFn fn = select_kernel(head_dim, G, comp);
    if (fn == nullptr) return PKV_ERR_UNSUPPORTED;
    const int smem = smem_bytes_for(head_dim, G, partition_blocks);
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_failure(e, "cudaFuncSetAttribute(decode)");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_kv_heads, P, num_seqs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fn, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_failure(e, "decode_kernel launch");
}

int pkv_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *seq_lens, float scale,
                         int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int32_t num_seqs, int32_t max_blocks_per_seq,
                         int32_t max_seq_len, int64_t num_blocks, void *workspace,
                         size_t workspace_bytes, pkv_stream_t stream) {
    return pkv_decode_attention_ex(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                                   num_heads, num_kv_heads, head_dim, block_size, num_seqs,
                                   max_blocks_per_seq, max_seq_len, num_blocks, workspace,
                                   workspace_bytes, nullptr, stream);
}

}  // extern "C"
