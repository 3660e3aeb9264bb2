// pkv_decode_common.cuh -- per-block arithmetic of paged decode attention,
// shared by both schedules ("deep-dive-into-vllm-05" §2 read loop, §3.2 GQA;
// "vLLM 技术内幕" §2.1: dot the query with the keys of each physical block in
// turn, accumulate the values block by block).
//
// A compute policy owns one warp's running state for the G query heads of
// one (sequence, kv_head): the running max m and sum l of the online softmax
// (log2 domain: scores are pre-multiplied by scale*log2(e)) and the
// unnormalised output o.  `block` folds one staged block of 16 keys/values
// into the state:
//     m' = max(m, max_t s_t),  alpha = 2^(m - m'),  p_t = 2^(s_t - m'),
//     l' = alpha*l + sum_t p_t,  o' = alpha*o + sum_t p_t v_t.
// Staged rows sit `pitch` bytes apart in shared memory; the pitch is 16
// bytes more than a multiple of 128 so that 8 consecutive rows start in 8
// different 16-byte bank groups (conflict-free ldmatrix / vector loads).
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include <cmath>

#include "pkv_device.cuh"

namespace pkv {
namespace dec {

constexpr int kBS = 16;      // tokens per physical block on the decode path
constexpr int kRowPad = 16;  // staged row pitch = row bytes + 16
constexpr float kNegInf = -INFINITY;

// ---------------------------------------------------------------------------
// MMA policy: the G (<= 8) query heads are rows 0..G-1 of the 16-row A
// operand of m16n8k16 fp16 MMAs with fp32 accumulation; rows 8..15 are zero
// and never carried.  Lane l owns head row g = l/4 and columns 2*(l%4)+{0,1}
// of every 8-wide n-tile (tokens for S = Q K^T, head dims for O += P V).

template <int D, int G>
struct MmaPolicy {
    static constexpr int KS = D / 16;  // k-steps of S = Q K^T
    static constexpr int NT = D / 8;   // n-tiles of O
    static constexpr bool kZeroTailRows = true;  // reads all 16 value rows
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

    // One staged block: keys at kb, values at vb (rows `pitch` bytes apart),
    // nv valid tokens (1..16).  Key rows >= nv may hold anything (their
    // scores become -inf); value rows >= nv must hold finite numbers.
    __device__ __forceinline__ void block(uint32_t kb, uint32_t vb, uint32_t pitch, int nv,
                                          float scale_log2, int lane, float * /*pbuf*/) {
        const int tig = lane & 3;
        float s0[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f};
        // S = Q K^T: B fragments straight from the row-major key tile
        const uint32_t krow = kb + ((lane >> 4) * 8 + (lane & 7)) * pitch + ((lane >> 3) & 1) * 16;
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
        const uint32_t pa0 = pack_half2(exp2f(x[0] - mnew), exp2f(x[1] - mnew));
        const uint32_t pa2 = pack_half2(exp2f(x[2] - mnew), exp2f(x[3] - mnew));
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
        const uint32_t vrow = vb + (((lane >> 3) & 1) * 8 + (lane & 7)) * pitch + (lane >> 4) * 16;
#pragma unroll
        for (int nd = 0; nd < D / 16; ++nd) {
            uint32_t v0, v1, v2, v3;
            ldsm_x4_trans(v0, v1, v2, v3, vrow + nd * 32);
            mma_rows0_7(o[2 * nd][0], o[2 * nd][1], pa0, pa2, v0, v1);
            mma_rows0_7(o[2 * nd + 1][0], o[2 * nd + 1][1], pa0, pa2, v2, v3);
        }
    }

    __device__ __forceinline__ float l_total() const {
        float ls = l;
        ls += __shfl_xor_sync(0xffffffffu, ls, 1);
        ls += __shfl_xor_sync(0xffffffffu, ls, 2);
        return ls;
    }

    // Shared-memory export for a CTA merge: m[g], l[g], o[g][D] for g < G.
    __device__ __forceinline__ void export_state(float *mw, float *lw, float *ow, int lane) {
        const int g = lane >> 2, tig = lane & 3;
        const float ls = l_total();
        if (g < G) {
            if (tig == 0) {
                mw[g] = m;
                lw[g] = ls;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                *reinterpret_cast<float2 *>(ow + g * D + nt * 8 + tig * 2) =
                    make_float2(o[nt][0], o[nt][1]);
        }
    }

    // Final fp16 output o / l of heads g < G at out_g0 + g*D (zeros if empty).
    __device__ __forceinline__ void write_output(__half *out_g0, int lane) {
        const int g = lane >> 2, tig = lane & 3;
        const float ls = l_total();
        if (g < G) {
            const float inv = ls > 0.f ? 1.f / ls : 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                *reinterpret_cast<__half2 *>(out_g0 + g * D + nt * 8 + tig * 2) =
                    __floats2half2_rn(o[nt][0] * inv, o[nt][1] * inv);
        }
    }

    // Partial state to global memory: ml[g] = (m, l), o[g*D + d].
    __device__ __forceinline__ void write_partial(float2 *ml, float *og, int lane) {
        const int g = lane >> 2, tig = lane & 3;
        const float ls = l_total();
        if (g < G) {
            if (tig == 0) ml[g] = make_float2(m, ls);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                *reinterpret_cast<float2 *>(og + g * D + nt * 8 + tig * 2) =
                    make_float2(o[nt][0], o[nt][1]);
        }
    }
};

// ---------------------------------------------------------------------------
// MMA policy over FP8 (E4M3) staged tiles, fed to the fp16 MMA without a
// shared-memory round trip.  Keys: a non-transposed ldmatrix gives lane l
// the 4 codes of dims 4*(l%4)..+3 of token l/4 (per 16-dim, 8-token
// matrix); their fp16 conversion is the B fragment of a k16 step under the
// contraction-index permutation k = 2t+j -> 4t+j, k = 8+2t+j -> 4t+2+j,
// which the query fragments follow (one 64-bit load per k-step).  Values: a
// transposed ldmatrix gives lane l the codes of tokens 2*(l%4)+{0,1} at
// dims 2*(l/4)+{0,1}; byte permutes split them into an even-dim and an
// odd-dim B fragment, so O's n-tile 2c+e holds dims 16c + 2n + e.
// The key scale multiplies the score and the value scale the softmax weight
// (each factors out of its sum); the weights also carry an exact factor of
// 256, removed on output, to keep them clear of fp16 subnormals.

__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint32_t two_codes) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
        static_cast<__nv_fp8x2_storage_t>(two_codes & 0xffffu), __NV_E4M3);
    return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

__device__ __forceinline__ uint32_t byte_perm(uint32_t x, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(0u), "r"(sel));
    return r;
}

template <int D, int G>
struct MmaFp8Policy {
    static constexpr int KS = D / 16;
    static constexpr int NT = D / 8;
    static constexpr float kWeightBoost = 256.f;  // exact; removed on output
    uint32_t qa[KS][2];
    float o[NT][2];
    float m, l;

    __device__ __forceinline__ void init(const __half *qg, float /*scale_log2*/, int lane) {
        const int g = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            if (g < G) {
                const uint2 w = __ldg(reinterpret_cast<const uint2 *>(qg + g * D + kk * 16 + tig * 4));
                qa[kk][0] = w.x;
                qa[kk][1] = w.y;
            } else {
                qa[kk][0] = qa[kk][1] = 0u;
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = 0.f;
        m = kNegInf;
        l = 0.f;
    }

    // kb8 / vb8: this head's key / value codes of the staged block (rows
    // `pitch` bytes apart); value rows >= nv must hold finite codes.
    __device__ __forceinline__ void block(uint32_t kb8, uint32_t vb8, uint32_t pitch, int nv,
                                          float scale_log2, int lane, const float (&ks)[4],
                                          const float (&vs)[4]) {
        const int tig = lane & 3;
        const uint32_t row = (((lane >> 3) & 1) * 8 + (lane & 7)) * pitch + (lane >> 4) * 16;
        float s0[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f};
#pragma unroll
        for (int kp = 0; kp < D / 32; ++kp) {
            uint32_t r0, r1, r2, r3;  // tokens 0-7 / 8-15, dims 32kp.. / 32kp+16..
            ldsm_x4(r0, r1, r2, r3, kb8 + row + kp * 32);
            mma_rows0_7(s0[0], s0[1], qa[2 * kp][0], qa[2 * kp][1], e4m3x2_to_half2(r0),
                        e4m3x2_to_half2(r0 >> 16));
            mma_rows0_7(s1[0], s1[1], qa[2 * kp][0], qa[2 * kp][1], e4m3x2_to_half2(r1),
                        e4m3x2_to_half2(r1 >> 16));
            mma_rows0_7(s0[0], s0[1], qa[2 * kp + 1][0], qa[2 * kp + 1][1], e4m3x2_to_half2(r2),
                        e4m3x2_to_half2(r2 >> 16));
            mma_rows0_7(s1[0], s1[1], qa[2 * kp + 1][0], qa[2 * kp + 1][1], e4m3x2_to_half2(r3),
                        e4m3x2_to_half2(r3 >> 16));
        }
        float x[4] = {s0[0], s0[1], s1[0], s1[1]};
        const int t0 = tig * 2;
        const int tok[4] = {t0, t0 + 1, t0 + 8, t0 + 9};
        float mx = kNegInf;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[i] = tok[i] < nv ? (x[i] * ks[i]) * scale_log2 : kNegInf;
            mx = fmaxf(mx, x[i]);
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mnew = fmaxf(m, mx);
        const float alpha = exp2f(m - mnew);
        float pw[4], psum = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float pi = exp2f(x[i] - mnew);
            psum += pi;
            pw[i] = tok[i] < nv ? pi * (vs[i] * kWeightBoost) : 0.f;
        }
        const uint32_t pa0 = pack_half2(pw[0], pw[1]);
        const uint32_t pa2 = pack_half2(pw[2], pw[3]);
        l = l * alpha + psum;
        m = mnew;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            o[nt][0] *= alpha;
            o[nt][1] *= alpha;
        }
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
            uint32_t r0, r1, r2, r3;  // tokens 0-7 / 8-15, dims 32q.. / 32q+16..
            ldsm_x4_trans(r0, r1, r2, r3, vb8 + row + q * 32);
            // even dims: bytes 0 and 2; odd dims: bytes 1 and 3
            mma_rows0_7(o[4 * q][0], o[4 * q][1], pa0, pa2,
                        e4m3x2_to_half2(byte_perm(r0, 0x20)), e4m3x2_to_half2(byte_perm(r1, 0x20)));
            mma_rows0_7(o[4 * q + 1][0], o[4 * q + 1][1], pa0, pa2,
                        e4m3x2_to_half2(byte_perm(r0, 0x31)), e4m3x2_to_half2(byte_perm(r1, 0x31)));
            mma_rows0_7(o[4 * q + 2][0], o[4 * q + 2][1], pa0, pa2,
                        e4m3x2_to_half2(byte_perm(r2, 0x20)), e4m3x2_to_half2(byte_perm(r3, 0x20)));
            mma_rows0_7(o[4 * q + 3][0], o[4 * q + 3][1], pa0, pa2,
                        e4m3x2_to_half2(byte_perm(r2, 0x31)), e4m3x2_to_half2(byte_perm(r3, 0x31)));
        }
    }

    __device__ __forceinline__ float l_total() const {
        float ls = l;
        ls += __shfl_xor_sync(0xffffffffu, ls, 1);
        ls += __shfl_xor_sync(0xffffffffu, ls, 2);
        return ls;
    }

    // n-tile pair (2c, 2c+1), element j: dims 16c + 4t + 2j and the next one
    __device__ __forceinline__ void write_output(__half *out_g0, int lane) {
        const int g = lane >> 2, tig = lane & 3;
        const float ls = l_total();
        if (g < G) {
            const float inv = ls > 0.f ? (1.f / kWeightBoost) / ls : 0.f;
#pragma unroll
            for (int c = 0; c < NT / 2; ++c)
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    *reinterpret_cast<__half2 *>(out_g0 + g * D + 16 * c + 4 * tig + 2 * j) =
                        __floats2half2_rn(o[2 * c][j] * inv, o[2 * c + 1][j] * inv);
        }
    }

    __device__ __forceinline__ void write_partial(float2 *ml, float *og, int lane) {
        const int g = lane >> 2, tig = lane & 3;
        const float ls = l_total();
        if (g < G) {
            if (tig == 0) ml[g] = make_float2(m, ls);
            const float u = 1.f / kWeightBoost;
#pragma unroll
            for (int c = 0; c < NT / 2; ++c)
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    *reinterpret_cast<float2 *>(og + g * D + 16 * c + 4 * tig + 2 * j) =
                        make_float2(o[2 * c][j] * u, o[2 * c + 1][j] * u);
        }
    }
};

// Zero the value codes of rows [nv, 16) of one head (D bytes per row), then
// order those generic-proxy writes before later bulk copies into the stage.
template <int D>
__device__ __forceinline__ void zero_tail_rows_fp8(uint32_t vb8, uint32_t pitch, int nv, int lane) {
    for (int e = lane; e < (kBS - nv) * (D / 16); e += 32) {
        const uint32_t a = vb8 + (nv + e / (D / 16)) * pitch + (e % (D / 16)) * 16;
        asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(a), "r"(0u) : "memory");
    }
    fence_proxy_async_smem();
    __syncwarp();
}

// ---------------------------------------------------------------------------
// SIMT policy (fp32 FMAs on CUDA cores): lane l owns dims [l*DPL, (l+1)*DPL)
// of every head.  A chunk of TC tokens gives each lane TC*G partial dot
// products; a butterfly reduce-scatter leaves lane l with the full product
// of index l / R (index = token*G + head).

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
    static constexpr int DPL = D / 32;                        // dims per lane: 4 or 2
    static constexpr int TC = (32 / G) < kBS ? 32 / G : kBS;  // tokens per chunk
    static constexpr int NCH = kBS / TC;                      // chunks per block
    static constexpr int NV = TC * G;                         // values per chunk per lane
    static constexpr int R = 32 / NV;                         // lanes holding one result
    static constexpr bool kZeroTailRows = false;              // reads rows < nv only
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
            x[0] = f0.x;
            x[1] = f0.y;
            x[2] = f1.x;
            x[3] = f1.y;
        } else {
            uint32_t a;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a) : "r"(addr));
            const float2 f0 = unpack_half2(a);
            x[0] = f0.x;
            x[1] = f0.y;
        }
    }

    __device__ __forceinline__ void block(uint32_t kb, uint32_t vb, uint32_t pitch, int nv,
                                          float /*scale*/, int lane, float *pbuf) {
        const uint32_t lane_off = lane * DPL * 2;
        const int idx = lane / R;  // result index held by this lane: token*G + head
        float s[NCH];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            float part[NV];
#pragma unroll
            for (int t = 0; t < TC; ++t) {
                float kx[DPL];
                load_row(kb + (c * TC + t) * pitch + lane_off, kx);
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
            load_row(vb + t * pitch + lane_off, vx);
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

    // Sum of this lane's head over the lanes sharing it.
    __device__ __forceinline__ float l_own_total() const {
        float ls = l_own;
#pragma unroll
        for (int h = R * G; h < 32; h <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, h);
        return ls;
    }

    __device__ __forceinline__ void export_state(float *mw, float *lw, float *ow, int lane) {
        const float ls = l_own_total();
        if (lane < G * R && lane % R == 0) {
            mw[own_head(lane)] = m_own;
            lw[own_head(lane)] = ls;
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int i = 0; i < DPL; ++i) ow[g * D + lane * DPL + i] = o[g][i];
    }

    __device__ __forceinline__ void write_output(__half *out_g0, int lane) {
        const float ls = l_own_total();
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float lg = __shfl_sync(0xffffffffu, ls, g * R);
            const float inv = lg > 0.f ? 1.f / lg : 0.f;
#pragma unroll
            for (int i = 0; i < DPL; i += 2)
                *reinterpret_cast<__half2 *>(out_g0 + g * D + lane * DPL + i) =
                    __floats2half2_rn(o[g][i] * inv, o[g][i + 1] * inv);
        }
    }

    __device__ __forceinline__ void write_partial(float2 *ml, float *og, int lane) {
        const float ls = l_own_total();
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float lg = __shfl_sync(0xffffffffu, ls, g * R);
            if (lane == 0) ml[g] = make_float2(m_all[g], lg);
#pragma unroll
            for (int i = 0; i < DPL; ++i) og[g * D + lane * DPL + i] = o[g][i];
        }
    }
};

// Zero value rows [nv, 16) of one head's staged tile (row bytes D*2), then
// order those generic-proxy writes before later bulk copies into the stage.
template <int D>
__device__ __forceinline__ void zero_tail_rows(uint32_t vb, uint32_t pitch, int nv, int lane) {
    for (int e = lane; e < (kBS - nv) * (D / 8); e += 32) {
        const uint32_t a = vb + (nv + e / (D / 8)) * pitch + (e % (D / 8)) * 16;
        asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(a), "r"(0u) : "memory");
    }
    fence_proxy_async_smem();
    __syncwarp();
}

}  // namespace dec
}  // namespace pkv
