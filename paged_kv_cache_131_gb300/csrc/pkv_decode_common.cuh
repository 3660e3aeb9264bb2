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
// A staged tile is the 16 token rows of one block, brought by one tiled
// tensor copy (TMA) and laid out chunk-major with the copy's swizzle
// (SwizzledTile): 8 tokens reading the same 16 bytes of their rows hit 8
// different 16-byte bank groups, so every ldmatrix is conflict-free.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include <cmath>

#include "pkv_decode_host.h"
#include "pkv_device.cuh"

namespace pkv {
namespace dec {

constexpr int kBS = 16;  // tokens per physical block on the decode path
constexpr float kNegInf = -INFINITY;

// Where byte b of token t's row sits in a staged tile.  The tensor copy
// stores the tile chunk-major -- chunk c (bytes [c*C, (c+1)*C) of every row)
// is 16 rows of C bytes -- and swizzles the 16-byte units of each row: unit
// u of token t lands at u ^ (t & 7) for C = 128 (the 128-byte swizzle) or
// u ^ ((t >> 1) & 3) for C = 64 (the 64-byte swizzle).  The tile base is
// 1024-byte aligned.  b keeps its low 4 bits.
struct SwizzledTile {
    uint32_t log_c;  // log2 of the chunk bytes: 7 or 6
    __device__ __forceinline__ uint32_t at(int t, uint32_t b) const {
        const uint32_t c = b >> log_c;
        const uint32_t u = (b >> 4) & ((1u << (log_c - 4)) - 1u);
        const uint32_t x = log_c == 7 ? (t & 7) : ((t >> 1) & 3);
        return (c << (log_c + 4)) + (static_cast<uint32_t>(t) << log_c) + ((u ^ x) << 4) +
               (b & 15u);
    }
};

// ---------------------------------------------------------------------------
// MMA policy (fp16 tiles, m16n8k16 MMAs with fp32 accumulation), both
// products transposed so that the 16 MMA rows are tokens or head dims and
// the G (<= 8) query heads are the 8 columns:
//   S^T = K Q^T: A = the key tile (ldmatrix, rows = tokens), B = the query
//     (loaded once per sequence).  Lane l holds the scores of tokens l/4 and
//     l/4 + 8 for heads 2*(l%4) and 2*(l%4)+1 and keeps the online-softmax
//     state of those two heads (max over tokens: a butterfly over the lanes
//     of one l%4).
//   O^T = V^T P^T: A = the value tile (transposed ldmatrix, rows = dims),
//     B = the fp16 weights, transposed per 8x8 half by movmatrix.  O^T's
//     columns are the same two heads.

template <int D, int G>
struct MmaPolicy {
    static constexpr bool kColumns = false;  // columns = the G heads of one new token
    static constexpr int kRows = G;          // partial-state rows per (sequence, kv head)
    static constexpr int KS = D / 16;  // k-steps of S^T (16 head dims each)
    static constexpr int MT = D / 16;  // m-tiles (16 head dims each) of O^T
    static constexpr bool kZeroTailRows = true;  // reads all 16 value rows
    uint32_t qb[KS][2];  // B operand of S^T: query dims of head l/4
    // O^T, m-tile mt: c0 / c2 = dims 16mt + g / + g + 8 of head 2t, c1 / c3
    // the same dims of head 2t+1 (g = lane/4, t = lane%4)
    float o[MT][4];
    float m[2], l[2];  // softmax state of heads 2t, 2t+1 (l: this lane's tokens)

    __device__ __forceinline__ void init(const __half *qg, float /*scale_log2*/, int lane) {
        const int g = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            if (g < G) {
                const uint32_t *row = reinterpret_cast<const uint32_t *>(qg + g * D + kk * 16);
                qb[kk][0] = __ldg(row + tig);
                qb[kk][1] = __ldg(row + 4 + tig);
            } else {
                qb[kk][0] = qb[kk][1] = 0u;
            }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m[0] = m[1] = kNegInf;
        l[0] = l[1] = 0.f;
    }

    // One staged block: key tile at kb, value tile at vb, this head's bytes
    // starting at `head` within each row; nv valid tokens (1..16).  Key rows
    // >= nv may hold anything (their scores become -inf); value rows >= nv
    // must hold finite numbers.
    __device__ __forceinline__ void block(uint32_t kb, uint32_t vb, SwizzledTile tile,
                                          uint32_t head, int nv, float scale_log2, int lane,
                                          float * /*pbuf*/) {
        const int g = lane >> 2;
        // S^T = K Q^T; ldmatrix matrices: tokens 0-7 / 8-15 (rows g / g+8 of
        // A) at dims 0-7, then the same at dims 8-15; two accumulator chains
        const int rt = ((lane >> 3) & 1) * 8 + (lane & 7);
        const uint32_t kcol = head + (lane >> 4) * 16;
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < KS; kk += 2) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(a0, a1, a2, a3, kb + tile.at(rt, kcol + kk * 32));
            mma_16816(sa, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
            if (kk + 1 < KS) {
                ldsm_x4(a0, a1, a2, a3, kb + tile.at(rt, kcol + kk * 32 + 32));
                mma_16816(sb, a0, a1, a2, a3, qb[kk + 1][0], qb[kk + 1][1]);
            }
        }
        float x[4];  // token g: heads 2t, 2t+1; token g+8: heads 2t, 2t+1
        float mx[2] = {kNegInf, kNegInf};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int tok = g + 8 * (j >> 1);
            x[j] = tok < nv ? (sa[j] + sb[j]) * scale_log2 : kNegInf;
            mx[j & 1] = fmaxf(mx[j & 1], x[j]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 4));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 8));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 16));
        }
        float alpha[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float mnew = fmaxf(m[h], mx[h]);  // finite: nv >= 1
            alpha[h] = exp2f(m[h] - mnew);
            m[h] = mnew;
        }
        // weights rows = tokens 0-7 / 8-15, columns = heads
        const uint32_t p0 = pack_half2(exp2f(x[0] - m[0]), exp2f(x[1] - m[1]));
        const uint32_t p1 = pack_half2(exp2f(x[2] - m[0]), exp2f(x[3] - m[1]));
        // the normaliser sums the same fp16-rounded weights the MMA applies
        const float2 u0 = unpack_half2(p0), u1 = unpack_half2(p1);
        l[0] = l[0] * alpha[0] + (u0.x + u1.x);
        l[1] = l[1] * alpha[1] + (u0.y + u1.y);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            o[mt][0] *= alpha[0];
            o[mt][1] *= alpha[1];
            o[mt][2] *= alpha[0];
            o[mt][3] *= alpha[1];
        }
        const uint32_t pb0 = movmatrix_trans(p0), pb1 = movmatrix_trans(p1);
        // O^T += V^T P^T; transposed-ldmatrix matrices: tokens 0-7 at dims
        // 0-7 (A row g) and 8-15 (row g+8), then tokens 8-15 at the same
        const int vt = (lane >> 4) * 8 + (lane & 7);
        const uint32_t vcol = head + ((lane >> 3) & 1) * 16;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(a0, a1, a2, a3, vb + tile.at(vt, vcol + mt * 32));
            mma_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
        }
    }

    // Softmax sum of head 2t + h over all tokens (every lane of one t).
    __device__ __forceinline__ float l_total(int h) const {
        float ls = l[h];
        ls += __shfl_xor_sync(0xffffffffu, ls, 4);
        ls += __shfl_xor_sync(0xffffffffu, ls, 8);
        ls += __shfl_xor_sync(0xffffffffu, ls, 16);
        return ls;
    }

    // Shared-memory export for a CTA merge: m[h], l[h], o[h][D] for h < G.
    __device__ __forceinline__ void export_state(float *mw, float *lw, float *ow, int lane) {
        const int g = lane >> 2, t = lane & 3;
        const float l0 = l_total(0), l1 = l_total(1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int hd = 2 * t + h;
            if (hd < G) {
                if (g == 0) {
                    mw[hd] = m[h];
                    lw[hd] = h ? l1 : l0;
                }
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    ow[hd * D + 16 * mt + g] = o[mt][h];
                    ow[hd * D + 16 * mt + g + 8] = o[mt][2 + h];
                }
            }
        }
    }

    // Final fp16 output o / l of heads h < G at out_g0 + h*D (zeros if empty).
    __device__ __forceinline__ void write_output(__half *out_g0, int lane) {
        const int g = lane >> 2, t = lane & 3;
        const float l0 = l_total(0), l1 = l_total(1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int hd = 2 * t + h;
            const float ls = h ? l1 : l0;
            const float inv = ls > 0.f ? 1.f / ls : 0.f;
            if (hd < G) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    out_g0[hd * D + 16 * mt + g] = __float2half_rn(o[mt][h] * inv);
                    out_g0[hd * D + 16 * mt + g + 8] = __float2half_rn(o[mt][2 + h] * inv);
                }
            }
        }
    }

    // Partial state to global memory: ml[h] = (m, l), o[h*D + d] for h < G.
    __device__ __forceinline__ void write_partial(float2 *ml, float *og, int lane) {
        const int g = lane >> 2, t = lane & 3;
        const float l0 = l_total(0), l1 = l_total(1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int hd = 2 * t + h;
            if (hd < G) {
                if (g == 0) ml[hd] = make_float2(m[h], h ? l1 : l0);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    og[hd * D + 16 * mt + g] = o[mt][h];
                    og[hd * D + 16 * mt + g + 8] = o[mt][2 + h];
                }
            }
        }
    }
};

// ---------------------------------------------------------------------------
// MMA policy for several new tokens per sequence (chunked prefill, draft
// verification: "vLLM 技术内幕" §3.2, §7.4) on the same transposed products
// as MmaPolicy.  The 8*NT columns of S^T = K Q^T and O^T = V^T P^T are
// (new token j, query head g of the group) pairs, column c = j*G + g, each
// with its own causal limit: token j of a sequence with L tokens, the last Q
// of them new, sees the keys 0 .. L - Q + j.  One new token (Q = 1) is a
// decode with G columns.

// The query rows one (sequence, kv head) contributes.
struct QueryRows {
    const __half *q;  // q [rows, H, D]
    __half *out;      // out [rows, H, D]
    int64_t row0;     // query row of the sequence's first new token
    int H;            // query heads
    int kvh;          // kv head
    int ncols;        // valid columns: Q * G
    int lim0;         // last key position token 0 sees: L - Q
};

template <int D, int G, int NT>
struct MmaColsPolicy {
    static constexpr bool kColumns = true;
    static constexpr int kRows = 8 * NT;  // partial-state rows (columns) per (sequence, kv head)
    static constexpr bool kZeroTailRows = true;
    static constexpr int KS = D / 16;
    static constexpr int MT = D / 16;
    uint32_t qb[NT][KS][2];  // B operand of S^T: query dims of column 8c + l/4
    // O^T, n-tile c, m-tile mt: c0 / c2 = dims 16mt + g / + g + 8 of column
    // 8c + 2t, c1 / c3 the same of column 8c + 2t + 1
    float o[NT][MT][4];
    float m[NT][2], l[NT][2];  // softmax state of columns 8c + 2t + h
    int lim[NT][2];            // last key position of those columns (-1: no column)

    __device__ __forceinline__ void init(const QueryRows &qr, int lane) {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int c = 0; c < NT; ++c) {
            const int col = 8 * c + g;
            const __half *qrow = nullptr;
            if (col < qr.ncols)
                qrow = qr.q + ((qr.row0 + col / G) * qr.H + qr.kvh * G + col % G) * D;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                if (qrow) {
                    const uint32_t *r = reinterpret_cast<const uint32_t *>(qrow + kk * 16);
                    qb[c][kk][0] = __ldg(r + t);
                    qb[c][kk][1] = __ldg(r + 4 + t);
                } else {
                    qb[c][kk][0] = qb[c][kk][1] = 0u;
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int cc = 8 * c + 2 * t + h;
                lim[c][h] = cc < qr.ncols ? qr.lim0 + cc / G : -1;
                m[c][h] = kNegInf;
                l[c][h] = 0.f;
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
                o[c][mt][0] = o[c][mt][1] = o[c][mt][2] = o[c][mt][3] = 0.f;
        }
    }

    // One staged block whose first key is at position kp: key tile at kb,
    // value tile at vb, this head's bytes from `head`; nv valid tokens.
    __device__ __forceinline__ void block(uint32_t kb, uint32_t vb, SwizzledTile tile,
                                          uint32_t head, int nv, int kp, float scale_log2,
                                          int lane) {
        const int g = lane >> 2;
        const int rt = ((lane >> 3) & 1) * 8 + (lane & 7);
        const uint32_t kcol = head + (lane >> 4) * 16;
        float sa[NT][4], sb[NT][4];
#pragma unroll
        for (int c = 0; c < NT; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e) sa[c][e] = sb[c][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; kk += 2) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(a0, a1, a2, a3, kb + tile.at(rt, kcol + kk * 32));
#pragma unroll
            for (int c = 0; c < NT; ++c) mma_16816(sa[c], a0, a1, a2, a3, qb[c][kk][0], qb[c][kk][1]);
            if (kk + 1 < KS) {
                ldsm_x4(a0, a1, a2, a3, kb + tile.at(rt, kcol + kk * 32 + 32));
#pragma unroll
                for (int c = 0; c < NT; ++c)
                    mma_16816(sb[c], a0, a1, a2, a3, qb[c][kk + 1][0], qb[c][kk + 1][1]);
            }
        }
        // element e: token g + 8*(e>>1), column 8c + 2t + (e&1)
        float x[NT][4];
        float mx[NT][2];
#pragma unroll
        for (int c = 0; c < NT; ++c) {
            mx[c][0] = mx[c][1] = kNegInf;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = g + 8 * (e >> 1);
                const bool vis = tok < nv && kp + tok <= lim[c][e & 1];
                x[c][e] = vis ? (sa[c][e] + sb[c][e]) * scale_log2 : kNegInf;
                mx[c][e & 1] = fmaxf(mx[c][e & 1], x[c][e]);
            }
        }
        float alpha[NT][2], msafe[NT][2];
#pragma unroll
        for (int c = 0; c < NT; ++c)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v = mx[c][h];
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                const float mnew = fmaxf(m[c][h], v);
                // a column with no visible key yet keeps m = -inf, l = 0, o = 0
                msafe[c][h] = mnew == kNegInf ? 0.f : mnew;
                alpha[c][h] = exp2f(m[c][h] - msafe[c][h]);
                m[c][h] = mnew;
            }
        uint32_t pb[NT][2];
#pragma unroll
        for (int c = 0; c < NT; ++c) {
            const uint32_t p0 = pack_half2(exp2f(x[c][0] - msafe[c][0]), exp2f(x[c][1] - msafe[c][1]));
            const uint32_t p1 = pack_half2(exp2f(x[c][2] - msafe[c][0]), exp2f(x[c][3] - msafe[c][1]));
            // the normaliser sums the same fp16-rounded weights the MMA applies
            const float2 u0 = unpack_half2(p0), u1 = unpack_half2(p1);
            l[c][0] = l[c][0] * alpha[c][0] + (u0.x + u1.x);
            l[c][1] = l[c][1] * alpha[c][1] + (u0.y + u1.y);
            pb[c][0] = movmatrix_trans(p0);
            pb[c][1] = movmatrix_trans(p1);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                o[c][mt][0] *= alpha[c][0];
                o[c][mt][1] *= alpha[c][1];
                o[c][mt][2] *= alpha[c][0];
                o[c][mt][3] *= alpha[c][1];
            }
        }
        const int vt = (lane >> 4) * 8 + (lane & 7);
        const uint32_t vcol = head + ((lane >> 3) & 1) * 16;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(a0, a1, a2, a3, vb + tile.at(vt, vcol + mt * 32));
#pragma unroll
            for (int c = 0; c < NT; ++c) mma_16816(o[c][mt], a0, a1, a2, a3, pb[c][0], pb[c][1]);
        }
    }

    __device__ __forceinline__ float l_total(int c, int h) const {
        float ls = l[c][h];
        ls += __shfl_xor_sync(0xffffffffu, ls, 4);
        ls += __shfl_xor_sync(0xffffffffu, ls, 8);
        ls += __shfl_xor_sync(0xffffffffu, ls, 16);
        return ls;
    }

    // Final fp16 output o / l of every valid column.
    __device__ __forceinline__ void write_output(const QueryRows &qr, int lane) {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int c = 0; c < NT; ++c)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float ls = l_total(c, h);
                const int col = 8 * c + 2 * t + h;
                if (col >= qr.ncols) continue;
                const float inv = ls > 0.f ? 1.f / ls : 0.f;
                __half *dst = qr.out + ((qr.row0 + col / G) * qr.H + qr.kvh * G + col % G) * D;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    dst[16 * mt + g] = __float2half_rn(o[c][mt][h] * inv);
                    dst[16 * mt + g + 8] = __float2half_rn(o[c][mt][2 + h] * inv);
                }
            }
    }

    // Partial state to global memory, one row per column: ml[col] = (m, l),
    // o[col*D + d] (columns >= ncols are not written).
    __device__ __forceinline__ void write_partial(float2 *ml, float *og, int ncols, int lane) {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int c = 0; c < NT; ++c)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float ls = l_total(c, h);
                const int col = 8 * c + 2 * t + h;
                if (col >= ncols) continue;
                if (g == 0) ml[col] = make_float2(m[c][h], ls);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    og[col * D + 16 * mt + g] = o[c][mt][h];
                    og[col * D + 16 * mt + g + 8] = o[c][mt][2 + h];
                }
            }
    }
};

// ---------------------------------------------------------------------------
// MMA policy over FP8 (E4M3) staged tiles, fed to the fp16 MMA without a
// shared-memory round trip.  Tokens are tiled 0-7 / 8-15 as in MmaPolicy.
//
// Codes become fp16 through the hardware conversion of an E4M3 pair to an
// f16 pair (exact: every E4M3 value is an fp16 value).  Measured against an
// all-integer conversion (moving the sign and the 7 other bits of each code
// into place, ~3.5 ALU operations a pair) it is the faster: the conversions
// are most of the FP8 consumer's extra work.
//
// Scores are computed transposed, S^T = K Q^T (16 tokens by 8 query-head
// columns per MMA, so no row is wasted on keys): a non-transposed ldmatrix
// gives lane l the 4 codes of dims 4*(l%4)..+3 of the matrix's token l/4
// (per 16-dim, 8-token matrix); the low code pair is A row l/4 at k-slots
// 2*(l%4)+{0,1} and the high pair the same row at k-slots +8, under the
// contraction-index permutation k = 2t+j -> 4t+j, k = 8+2t+j -> 4t+2+j,
// which the query fragments (the B operand, one 64-bit load per k-step)
// follow.  Lane l then holds the scores of tokens l/4 and l/4+8 for heads
// 2*(l%4) and 2*(l%4)+1, and keeps the online-softmax state of those two
// heads (the max over tokens is a butterfly over the lanes of one l%4).
// Values: a transposed ldmatrix gives lane l the codes of k-slots
// 2*(l%4)+{0,1} at dims 2*(l/4)+{0,1}.  They go in as the A operand of
// O^T = V^T P^T (16 head dims by 16 tokens): a byte permute gathers the two
// k-slots of the even dim, which become A row l/4, and those of the odd dim,
// A row l/4 + 8.  The fp16 weights, transposed per 8x8 half by movmatrix,
// are the B operand, one column per query head; O^T's columns are then the
// same two heads whose softmax state the lane keeps.
// The key scale multiplies the score and the value scale the softmax weight
// (each factors out of its sum); the weights also carry an exact factor of
// 256, removed on output, to keep them clear of fp16 subnormals.

// f16x2 of the E4M3 codes in the low 16 bits of x (low code -> low half).
__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint32_t x) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<unsigned short>(x)));
    return r;
}

__device__ __forceinline__ uint32_t byte_perm(uint32_t x, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(0u), "r"(sel));
    return r;
}

template <int D, int G>
struct MmaFp8Policy {
    static constexpr bool kColumns = false;
    static constexpr int kRows = G;
    static constexpr int KS = D / 16;  // k-steps of S^T = K Q^T
    static constexpr int MT = D / 16;  // m-tiles (16 head dims each) of O^T
    static constexpr int kLaneTokens = 2;  // tokens whose scales a lane needs per block
    static constexpr float kWeightBoost = 256.f;  // exact; removed on output
    uint32_t qb[KS][2];  // B operand of S^T: query dims of head l/4
    // O^T, m-tile mt: c0 / c2 = dims 16mt + 2g / +1 of head 2t, c1 / c3 the
    // same dims of head 2t+1 (g = lane/4, t = lane%4)
    float o[MT][4];
    float m[2], l[2];  // online-softmax state of heads 2t, 2t+1 (l: this lane's tokens)

    // Token of this lane's i-th score row (i = 0, 1).
    __device__ __forceinline__ static int token_of(int lane, int i) { return (lane >> 2) + 8 * i; }

    __device__ __forceinline__ void init(const __half *qg, float /*scale_log2*/, int lane) {
        const int g = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            if (g < G) {
                const uint2 w =
                    __ldg(reinterpret_cast<const uint2 *>(qg + g * D + kk * 16 + tig * 4));
                qb[kk][0] = w.x;
                qb[kk][1] = w.y;
            } else {
                qb[kk][0] = qb[kk][1] = 0u;
            }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m[0] = m[1] = kNegInf;
        l[0] = l[1] = 0.f;
    }

    // NB (1 or 2) staged blocks of one sequence in one online-softmax step.
    // kb8 / vb8: the key / value code tiles of each block, this head's codes
    // starting at byte `head` of each row; value rows >= nv must hold finite
    // codes.  ks / vs: the key / value scales of this lane's tokens
    // (token_of) in each block.
    template <int NB>
    __device__ __forceinline__ void step(const uint32_t (&kb8)[NB], const uint32_t (&vb8)[NB],
                                         SwizzledTile tile, uint32_t head, const int (&nv)[NB],
                                         float scale_log2, int lane,
                                         const float (&ks)[NB][kLaneTokens],
                                         const float (&vs)[NB][kLaneTokens]) {
        // matrices 0/1: tokens 0-7 / 8-15, codes 0-15 of a 32-code step;
        // 2/3: the same for codes 16-31
        const int rt = ((lane >> 3) & 1) * 8 + (lane & 7);
        const uint32_t col = head + (lane >> 4) * 16;
        // S^T = K Q^T, two accumulator chains per block
        float x[NB][4];  // token g: heads 2t, 2t+1; token g+8: heads 2t, 2t+1
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kp = 0; kp < D / 32; ++kp) {
                uint32_t r0, r1, r2, r3;  // tokens 0-7 / 8-15, dims 32kp.. / 32kp+16..
                ldsm_x4(r0, r1, r2, r3, kb8[b] + tile.at(rt, col + kp * 32));
                mma_16816(sa, e4m3x2_to_half2(r0), e4m3x2_to_half2(r1),
                          e4m3x2_to_half2(r0 >> 16), e4m3x2_to_half2(r1 >> 16), qb[2 * kp][0],
                          qb[2 * kp][1]);
                mma_16816(sb, e4m3x2_to_half2(r2), e4m3x2_to_half2(r3),
                          e4m3x2_to_half2(r2 >> 16), e4m3x2_to_half2(r3 >> 16),
                          qb[2 * kp + 1][0], qb[2 * kp + 1][1]);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) x[b][j] = sa[j] + sb[j];
        }
        // scale, mask, and the block max of each of the lane's two heads
        float mx[2] = {kNegInf, kNegInf};
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = j >> 1;  // token row: g or g+8
                x[b][j] = token_of(lane, r) < nv[b] ? (x[b][j] * ks[b][r]) * scale_log2 : kNegInf;
                mx[j & 1] = fmaxf(mx[j & 1], x[b][j]);
            }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 4));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 8));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 16));
        }
        float alpha[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float mnew = fmaxf(m[h], mx[h]);  // finite: some token is valid
            alpha[h] = exp2f(m[h] - mnew);
            m[h] = mnew;
            l[h] *= alpha[h];
        }
        uint32_t pb[NB][2];  // B fragments of O^T += V^T P^T
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float pw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = j >> 1;
                const float p = exp2f(x[b][j] - m[j & 1]);
                l[j & 1] += p;
                pw[j] = token_of(lane, r) < nv[b] ? p * (vs[b][r] * kWeightBoost) : 0.f;
            }
            // rows = tokens 0-7 / 8-15, columns = heads; transposed to
            // (token pair, head) B fragments
            pb[b][0] = movmatrix_trans(pack_half2(pw[0], pw[1]));
            pb[b][1] = movmatrix_trans(pack_half2(pw[2], pw[3]));
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            o[mt][0] *= alpha[0];
            o[mt][1] *= alpha[1];
            o[mt][2] *= alpha[0];
            o[mt][3] *= alpha[1];
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t r0, r1, r2, r3;  // k-slots 0-7 / 8-15, dims 32q.. / 32q+16..
                ldsm_x4_trans(r0, r1, r2, r3, vb8[b] + tile.at(rt, col + q * 32));
                // A = V^T: row g <- the even dim (bytes 0, 2), row g+8 <- the odd one
                mma_16816(o[2 * q], e4m3x2_to_half2(byte_perm(r0, 0x20)),
                          e4m3x2_to_half2(byte_perm(r0, 0x31)),
                          e4m3x2_to_half2(byte_perm(r1, 0x20)),
                          e4m3x2_to_half2(byte_perm(r1, 0x31)), pb[b][0], pb[b][1]);
                mma_16816(o[2 * q + 1], e4m3x2_to_half2(byte_perm(r2, 0x20)),
                          e4m3x2_to_half2(byte_perm(r2, 0x31)),
                          e4m3x2_to_half2(byte_perm(r3, 0x20)),
                          e4m3x2_to_half2(byte_perm(r3, 0x31)), pb[b][0], pb[b][1]);
            }
        }
    }

    // Softmax sum of head 2t + h over all tokens (every lane of one t).
    __device__ __forceinline__ float l_total(int h) const {
        float ls = l[h];
        ls += __shfl_xor_sync(0xffffffffu, ls, 4);
        ls += __shfl_xor_sync(0xffffffffu, ls, 8);
        ls += __shfl_xor_sync(0xffffffffu, ls, 16);
        return ls;
    }

    // Final fp16 output o / l of heads h < G at out_g0 + h*D (zeros if empty).
    __device__ __forceinline__ void write_output(__half *out_g0, int lane) {
        const int g = lane >> 2, t = lane & 3;
        const float l0 = l_total(0), l1 = l_total(1);
        const float u = 1.f / kWeightBoost;
        const float i0 = l0 > 0.f ? u / l0 : 0.f, i1 = l1 > 0.f ? u / l1 : 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            if (2 * t < G)
                *reinterpret_cast<__half2 *>(out_g0 + (2 * t) * D + 16 * mt + 2 * g) =
                    __floats2half2_rn(o[mt][0] * i0, o[mt][2] * i0);
            if (2 * t + 1 < G)
                *reinterpret_cast<__half2 *>(out_g0 + (2 * t + 1) * D + 16 * mt + 2 * g) =
                    __floats2half2_rn(o[mt][1] * i1, o[mt][3] * i1);
        }
    }

    // Partial state to global memory: ml[h] = (m, l), o[h*D + d] for h < G.
    __device__ __forceinline__ void write_partial(float2 *ml, float *og, int lane) {
        const int g = lane >> 2, t = lane & 3;
        const float l0 = l_total(0), l1 = l_total(1);
        if (g == 0) {
            if (2 * t < G) ml[2 * t] = make_float2(m[0], l0);
            if (2 * t + 1 < G) ml[2 * t + 1] = make_float2(m[1], l1);
        }
        const float u = 1.f / kWeightBoost;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            if (2 * t < G)
                *reinterpret_cast<float2 *>(og + (2 * t) * D + 16 * mt + 2 * g) =
                    make_float2(o[mt][0] * u, o[mt][2] * u);
            if (2 * t + 1 < G)
                *reinterpret_cast<float2 *>(og + (2 * t + 1) * D + 16 * mt + 2 * g) =
                    make_float2(o[mt][1] * u, o[mt][3] * u);
        }
    }
};

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
    static constexpr bool kColumns = false;
    static constexpr int kRows = G;
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

    __device__ __forceinline__ void block(uint32_t kb, uint32_t vb, SwizzledTile tile,
                                          uint32_t head, int nv, float /*scale*/, int lane,
                                          float *pbuf) {
        const uint32_t lane_off = head + lane * DPL * 2;
        const int idx = lane / R;  // result index held by this lane: token*G + head
        float s[NCH];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            float part[NV];
#pragma unroll
            for (int t = 0; t < TC; ++t) {
                float kx[DPL];
                load_row(kb + tile.at(c * TC + t, lane_off), kx);
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
            load_row(vb + tile.at(t, lane_off), vx);
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

// Zero bytes [head, head + ROW_BYTES) of value rows [nv, 16) of a staged
// tile (one head's slice), then order those generic-proxy writes before
// later bulk copies into the stage.
template <int ROW_BYTES>
__device__ __forceinline__ void zero_tail_bytes(uint32_t vb, SwizzledTile tile, uint32_t head,
                                                int nv, int lane) {
    constexpr int kUnits = ROW_BYTES / 16;
    for (int e = lane; e < (kBS - nv) * kUnits; e += 32) {
        const uint32_t a = vb + tile.at(nv + e / kUnits, head + (e % kUnits) * 16);
        asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(a), "r"(0u) : "memory");
    }
    fence_proxy_async_smem();
    __syncwarp();
}

// Zero value rows [nv, 16) of one head's fp16 slice (D*2 bytes at `head`).
template <int D>
__device__ __forceinline__ void zero_tail_rows(uint32_t vb, SwizzledTile tile, uint32_t head,
                                               int nv, int lane) {
    zero_tail_bytes<D * 2>(vb, tile, head, nv, lane);
}

}  // namespace dec
}  // namespace pkv
