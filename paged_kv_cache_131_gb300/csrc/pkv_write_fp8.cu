// pkv_write_fp8.cu -- quantize-on-write into an FP8 (E4M3) KV cache
// ("deep-dive-into-vllm-05" §3.4: the KV is stored at low precision when it
// is written, with its scale kept alongside, still managed per block).
//
// Each (token, KV head) row of head_dim fp16 values becomes head_dim E4M3
// codes and one fp32 scale, all computed in fp32: amax = max |x|,
// s = amax / 448 (448 is E4M3's largest finite value), code = RNE(x / s)
// saturated to +-448; s == 0 gives zero codes.  One warp per row (token,
// cache, KV head), grid-stride, so the rows of a token quantize in parallel;
// head_dim/32 values per lane; amax by a warp max-reduction.
// For the token-major cache [num_blocks, block_size, Hk, D] a slot is also
// the row index: row (slot, h) sits at (slot*Hk + h)*D.
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "../../include/pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;

struct Fp8WriteParams {
    const __half *src[2];  // k, v rows [T, Hk, D] (v may be null)
    uint8_t *cache[2];     // [NB, bs, Hk, D] codes
    float *scale[2];       // [NB, bs, Hk]
    const int64_t *slot_mapping;
    int64_t num_tokens;
    int64_t num_slots;
    int32_t num_kv_heads;
    int32_t num_caches;
    ErrorRecord *err;
};

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Quantize one row of D fp16 values (whole warp); lane owns D/32 of them.
template <int D>
__device__ __forceinline__ void quantize_row(const __half *x, uint8_t *codes, float *scale,
                                             int lane) {
    constexpr int PL = D / 32;
    float v[PL];
    if constexpr (PL == 4) {
        const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(x) + lane);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
        v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    } else {
        const unsigned int raw = __ldg(reinterpret_cast<const unsigned int *>(x) + lane);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&raw));
        v[0] = a.x; v[1] = a.y;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < PL; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax / 448.f;  // IEEE division (no fast-math in this build)
    float y[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) y[i] = s == 0.f ? 0.f : v[i] / s;
    if constexpr (PL == 4) {
        const uint32_t w = e4m3x2(y[0], y[1]) | (e4m3x2(y[2], y[3]) << 16);
        reinterpret_cast<uint32_t *>(codes)[lane] = w;
    } else {
        reinterpret_cast<uint16_t *>(codes)[lane] = static_cast<uint16_t>(e4m3x2(y[0], y[1]));
    }
    if (lane == 0) *scale = s;
}

template <int D>
__global__ void __launch_bounds__(kThreads)
    cache_write_fp8_kernel(const __grid_constant__ Fp8WriteParams p) {
    grid_launch_dependents();  // a following decode may launch; it waits for us
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int Hk = p.num_kv_heads;
    const int64_t rows_per_token = static_cast<int64_t>(p.num_caches) * Hk;
    const int64_t nrows = p.num_tokens * rows_per_token;
    for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         r < nrows; r += nwarps) {
        const int64_t t = r / rows_per_token;
        const int c = static_cast<int>((r - t * rows_per_token) / Hk);
        const int h = static_cast<int>(r - t * rows_per_token - static_cast<int64_t>(c) * Hk);
        const int64_t slot = __ldg(p.slot_mapping + t);
        if (slot < 0) continue;  // padding
        if (slot >= p.num_slots) {
            if (lane == 0 && c == 0 && h == 0) record_error(p.err, PKV_DEVERR_SLOT, t);
            continue;
        }
        quantize_row<D>(p.src[c] + (t * Hk + h) * D, p.cache[c] + (slot * Hk + h) * D,
                        p.scale[c] + slot * Hk + h, lane);
    }
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_cache_write_fp8(const void *k, const void *v, const int64_t *slot_mapping,
                                   int64_t num_tokens, void *k_cache, void *v_cache,
                                   float *k_scale, float *v_scale, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                   pkv_stream_t stream) {
    using namespace pkv;
    if (num_tokens < 0) return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !k_cache || !k_scale || !slot_mapping) return PKV_ERR_NULL;
    if ((v == nullptr) != (v_cache == nullptr) || (v == nullptr) != (v_scale == nullptr))
        return PKV_ERR_NULL;
    if (num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0 ||
        num_blocks > INT64_MAX / block_size || num_tokens > INT64_MAX / (2 * num_kv_heads))
        return PKV_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    const uintptr_t need = head_dim == 128 ? 8 : 4;  // fp16 source vector
    if (!aligned(k, need) || (v && !aligned(v, need)) || !aligned(k_cache, 4) ||
        (v_cache && !aligned(v_cache, 4)) || !aligned(k_scale, 4) ||
        (v_scale && !aligned(v_scale, 4)) || !aligned(slot_mapping, 8))
        return PKV_ERR_ALIGNMENT;
    Fp8WriteParams p{};
    p.src[0] = static_cast<const __half *>(k);
    p.cache[0] = static_cast<uint8_t *>(k_cache);
    p.scale[0] = k_scale;
    p.num_caches = 1;
    if (v) {
        p.src[1] = static_cast<const __half *>(v);
        p.cache[1] = static_cast<uint8_t *>(v_cache);
        p.scale[1] = v_scale;
        p.num_caches = 2;
    }
    p.slot_mapping = slot_mapping;
    p.num_tokens = num_tokens;
    p.num_slots = num_blocks * block_size;
    p.num_kv_heads = num_kv_heads;
    p.err = device_error_record();
    if (p.err == nullptr) return PKV_ERR_CUDA;
    const int64_t rows = num_tokens * p.num_caches * num_kv_heads;
    const int64_t want = (rows + kThreads / 32 - 1) / (kThreads / 32);
    const int grid = static_cast<int>(
        std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(sm_count()) * 16)));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (head_dim == 128)
        cache_write_fp8_kernel<128><<<grid, kThreads, 0, s>>>(p);
    else
        cache_write_fp8_kernel<64><<<grid, kThreads, 0, s>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_failure(e, "cache_write_fp8_kernel launch");
}
