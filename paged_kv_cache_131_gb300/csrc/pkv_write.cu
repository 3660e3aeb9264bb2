// pkv_write.cu -- the paged KV-cache write ("vLLM KV Cache Layout 可视化":
// 查一个 token, kernel 那一侧; "deep-dive-into-vllm-05" §2 prefill / decode
// writes): split each token's slot back into (block, position) and copy its
// row to offset + layer*layer_stride + block*block_stride + position*row_width.
//
// One warp per token row, grid-stride over tokens.  Rows are moved with the
// widest vector (16, 8, 4, 2 or 1 bytes) that every address and stride of
// the call allows, four vectors in flight per lane.  This is a pure byte
// copy bound by HBM bandwidth (and, for small calls, by launch latency).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "../../include/pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

struct WriteParams {
    const uint8_t *k;
    const uint8_t *v;
    const int64_t *slot_mapping;
    uint8_t *k_cache;  // already offset by view.offset + view.layer * view.layer_stride
    uint8_t *v_cache;
    int64_t num_tokens;
    int64_t block_stride;
    int64_t row_width;
    int64_t block_size;
    int64_t num_slots;  // num_blocks * block_size
    ErrorRecord *err;
};

constexpr int kWriteThreads = 256;
constexpr int kUnroll = 4;

template <typename VT>
__device__ __forceinline__ VT load_stream(const VT *p) {
    return __ldg(p);
}

template <typename VT>
__device__ __forceinline__ void copy_row(uint8_t *dst_bytes, const uint8_t *src_bytes,
                                         int64_t nvec, int lane) {
    VT *dst = reinterpret_cast<VT *>(dst_bytes);
    const VT *src = reinterpret_cast<const VT *>(src_bytes);
    for (int64_t base = 0; base < nvec; base += 32 * kUnroll) {
        VT r[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = base + u * 32 + lane;
            if (i < nvec) r[u] = load_stream(src + i);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = base + u * 32 + lane;
            if (i < nvec) dst[i] = r[u];
        }
    }
}

template <typename VT>
__global__ void __launch_bounds__(kWriteThreads) cache_write_kernel(const WriteParams p) {
    // a dependent launch (the decode kernel) may be scheduled now; it still
    // waits for this grid's completion before it reads anything
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t nvec = p.row_width / static_cast<int64_t>(sizeof(VT));
    for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         t < p.num_tokens; t += nwarps) {
        const int64_t slot = __ldg(p.slot_mapping + t);
        if (slot < 0) continue;  // padding
        if (slot >= p.num_slots) {
            if (lane == 0) record_error(p.err, PKV_DEVERR_SLOT, t);
            continue;
        }
        const int64_t block = slot / p.block_size;
        const int64_t pos = slot - block * p.block_size;
        const int64_t dst = block * p.block_stride + pos * p.row_width;
        const int64_t src = t * p.row_width;
        copy_row<VT>(p.k_cache + dst, p.k + src, nvec, lane);
        if (p.v != nullptr) copy_row<VT>(p.v_cache + dst, p.v + src, nvec, lane);
    }
}

template <typename VT>
int launch_write(const WriteParams &p, cudaStream_t stream) {
    const int64_t warps_per_cta = kWriteThreads / 32;
    const int64_t want = (p.num_tokens + warps_per_cta - 1) / warps_per_cta;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min(want, cap)));
    cache_write_kernel<VT><<<grid, kWriteThreads, 0, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_failure(e, "cache_write_kernel launch");
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_cache_write(const void *k, const void *v, const int64_t *slot_mapping,
                               int64_t num_tokens, void *k_cache, void *v_cache, pkv_view view,
                               int32_t block_size, int64_t num_blocks, pkv_stream_t stream) {
    using namespace pkv;
    if (num_tokens < 0) return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;  // nothing to do; pointers may be NULL
    if (k == nullptr || slot_mapping == nullptr || k_cache == nullptr) return PKV_ERR_NULL;
    if ((v == nullptr) != (v_cache == nullptr)) return PKV_ERR_NULL;
    if (block_size <= 0 || num_blocks <= 0 || view.row_width <= 0 || view.block_stride <= 0 ||
        view.offset < 0 || view.layer < 0 || view.layer_stride < 0)
        return PKV_ERR_INVALID;
    if (num_blocks > INT64_MAX / block_size) return PKV_ERR_INVALID;
    if (view.layer > 0 && view.layer_stride > (INT64_MAX - view.offset) / view.layer)
        return PKV_ERR_INVALID;
    if (!aligned(slot_mapping, alignof(int64_t))) return PKV_ERR_ALIGNMENT;

    const int64_t base = view.offset + static_cast<int64_t>(view.layer) * view.layer_stride;
    WriteParams p;
    p.k = static_cast<const uint8_t *>(k);
    p.v = static_cast<const uint8_t *>(v);
    p.slot_mapping = slot_mapping;
    p.k_cache = static_cast<uint8_t *>(k_cache) + base;
    p.v_cache = v_cache ? static_cast<uint8_t *>(v_cache) + base : nullptr;
    p.num_tokens = num_tokens;
    p.block_stride = view.block_stride;
    p.row_width = view.row_width;
    p.block_size = block_size;
    p.num_slots = num_blocks * block_size;
    p.err = device_error_record();
    if (p.err == nullptr) return PKV_ERR_CUDA;

    // widest vector every address of the call is a multiple of
    uintptr_t bits = reinterpret_cast<uintptr_t>(p.k) | reinterpret_cast<uintptr_t>(p.k_cache) |
                     static_cast<uintptr_t>(view.block_stride) |
                     static_cast<uintptr_t>(view.row_width);
    if (p.v) bits |= reinterpret_cast<uintptr_t>(p.v) | reinterpret_cast<uintptr_t>(p.v_cache);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((bits & 15) == 0) return launch_write<uint4>(p, s);
    if ((bits & 7) == 0) return launch_write<uint2>(p, s);
    if ((bits & 3) == 0) return launch_write<unsigned int>(p, s);
    if ((bits & 1) == 0) return launch_write<unsigned short>(p, s);
    return launch_write<unsigned char>(p, s);
}
