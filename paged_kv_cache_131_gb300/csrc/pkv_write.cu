// pkv_write.cu -- the paged KV-cache write ("vLLM KV Cache Layout 可视化":
// 查一个 token, kernel 那一侧; "deep-dive-into-vllm-05" §2 prefill / decode
// writes): split each token's slot back into (block, position) and copy its
// row to offset + layer*layer_stride + block*block_stride + position*row_width.
//
// One launch serves a list of write descriptors that share one slot_mapping
// (K and V of a layer, or every (cache, layer) view of a multi-cache layout
// such as the two-cache MLA + indexer example of "两种 cache 共用一张 block
// table").  One warp per token, grid-stride over tokens: the warp splits the
// slot once and copies the token's row for every descriptor, each with the
// widest vector (16, 8, 4, 2 or 1 bytes) its addresses and strides allow (a
// kernel instance per width when all descriptors share one, else one that
// switches per descriptor).
// This is a byte copy bound by HBM bandwidth, or by latency for small calls.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "../../include/pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kWriteThreads = 256;
constexpr int kUnroll = 4;
constexpr int kMaxDescs = PKV_MAX_WRITE_DESCS;

struct Desc {
    const uint8_t *src;  // num_tokens rows of row_width bytes
    uint8_t *dst;        // cache + view.offset + view.layer * view.layer_stride
    int64_t block_stride;
    int64_t row_width;
    int32_t vec;         // bytes per vector: 16, 8, 4, 2 or 1
};

struct WriteParams {
    Desc d[kMaxDescs];
    int32_t num_descs;
    const int64_t *slot_mapping;
    int64_t num_tokens;
    int64_t block_size;
    int64_t num_slots;  // num_blocks * block_size
    ErrorRecord *err;
};

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
            if (i < nvec) r[u] = __ldg(src + i);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = base + u * 32 + lane;
            if (i < nvec) dst[i] = r[u];
        }
    }
}

__device__ __forceinline__ void copy_any(uint8_t *dst, const uint8_t *src, int64_t nvec, int vec,
                                         int lane) {
    switch (vec) {
        case 16: copy_row<uint4>(dst, src, nvec, lane); break;
        case 8: copy_row<uint2>(dst, src, nvec, lane); break;
        case 4: copy_row<unsigned int>(dst, src, nvec, lane); break;
        case 2: copy_row<unsigned short>(dst, src, nvec, lane); break;
        default: copy_row<unsigned char>(dst, src, nvec, lane); break;
    }
}

// VEC > 0: every descriptor moves VEC-byte vectors; VEC == 0: each its own.
template <int VEC>
struct VecType;
template <> struct VecType<16> { using T = uint4; };
template <> struct VecType<8> { using T = uint2; };
template <> struct VecType<4> { using T = unsigned int; };
template <> struct VecType<2> { using T = unsigned short; };
template <> struct VecType<1> { using T = unsigned char; };

template <int VEC>
__device__ __forceinline__ void copy_desc(uint8_t *dst, const uint8_t *src, const Desc &d,
                                          int lane) {
    if constexpr (VEC == 0) {
        copy_any(dst, src, d.row_width / d.vec, d.vec, lane);
    } else {
        copy_row<typename VecType<VEC>::T>(dst, src, d.row_width / VEC, lane);
    }
}

template <int VEC>
__global__ void __launch_bounds__(kWriteThreads, VEC == 0 ? 4 : 1)
    cache_write_kernel(const __grid_constant__ WriteParams p) {
    // a dependent launch (the decode kernel) may be scheduled now; it still
    // waits for this grid's completion before it reads the caches
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
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
        if (p.num_descs > 1) {
            // warm L2 with every source row of this token first (one 128-byte
            // line per lane and prefetch, no registers held), so the row copies
            // below wait on L2 rather than on DRAM one descriptor after another
            for (int k = 0; k < p.num_descs; ++k) {
                const uint8_t *src = p.d[k].src + t * p.d[k].row_width;
                for (int64_t off = lane * 128; off < p.d[k].row_width; off += 32 * 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(src + off));
            }
        }
        for (int k = 0; k < p.num_descs; ++k) {
            const Desc &d = p.d[k];
            copy_desc<VEC>(d.dst + block * d.block_stride + pos * d.row_width,
                           d.src + t * d.row_width, d, lane);
        }
    }
}

bool view_ok(const pkv_view &v) {
    if (v.row_width <= 0 || v.block_stride <= 0 || v.offset < 0 || v.layer < 0 ||
        v.layer_stride < 0)
        return false;
    return !(v.layer > 0 && v.layer_stride > (INT64_MAX - v.offset) / v.layer);
}

// One descriptor; its vector is the widest size that every address and
// stride of the descriptor is a multiple of.
Desc make_desc(const void *src, void *cache, const pkv_view &v) {
    Desc d;
    d.src = static_cast<const uint8_t *>(src);
    d.dst = static_cast<uint8_t *>(cache) + v.offset +
            static_cast<int64_t>(v.layer) * v.layer_stride;
    d.block_stride = v.block_stride;
    d.row_width = v.row_width;
    const uintptr_t bits = reinterpret_cast<uintptr_t>(d.src) |
                           reinterpret_cast<uintptr_t>(d.dst) |
                           static_cast<uintptr_t>(v.block_stride) |
                           static_cast<uintptr_t>(v.row_width);
    d.vec = (bits & 15) == 0 ? 16 : (bits & 7) == 0 ? 8 : (bits & 3) == 0 ? 4
          : (bits & 1) == 0 ? 2 : 1;
    return d;
}

int launch_write(WriteParams &p, cudaStream_t stream) {
    const int64_t warps_per_cta = kWriteThreads / 32;
    const int64_t want = (p.num_tokens + warps_per_cta - 1) / warps_per_cta;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min(want, cap)));
    p.err = device_error_record();
    if (p.err == nullptr) return PKV_ERR_CUDA;
    int common = p.d[0].vec;
    for (int k = 1; k < p.num_descs; ++k)
        if (p.d[k].vec != common) common = 0;
    switch (common) {
        case 16: cache_write_kernel<16><<<grid, kWriteThreads, 0, stream>>>(p); break;
        case 8: cache_write_kernel<8><<<grid, kWriteThreads, 0, stream>>>(p); break;
        case 4: cache_write_kernel<4><<<grid, kWriteThreads, 0, stream>>>(p); break;
        case 2: cache_write_kernel<2><<<grid, kWriteThreads, 0, stream>>>(p); break;
        case 1: cache_write_kernel<1><<<grid, kWriteThreads, 0, stream>>>(p); break;
        default: cache_write_kernel<0><<<grid, kWriteThreads, 0, stream>>>(p); break;
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_failure(e, "cache_write_kernel launch");
}

int check_common(const int64_t *slot_mapping, int32_t block_size, int64_t num_blocks) {
    if (slot_mapping == nullptr) return PKV_ERR_NULL;
    if (block_size <= 0 || num_blocks <= 0 || num_blocks > INT64_MAX / block_size)
        return PKV_ERR_INVALID;
    if (!aligned(slot_mapping, alignof(int64_t))) return PKV_ERR_ALIGNMENT;
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_cache_write(const void *k, const void *v, const int64_t *slot_mapping,
                               int64_t num_tokens, void *k_cache, void *v_cache, pkv_view view,
                               int32_t block_size, int64_t num_blocks, pkv_stream_t stream) {
    using namespace pkv;
    if (num_tokens < 0) return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;  // nothing to do; pointers may be NULL
    if (k == nullptr || k_cache == nullptr) return PKV_ERR_NULL;
    if ((v == nullptr) != (v_cache == nullptr)) return PKV_ERR_NULL;
    const int st = check_common(slot_mapping, block_size, num_blocks);
    if (st != PKV_OK) return st;
    if (!view_ok(view)) return PKV_ERR_INVALID;
    WriteParams p{};
    p.d[0] = make_desc(k, k_cache, view);
    p.num_descs = 1;
    if (v != nullptr) p.d[p.num_descs++] = make_desc(v, v_cache, view);
    p.slot_mapping = slot_mapping;
    p.num_tokens = num_tokens;
    p.block_size = block_size;
    p.num_slots = num_blocks * block_size;
    return launch_write(p, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int pkv_cache_write_multi(const pkv_write_desc *descs, int32_t num_descs,
                                     const int64_t *slot_mapping, int64_t num_tokens,
                                     int32_t block_size, int64_t num_blocks,
                                     pkv_stream_t stream) {
    using namespace pkv;
    if (num_tokens < 0 || num_descs < 0 || num_descs > kMaxDescs) return PKV_ERR_INVALID;
    if (num_tokens == 0 || num_descs == 0) return PKV_OK;
    if (descs == nullptr) return PKV_ERR_NULL;
    const int st = check_common(slot_mapping, block_size, num_blocks);
    if (st != PKV_OK) return st;
    WriteParams p{};
    for (int i = 0; i < num_descs; ++i) {
        if (descs[i].src == nullptr || descs[i].cache == nullptr) return PKV_ERR_NULL;
        if (!view_ok(descs[i].view)) return PKV_ERR_INVALID;
        p.d[i] = make_desc(descs[i].src, descs[i].cache, descs[i].view);
    }
    p.num_descs = num_descs;
    p.slot_mapping = slot_mapping;
    p.num_tokens = num_tokens;
    p.block_size = block_size;
    p.num_slots = num_blocks * block_size;
    return launch_write(p, reinterpret_cast<cudaStream_t>(stream));
}
