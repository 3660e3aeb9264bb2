// pkv_blocks.cu -- whole-block copies for copy on write ("vLLM 技术内幕" §2.2:
// a sequence about to write into a block other sequences still reference
// (ref_cnt > 1) gets a new physical block holding a copy of the old one).
//
// For each (src, dst) pair and each layer of the view, the block's page
// (block_size * row_width bytes at offset + layer*layer_stride +
// block*block_stride) is copied from src to dst.  One CTA per (pair, layer)
// unit, grid-stride; 16-byte vectors when every address and stride allows,
// else 8, 4, 2 or 1 bytes.  Bound by HBM bandwidth (2 x page bytes per unit).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "../../include/pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;

struct CopyParams {
    uint8_t *base;  // cache + view.offset + view.layer * view.layer_stride
    int64_t layer_stride;
    int64_t block_stride;
    int64_t page_bytes;
    int32_t num_layers;
    int32_t vec;
    const int64_t *mapping;  // [num_pairs][2]
    int64_t num_pairs;
    int64_t num_blocks;
    ErrorRecord *err;
};

template <typename VT>
__device__ __forceinline__ void copy_page(uint8_t *dst, const uint8_t *src, int64_t nvec) {
    VT *d = reinterpret_cast<VT *>(dst);
    const VT *s = reinterpret_cast<const VT *>(src);
    for (int64_t i = threadIdx.x; i < nvec; i += blockDim.x * 4) {
        VT r[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (i + u * blockDim.x < nvec) r[u] = s[i + u * blockDim.x];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (i + u * blockDim.x < nvec) d[i + u * blockDim.x] = r[u];
    }
}

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const CopyParams p) {
    const int64_t units = p.num_pairs * p.num_layers;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int64_t pair = u / p.num_layers;
        const int64_t layer = u - pair * p.num_layers;
        const int64_t src = p.mapping[2 * pair], dst = p.mapping[2 * pair + 1];
        if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
            if (threadIdx.x == 0 && layer == 0) record_error(p.err, PKV_DEVERR_BLOCK_ID, pair);
            continue;
        }
        if (src == dst) continue;
        const uint8_t *s = p.base + layer * p.layer_stride + src * p.block_stride;
        uint8_t *d = p.base + layer * p.layer_stride + dst * p.block_stride;
        const int64_t nvec = p.page_bytes / p.vec;
        switch (p.vec) {
            case 16: copy_page<uint4>(d, s, nvec); break;
            case 8: copy_page<uint2>(d, s, nvec); break;
            case 4: copy_page<unsigned int>(d, s, nvec); break;
            case 2: copy_page<unsigned short>(d, s, nvec); break;
            default: copy_page<unsigned char>(d, s, nvec); break;
        }
    }
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_copy_blocks(void *cache, pkv_view view, int32_t num_layers,
                               int32_t block_size, const int64_t *block_mapping,
                               int64_t num_pairs, int64_t num_blocks, pkv_stream_t stream) {
    using namespace pkv;
    if (num_pairs < 0 || num_layers < 0) return PKV_ERR_INVALID;
    if (num_pairs == 0 || num_layers == 0) return PKV_OK;
    if (cache == nullptr || block_mapping == nullptr) return PKV_ERR_NULL;
    if (block_size <= 0 || num_blocks <= 0 || view.row_width <= 0 || view.block_stride <= 0 ||
        view.offset < 0 || view.layer < 0 || view.layer_stride < 0)
        return PKV_ERR_INVALID;
    if (num_layers > 1 && view.layer_stride <= 0) return PKV_ERR_INVALID;
    if (!aligned(block_mapping, alignof(int64_t))) return PKV_ERR_ALIGNMENT;
    CopyParams p{};
    p.base = static_cast<uint8_t *>(cache) + view.offset +
             static_cast<int64_t>(view.layer) * view.layer_stride;
    p.layer_stride = view.layer_stride;
    p.block_stride = view.block_stride;
    p.page_bytes = static_cast<int64_t>(block_size) * view.row_width;
    p.num_layers = num_layers;
    const uintptr_t bits = reinterpret_cast<uintptr_t>(p.base) |
                           static_cast<uintptr_t>(view.layer_stride) |
                           static_cast<uintptr_t>(view.block_stride) |
                           static_cast<uintptr_t>(p.page_bytes);
    p.vec = (bits & 15) == 0 ? 16 : (bits & 7) == 0 ? 8 : (bits & 3) == 0 ? 4
          : (bits & 1) == 0 ? 2 : 1;
    p.mapping = block_mapping;
    p.num_pairs = num_pairs;
    p.num_blocks = num_blocks;
    p.err = device_error_record();
    if (p.err == nullptr) return PKV_ERR_CUDA;
    const int64_t units = num_pairs * num_layers;
    const int grid = static_cast<int>(std::min<int64_t>(units, static_cast<int64_t>(sm_count()) * 8));
    copy_blocks_kernel<<<grid, kCopyThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_failure(e, "copy_blocks_kernel launch");
}
