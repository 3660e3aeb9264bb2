// pkv_tensor_map.cu -- tensor maps (TMA descriptors) over the token-major KV
// caches, for the decode kernels' one-copy-per-tile staging.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/pagedkv.h"
#include "pkv_decode_host.h"
#include "pkv_internal.h"

namespace pkv {
namespace dec {
namespace {

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's encoder, found once through the runtime (no link-time
// dependency on the driver library).
EncodeTiled encoder() {
    static const EncodeTiled fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiled>(nullptr);
        return reinterpret_cast<EncodeTiled>(f);
    }();
    return fn;
}

// Recently encoded maps (a map only encodes an address and sizes, so a hit
// is exact whatever happened to the memory in between).
struct MapEntry {
    int device;
    const void *cache;
    int64_t num_blocks;
    int row_bytes;
    int box_chunks;
    CUtensorMap map;
};
constexpr int kMapCache = 32;
MapEntry g_maps[kMapCache];
int g_maps_used = 0, g_maps_next = 0;
std::mutex g_maps_mutex;

int encode(CUtensorMap *map, const void *cache, int64_t num_blocks, int row_bytes,
           int box_chunks);

}  // namespace

int make_kv_tensor_map(CUtensorMap *map, const void *cache, int64_t num_blocks, int row_bytes,
                       int box_chunks) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_failure(cudaGetLastError(), "cudaGetDevice");
    {
        std::lock_guard<std::mutex> lock(g_maps_mutex);
        for (int i = 0; i < g_maps_used; ++i) {
            const MapEntry &e = g_maps[i];
            if (e.device == dev && e.cache == cache && e.num_blocks == num_blocks &&
                e.row_bytes == row_bytes && e.box_chunks == box_chunks) {
                *map = e.map;
                return PKV_OK;
            }
        }
    }
    const int st = encode(map, cache, num_blocks, row_bytes, box_chunks);
    if (st != PKV_OK) return st;
    std::lock_guard<std::mutex> lock(g_maps_mutex);
    MapEntry &e = g_maps[g_maps_next];
    e = MapEntry{dev, cache, num_blocks, row_bytes, box_chunks, *map};
    g_maps_next = (g_maps_next + 1) % kMapCache;
    if (g_maps_used < kMapCache) ++g_maps_used;
    return PKV_OK;
}

namespace {

int encode(CUtensorMap *map, const void *cache, int64_t num_blocks, int row_bytes,
           int box_chunks) {
    const int C = chunk_bytes_for_row(row_bytes);
    const int64_t rows = num_blocks * 16;
    // (tile coordinates are signed 32-bit: every row index must fit)
    if (row_bytes <= 0 || row_bytes % 64 != 0 || num_blocks <= 0 || rows > INT32_MAX ||
        box_chunks < 1 || box_chunks > 256 || box_chunks > row_bytes / C)
        return PKV_ERR_UNSUPPORTED;
    const EncodeTiled enc = encoder();
    if (enc == nullptr) {
        set_last_error("cuTensorMapEncodeTiled is not available from the driver");
        return PKV_ERR_CUDA;
    }
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(row_bytes / C)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes),
                                   static_cast<cuuint64_t>(C)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(C), 16u,
                               static_cast<cuuint32_t>(box_chunks)};
    const cuuint32_t elem_strides[3] = {1u, 1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(cache), dims,
                           strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           C == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[128];
        std::snprintf(msg, sizeof(msg), "cuTensorMapEncodeTiled failed (CUresult %d)",
                      static_cast<int>(r));
        set_last_error(msg);
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

}  // namespace
}  // namespace dec
}  // namespace pkv
