// pkv_tensor_map.cu -- tensor maps (TMA descriptors) over the token-major KV
// caches, for the kernels' one-copy-per-tile staging, and over the query rows
// of the chunk kernel.
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
    int kind;  // 0: KV cache, 1: query rows
    const void *ptr;
    int64_t a;  // blocks (KV) or tokens (query)
    int b, c, d;  // row bytes, box chunks (KV); heads, head dim, group (query)
    CUtensorMap map;
};
constexpr int kMapCache = 32;
MapEntry g_maps[kMapCache];
int g_maps_used = 0, g_maps_next = 0;
std::mutex g_maps_mutex;

int encode(CUtensorMap *map, const void *cache, int64_t num_blocks, int row_bytes,
           int box_chunks);
int encode_q(CUtensorMap *map, const void *q, int64_t num_tokens, int num_heads, int head_dim,
             int group);

// A cached map for this key, or a fresh one from `make` (then cached).
template <typename Make>
int cached_map(CUtensorMap *map, int kind, const void *ptr, int64_t a, int b, int c, int d,
               Make make) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_failure(cudaGetLastError(), "cudaGetDevice");
    {
        std::lock_guard<std::mutex> lock(g_maps_mutex);
        for (int i = 0; i < g_maps_used; ++i) {
            const MapEntry &e = g_maps[i];
            if (e.device == dev && e.kind == kind && e.ptr == ptr && e.a == a && e.b == b &&
                e.c == c && e.d == d) {
                *map = e.map;
                return PKV_OK;
            }
        }
    }
    const int st = make();
    if (st != PKV_OK) return st;
    std::lock_guard<std::mutex> lock(g_maps_mutex);
    MapEntry &e = g_maps[g_maps_next];
    e = MapEntry{dev, kind, ptr, a, b, c, d, *map};
    g_maps_next = (g_maps_next + 1) % kMapCache;
    if (g_maps_used < kMapCache) ++g_maps_used;
    return PKV_OK;
}

}  // namespace

int make_kv_tensor_map(CUtensorMap *map, const void *cache, int64_t num_blocks, int row_bytes,
                       int box_chunks) {
    return cached_map(map, 0, cache, num_blocks, row_bytes, box_chunks, 0, [&] {
        return encode(map, cache, num_blocks, row_bytes, box_chunks);
    });
}

int make_q_tensor_map(CUtensorMap *map, const void *q, int64_t num_tokens, int num_heads,
                      int head_dim, int group) {
    return cached_map(map, 1, q, num_tokens, num_heads, head_dim, group, [&] {
        return encode_q(map, q, num_tokens, num_heads, head_dim, group);
    });
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

int encode_q(CUtensorMap *map, const void *q, int64_t num_tokens, int num_heads, int head_dim,
             int group) {
    if (num_tokens <= 0 || num_tokens > INT32_MAX || num_heads <= 0 || group <= 0 ||
        group > 8 || num_heads % group != 0 || (head_dim != 64 && head_dim != 128))
        return PKV_ERR_UNSUPPORTED;
    const EncodeTiled enc = encoder();
    if (enc == nullptr) {
        set_last_error("cuTensorMapEncodeTiled is not available from the driver");
        return PKV_ERR_CUDA;
    }
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim) * 2,
                                static_cast<cuuint64_t>(num_heads),
                                static_cast<cuuint64_t>(num_tokens)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                   static_cast<cuuint64_t>(num_heads) * head_dim * 2};
    const cuuint32_t box[3] = {128u, static_cast<cuuint32_t>(group),
                               static_cast<cuuint32_t>(128 / group)};
    const cuuint32_t elem_strides[3] = {1u, 1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(q), dims,
                           strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[128];
        std::snprintf(msg, sizeof(msg), "cuTensorMapEncodeTiled (query rows) failed (CUresult %d)",
                      static_cast<int>(r));
        set_last_error(msg);
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

}  // namespace
}  // namespace dec
}  // namespace pkv
