// pkv_tensor_map.cu -- tensor maps (TMA descriptors) over the token-major KV
// caches, for the decode kernels' one-copy-per-tile staging.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

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

}  // namespace

int make_kv_tensor_map(CUtensorMap *map, const void *cache, int64_t num_blocks, int row_bytes,
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

}  // namespace dec
}  // namespace pkv
