// pkv_write.cu -- the paged KV-cache write ("vLLM KV Cache Layout 可视化":
// 查一个 token, kernel 那一侧; "deep-dive-into-vllm-05" §2 prefill / decode
// writes): split each token's slot back into (block, position) and copy its
// row to offset + layer*layer_stride + block*block_stride + position*row_width.
//
// One launch serves a list of write descriptors that share one slot_mapping
// (K and V of a layer, or every (cache, layer) view of a multi-cache layout
// such as the two-cache MLA + indexer example of "两种 cache 共用一张 block
// table").  The work is cut into items: for one descriptor, a batch of
// consecutive tokens whose source rows -- contiguous in the source -- fill
// about 16 KB.  A CTA takes an item, issues the loads of the whole batch at
// once (perfectly coalesced, every thread a few vectors of the widest size
// the descriptor's addresses and strides allow), meanwhile splits the
// batch's slots into destination offsets in shared memory, then stores each
// vector at its token's destination row.  Every load of a batch is in
// flight together, so the copy is not one round trip per row; the CTAs are
// small (8 KB of shared memory) and fit beside the decode kernel that may
// start early on the same SMs (see below).
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>

#include "../../include/pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kWriteThreads = 256;
constexpr int kVecsPerThread = 4;
constexpr int kBatchVecs = kWriteThreads * kVecsPerThread;  // vectors of one item
constexpr int kMaxDescs = PKV_MAX_WRITE_DESCS;
constexpr int64_t kMaxRowWidth = int64_t(1) << 30;  // byte offsets in a batch stay 32-bit

struct Desc {
    const uint8_t *src;  // num_tokens rows of row_width bytes
    uint8_t *dst;        // cache + view.offset + view.layer * view.layer_stride
    int64_t block_stride;
    int64_t item0;       // first item of this descriptor
    int32_t row_width;
    int32_t vec;           // bytes per vector: 16, 8, 4, 2 or 1
    int32_t batch_tokens;  // tokens per item
};

struct WriteParams {
    Desc d[kMaxDescs];
    int32_t num_descs;
    const int64_t *slot_mapping;
    int64_t num_tokens;
    int64_t block_size;
    int64_t num_slots;  // num_blocks * block_size
    int64_t num_items;
    ErrorRecord *err;
};

// One item: tokens t0 .. t0+n-1 of descriptor d (k: its index).  The batch's
// source bytes are loaded as VT vectors (a row is a whole number of them, so
// no vector straddles two rows), its slots are split into destination byte
// offsets (-1: skipped) in dst_off, and each vector is stored at its row.
template <typename VT>
__device__ __forceinline__ void write_item(const WriteParams &p, const Desc &d, int k, int64_t t0,
                                           int n, int64_t *dst_off) {
    constexpr int V = sizeof(VT);
    const int64_t R = d.row_width;
    const int64_t nvec = static_cast<int64_t>(n) * R / V;
    const VT *src = reinterpret_cast<const VT *>(d.src + t0 * R);
    for (int64_t base = 0; base < nvec; base += kBatchVecs) {
        VT r[kVecsPerThread];
#pragma unroll
        for (int u = 0; u < kVecsPerThread; ++u) {
            const int64_t i = base + u * kWriteThreads + threadIdx.x;
            if (i < nvec) r[u] = __ldg(src + i);
        }
        if (base == 0) {
            // the slot split, while the row loads are in flight
            for (int j = threadIdx.x; j < n; j += kWriteThreads) {
                const int64_t t = t0 + j;
                const int64_t slot = __ldg(p.slot_mapping + t);
                int64_t off = -1;  // padding (negative slot) or out of range: skipped
                if (slot >= p.num_slots) {
                    if (k == 0) record_error(p.err, PKV_DEVERR_SLOT, t);
                } else if (slot >= 0) {
                    const int64_t block = slot / p.block_size;
                    off = block * d.block_stride + (slot - block * p.block_size) * R;
                }
                dst_off[j] = off;
            }
            __syncthreads();
        }
#pragma unroll
        for (int u = 0; u < kVecsPerThread; ++u) {
            const int64_t i = base + u * kWriteThreads + threadIdx.x;
            if (i < nvec) {
                const int64_t byte = i * V;
                // n > 1 only when the batch holds at most kBatchVecs * 16 bytes
                const int tok = n == 1 ? 0
                                       : static_cast<int>(static_cast<uint32_t>(byte) /
                                                          static_cast<uint32_t>(R));
                const int64_t off = dst_off[tok];
                if (off >= 0)
                    *reinterpret_cast<VT *>(d.dst + off + (byte - tok * R)) = r[u];
            }
        }
    }
}

__global__ void __launch_bounds__(kWriteThreads)
    cache_write_kernel(const __grid_constant__ WriteParams p) {
    // a dependent launch (the decode kernel) may be scheduled now; it still
    // waits for this grid's completion before it reads the caches
    grid_launch_dependents();
    __shared__ int64_t dst_off[kBatchVecs];
    for (int64_t item = blockIdx.x; item < p.num_items; item += gridDim.x) {
        int k = 0;
        while (k + 1 < p.num_descs && p.d[k + 1].item0 <= item) ++k;
        const Desc &d = p.d[k];
        const int64_t t0 = (item - d.item0) * d.batch_tokens;
        const int n = static_cast<int>(min(static_cast<int64_t>(d.batch_tokens),
                                           p.num_tokens - t0));
        __syncthreads();  // the previous item's stores have read dst_off
        switch (d.vec) {
            case 16: write_item<uint4>(p, d, k, t0, n, dst_off); break;
            case 8: write_item<uint2>(p, d, k, t0, n, dst_off); break;
            case 4: write_item<unsigned int>(p, d, k, t0, n, dst_off); break;
            case 2: write_item<unsigned short>(p, d, k, t0, n, dst_off); break;
            default: write_item<unsigned char>(p, d, k, t0, n, dst_off); break;
        }
    }
}

bool view_ok(const pkv_view &v) {
    if (v.row_width <= 0 || v.row_width > kMaxRowWidth || v.block_stride <= 0 ||
        v.offset < 0 || v.layer < 0 || v.layer_stride < 0)
        return false;
    return !(v.layer > 0 && v.layer_stride > (INT64_MAX - v.offset) / v.layer);
}

// One descriptor; its vector is the widest size that every address and
// stride of the descriptor is a multiple of.
Desc make_desc(const void *src, void *cache, const pkv_view &v) {
    Desc d{};
    d.src = static_cast<const uint8_t *>(src);
    d.dst = static_cast<uint8_t *>(cache) + v.offset +
            static_cast<int64_t>(v.layer) * v.layer_stride;
    d.block_stride = v.block_stride;
    d.row_width = static_cast<int32_t>(v.row_width);
    const uintptr_t bits = reinterpret_cast<uintptr_t>(d.src) |
                           reinterpret_cast<uintptr_t>(d.dst) |
                           static_cast<uintptr_t>(v.block_stride) |
                           static_cast<uintptr_t>(v.row_width);
    d.vec = (bits & 15) == 0 ? 16 : (bits & 7) == 0 ? 8 : (bits & 3) == 0 ? 4
          : (bits & 1) == 0 ? 2 : 1;
    // tokens per item: as many whole rows as one item's vectors hold
    d.batch_tokens = static_cast<int32_t>(
        std::max<int64_t>(1, static_cast<int64_t>(kBatchVecs) * d.vec / v.row_width));
    return d;
}

int launch_write(WriteParams &p, cudaStream_t stream) {
    int64_t items = 0;
    for (int k = 0; k < p.num_descs; ++k) {
        p.d[k].item0 = items;
        items += (p.num_tokens + p.d[k].batch_tokens - 1) / p.d[k].batch_tokens;
    }
    p.num_items = items;
    // one wave of resident CTAs, each taking items in turn
    int per_sm = 0;
    const int st = prepare_kernel(reinterpret_cast<const void *>(cache_write_kernel),
                                  kWriteThreads, 0, &per_sm);
    if (st != PKV_OK) return st;
    const int64_t cap = static_cast<int64_t>(sm_count()) * std::max(1, per_sm);
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min(items, cap)));
    p.err = device_error_record();
    if (p.err == nullptr) return PKV_ERR_CUDA;
    cache_write_kernel<<<grid, kWriteThreads, 0, stream>>>(p);
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
