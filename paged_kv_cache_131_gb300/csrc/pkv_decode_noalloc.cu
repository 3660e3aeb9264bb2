// pkv_decode_noalloc.cu -- paged decode attention for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain scratch memory: a plugin running inside
// a host runtime that owns the whole device-memory budget and hands it only
// inputs and outputs, or a latency-critical loop that must never call
// cudaMalloc (which can synchronise the device).  This entry point runs the
// same decode kernels as pkv_decode_attention, but their scratch (split-
// sequence partials and the ticket counters) lives in a file-scope device
// array of fixed size instead of a caller-provided workspace.  It calls no
// cudaMalloc, cudaFree or other allocating routine.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstdio>

#include "../../include/pagedkv.h"
#include "pkv_decode_host.h"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr size_t kScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;

// The scratch.  Every device that loads the library holds these bytes until
// the process exits.  In host code this name is only a host-side stand-in:
// kernels get its device address from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 256;
void *g_scratch_ptr[kMaxDevices];  // device address per device, set up once

// Device address of the scratch on the current device (set up on first use,
// with that device current).  nullptr on failure (the CUDA error is kept).
void *scratch_on_current_device() {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cuda_failure(e == cudaSuccess ? cudaErrorInvalidDevice : e, "cudaGetDevice");
        return nullptr;
    }
    if (g_scratch_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            cuda_failure(e == cudaSuccess ? cudaErrorInvalidSymbol : e,
                         "cudaGetSymbolAddress(no-alloc scratch)");
            return nullptr;
        }
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_decode_attention_noalloc(void *out, const void *q, const void *k_cache,
                                            const void *v_cache, const int32_t *block_tables,
                                            const int32_t *seq_lens, float scale,
                                            int32_t num_heads, int32_t num_kv_heads,
                                            int32_t head_dim, int32_t block_size,
                                            int32_t num_seqs, int32_t max_blocks_per_seq,
                                            int32_t max_seq_len, int64_t num_blocks,
                                            pkv_stream_t stream) {
    using namespace pkv;
    if (num_seqs == 0) return PKV_OK;
    // Every check that can fail without a launch comes first, so a refused
    // call enqueues nothing and leaves the shared scratch alone.
    {
        const int st = dec::check_decode_args(out, q, k_cache, v_cache, block_tables, seq_lens,
                                              scale, num_heads, num_kv_heads, head_dim,
                                              block_size, num_seqs, max_blocks_per_seq,
                                              max_seq_len, num_blocks);
        if (st != PKV_OK) return st;
    }
    // The scratch must hold what the chosen schedule needs: the balanced
    // schedule's partials when they fit (it is then the one that runs), else
    // the grid schedule's.  Larger shapes are refused before anything runs.
    const int G = num_heads / num_kv_heads;
    const dec::BalancedShape bal =
        dec::balanced_shape(num_seqs, num_kv_heads, G, head_dim, sm_count(), false);
    const int64_t P = std::max<int64_t>(
        1, (static_cast<int64_t>(max_seq_len) + dec::kDefaultPartitionTokens - 1) /
               dec::kDefaultPartitionTokens);
    const int64_t grid_need = dec::grid_workspace_bytes(num_seqs, num_heads, head_dim, P);
    // (the balanced schedule also needs its flattened block index to fit 31 bits)
    const bool bal_fits = bal.ok && bal.workspace <= static_cast<int64_t>(kScratchBytes) &&
                          static_cast<int64_t>(num_seqs) * max_blocks_per_seq <= INT32_MAX;
    // the grid schedule's own limits: partitions per sequence, and the
    // combine's per-partition weights held in its staging ring
    if (!bal_fits && (P > 65535 || (P > 1 && (2 * G * P + 2 * G) * 4 >
                                                 dec::grid_ring_bytes(head_dim))))
        return PKV_ERR_UNSUPPORTED;
    if (!bal_fits && grid_need > static_cast<int64_t>(kScratchBytes)) {
        char msg[200];
        std::snprintf(msg, sizeof(msg),
                      "pkv_decode_attention_noalloc: this shape needs %lld bytes of scratch, "
                      "the built-in scratch holds %zu (use pkv_decode_attention)",
                      static_cast<long long>(bal.ok ? std::min(bal.workspace, grid_need)
                                                    : grid_need),
                      kScratchBytes);
        set_last_error(msg);
        return PKV_ERR_WORKSPACE;
    }
    void *scratch = scratch_on_current_device();
    if (scratch == nullptr) return PKV_ERR_CUDA;
    // The ticket counters must start at zero; the scratch keeps whatever the
    // previous call (of any shape) left, so clear the counter region (at most
    // num_seqs * num_heads int32, at the start of the scratch) every call.
    const size_t counters = (static_cast<size_t>(num_seqs) * num_heads * 4 + 255) / 256 * 256;
    cudaError_t e = cudaMemsetAsync(scratch, 0, std::min(counters, kScratchBytes),
                                    reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_failure(e, "cudaMemsetAsync(no-alloc scratch counters)");
    return pkv_decode_attention_ex(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                                   num_heads, num_kv_heads, head_dim, block_size, num_seqs,
                                   max_blocks_per_seq, max_seq_len, num_blocks, scratch,
                                   kScratchBytes, nullptr, stream);
}
