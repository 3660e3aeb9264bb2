// pkv_decode_api.cu -- the C ABI of paged decode attention: argument checks,
// workspace sizing and the choice between the two schedules
// (pkv_decode_grid.cu, pkv_decode_balanced.cu).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "../../include/pagedkv.h"
#include "pkv_decode_host.h"
#include "pkv_internal.h"

namespace pkv {
namespace dec {
namespace {

constexpr int kBlockSize = 16;

int resolve_partition(const pkv_decode_options *opts) {
    return (opts && opts->partition_size) ? opts->partition_size : kDefaultPartitionTokens;
}

int64_t num_partitions(int64_t max_seq_len, int pt) {
    return std::max<int64_t>(1, (max_seq_len + pt - 1) / pt);
}

bool balanced_fits_index(int64_t num_seqs, int64_t max_blocks_per_seq) {
    return num_seqs * max_blocks_per_seq <= INT32_MAX;
}

}  // namespace

int check_decode_args(const void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, const int32_t *seq_lens, float scale,
                      int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t num_seqs, int32_t max_blocks_per_seq,
                      int32_t max_seq_len, int64_t num_blocks) {
    if (num_seqs < 0) return PKV_ERR_INVALID;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PKV_ERR_NULL;
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || max_seq_len < 0 ||
        !std::isfinite(scale))
        return PKV_ERR_INVALID;
    const int G = num_heads / num_kv_heads;
    if (!(G == 1 || G == 2 || G == 4 || G == 8)) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
    if (!pkv::aligned(out, 16) || !pkv::aligned(q, 16) || !pkv::aligned(k_cache, 16) ||
        !pkv::aligned(v_cache, 16) || !pkv::aligned(block_tables, 4) ||
        !pkv::aligned(seq_lens, 4))
        return PKV_ERR_ALIGNMENT;
    return PKV_OK;
}

}  // namespace dec
}  // namespace pkv

extern "C" {

size_t pkv_decode_workspace_bytes_ex(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t max_seq_len,
                                     int32_t partition_size) {
    using namespace pkv::dec;
    const int pt = partition_size ? partition_size : kDefaultPartitionTokens;
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        max_seq_len <= 0 || pt <= 0 || num_heads % num_kv_heads != 0)
        return 0;
    const int64_t grid_ws =
        grid_workspace_bytes(num_seqs, num_heads, head_dim, num_partitions(max_seq_len, pt));
    const int G = num_heads / num_kv_heads;
    int64_t need = grid_ws;
    for (const bool fp8 : {false, true}) {
        const BalancedShape b =
            balanced_shape(num_seqs, num_kv_heads, G, head_dim, pkv::sm_count(), fp8);
        if (b.ok) need = std::max(need, b.workspace);
    }
    return static_cast<size_t>(need);
}

size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_seq_len) {
    return pkv_decode_workspace_bytes_ex(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len,
                                         0);
}

int pkv_decode_workspace_init(void *workspace, size_t workspace_bytes, pkv_stream_t stream) {
    if (workspace_bytes == 0) return PKV_OK;
    if (workspace == nullptr) return PKV_ERR_NULL;
    cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes,
                                    reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : pkv::cuda_failure(e, "cudaMemsetAsync(workspace)");
}

int pkv_decode_attention_ex(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *seq_lens, float scale,
                            int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_seqs, int32_t max_blocks_per_seq,
                            int32_t max_seq_len, int64_t num_blocks, void *workspace,
                            size_t workspace_bytes, const pkv_decode_options *opts,
                            pkv_stream_t stream) {
    using namespace pkv;
    using namespace pkv::dec;
    if (num_seqs == 0) return PKV_OK;
    {
        const int st = check_decode_args(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                                         num_heads, num_kv_heads, head_dim, block_size, num_seqs,
                                         max_blocks_per_seq, max_seq_len, num_blocks);
        if (st != PKV_OK) return st;
    }
    const int G = num_heads / num_kv_heads;
    const int pt = resolve_partition(opts);
    if (pt < kBlockSize || pt > kMaxPartitionTokens || pt % kBlockSize != 0)
        return PKV_ERR_INVALID;
    const int compute = opts ? opts->compute : PKV_COMPUTE_AUTO;
    if (compute < PKV_COMPUTE_AUTO || compute > PKV_COMPUTE_MMA) return PKV_ERR_INVALID;
    const int schedule = opts ? opts->schedule : PKV_SCHEDULE_AUTO;
    if (schedule < PKV_SCHEDULE_AUTO || schedule > PKV_SCHEDULE_BALANCED) return PKV_ERR_INVALID;
    if (workspace != nullptr && !aligned(workspace, 16)) return PKV_ERR_ALIGNMENT;
    const bool simt = compute == PKV_COMPUTE_SIMT;  // measured: the MMA policy is faster
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);

    // ---- balanced schedule: the default whenever the shape and workspace allow
    if (schedule != PKV_SCHEDULE_GRID) {
        BalancedShape shape{};
        bool usable = balanced_fits_index(num_seqs, max_blocks_per_seq);
        if (usable) {
            shape = balanced_shape(num_seqs, num_kv_heads, G, head_dim, sm_count(), false);
            usable = shape.ok && workspace != nullptr &&
                     static_cast<int64_t>(workspace_bytes) >= shape.workspace;
        }
        if (schedule == PKV_SCHEDULE_BALANCED && !usable) {
            if (shape.ok && (workspace == nullptr ||
                             static_cast<int64_t>(workspace_bytes) < shape.workspace))
                return PKV_ERR_WORKSPACE;
            return PKV_ERR_UNSUPPORTED;
        }
        if (usable) {
            BalancedParams p{};
            p.out = static_cast<__half *>(out);
            p.q = static_cast<const __half *>(q);
            p.k_cache = static_cast<const __half *>(k_cache);
            p.v_cache = static_cast<const __half *>(v_cache);
            p.block_tables = block_tables;
            p.seq_lens = seq_lens;
            p.scale_log2 = scale_log2;
            p.num_seqs = num_seqs;
            p.num_heads = num_heads;
            p.num_kv_heads = num_kv_heads;
            p.max_blocks_per_seq = max_blocks_per_seq;
            p.num_blocks = num_blocks;
            const int st = setup_balanced(p, shape, G, workspace, k_cache, v_cache);
            if (st != PKV_OK) return st;
            p.err = device_error_record();
            if (p.err == nullptr) return PKV_ERR_CUDA;
            return launch_balanced(p, shape, head_dim, G, simt, false, s);
        }
    }

    // ---- grid schedule
    const int64_t P64 = num_partitions(max_seq_len, pt);
    if (P64 > 65535) return PKV_ERR_UNSUPPORTED;
    const int P = static_cast<int>(P64);
    GridParams p{};
    p.out = static_cast<__half *>(out);
    p.q = static_cast<const __half *>(q);
    p.k_cache = static_cast<const __half *>(k_cache);
    p.v_cache = static_cast<const __half *>(v_cache);
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.scale_log2 = scale_log2;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_partitions = P;
    p.partition_blocks = pt / kBlockSize;
    p.num_blocks = num_blocks;
    if (P > 1) {
        const int64_t need = grid_workspace_bytes(num_seqs, num_heads, head_dim, P);
        if (workspace == nullptr || static_cast<int64_t>(workspace_bytes) < need)
            return PKV_ERR_WORKSPACE;
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        const int64_t c_bytes = align256(static_cast<int64_t>(num_seqs) * num_heads * 4);
        const int64_t ml_bytes = align256(static_cast<int64_t>(num_seqs) * num_heads * P * 8);
        p.counters = reinterpret_cast<int *>(ws);
        p.part_ml = reinterpret_cast<float2 *>(ws + c_bytes);
        p.part_o = reinterpret_cast<float *>(ws + c_bytes + ml_bytes);
        // the combine's per-partition weights must fit in the (reused) ring
        if (static_cast<int64_t>(2 * G * P + 2 * G) * 4 > grid_ring_bytes(head_dim))
            return PKV_ERR_UNSUPPORTED;
    }
    {
        // per-head boxes: kv_head's head_dim*2 bytes are whole 128-byte chunks
        const int row_bytes = num_kv_heads * head_dim * 2;
        const int box = head_dim * 2 / chunk_bytes_for_row(row_bytes);
        int st = make_kv_tensor_map(&p.tm_k, k_cache, num_blocks, row_bytes, box);
        if (st == PKV_OK) st = make_kv_tensor_map(&p.tm_v, v_cache, num_blocks, row_bytes, box);
        if (st != PKV_OK) return st;
    }
    p.err = device_error_record();
    if (p.err == nullptr) return PKV_ERR_CUDA;
    return launch_grid(p, head_dim, G, simt, num_seqs, s);
}

int pkv_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *seq_lens, float scale,
                         int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int32_t num_seqs, int32_t max_blocks_per_seq,
                         int32_t max_seq_len, int64_t num_blocks, void *workspace,
                         size_t workspace_bytes, pkv_stream_t stream) {
    return pkv_decode_attention_ex(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                                   num_heads, num_kv_heads, head_dim, block_size, num_seqs,
                                   max_blocks_per_seq, max_seq_len, num_blocks, workspace,
                                   workspace_bytes, nullptr, stream);
}

}  // extern "C"

extern "C" int pkv_decode_attention_fp8(void *out, const void *q, const void *k_cache,
                                        const void *v_cache, const float *k_scale,
                                        const float *v_scale, const int32_t *block_tables,
                                        const int32_t *seq_lens, float scale, int32_t num_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t block_size, int32_t num_seqs,
                                        int32_t max_blocks_per_seq, int32_t max_seq_len,
                                        int64_t num_blocks, void *workspace,
                                        size_t workspace_bytes, pkv_stream_t stream) {
    using namespace pkv;
    using namespace pkv::dec;
    if (num_seqs < 0) return PKV_ERR_INVALID;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !k_scale || !v_scale || !block_tables || !seq_lens)
        return PKV_ERR_NULL;
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || max_seq_len < 0 ||
        !std::isfinite(scale))
        return PKV_ERR_INVALID;
    const int G = num_heads / num_kv_heads;
    if (!(G == 1 || G == 2 || G == 4 || G == 8)) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || !balanced_fits_index(num_seqs, max_blocks_per_seq))
        return PKV_ERR_UNSUPPORTED;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(k_scale, 16) || !aligned(v_scale, 16) || !aligned(block_tables, 4) ||
        !aligned(seq_lens, 4) || (workspace != nullptr && !aligned(workspace, 16)))
        return PKV_ERR_ALIGNMENT;
    const BalancedShape shape = balanced_shape(num_seqs, num_kv_heads, G, head_dim, sm_count(), true);
    if (!shape.ok) return PKV_ERR_UNSUPPORTED;
    if (workspace == nullptr || static_cast<int64_t>(workspace_bytes) < shape.workspace)
        return PKV_ERR_WORKSPACE;
    BalancedParams p{};
    p.out = static_cast<__half *>(out);
    p.q = static_cast<const __half *>(q);
    p.k_cache = static_cast<const __half *>(k_cache);  // E4M3 bytes, read as such
    p.v_cache = static_cast<const __half *>(v_cache);
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    const int st = setup_balanced(p, shape, G, workspace, k_cache, v_cache);
    if (st != PKV_OK) return st;
    p.err = device_error_record();
    if (p.err == nullptr) return PKV_ERR_CUDA;
    return launch_balanced(p, shape, head_dim, G, false, true,
                           reinterpret_cast<cudaStream_t>(stream));
}
