// pkv_api.cu -- status strings, the device error record and workspace sizing
// of libpagedkv (the C ABI declared in include/pagedkv.h).
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

__device__ ErrorRecord g_error_record;

namespace {
constexpr int kMaxDevices = 256;
ErrorRecord *g_error_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];
thread_local char g_last_error[256] = "no error";

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}
}  // namespace

int cuda_failure(cudaError_t e, const char *where) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return PKV_ERR_CUDA;
}

void set_last_error(const char *msg) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
}

ErrorRecord *device_error_record() {
    const int dev = current_device();
    if (dev < 0) {
        cuda_failure(cudaGetLastError(), "cudaGetDevice");
        return nullptr;
    }
    if (g_error_ptr[dev] == nullptr) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_error_record);
        if (e != cudaSuccess) {
            cuda_failure(e, "cudaGetSymbolAddress(error record)");
            return nullptr;
        }
        g_error_ptr[dev] = static_cast<ErrorRecord *>(p);
    }
    return g_error_ptr[dev];
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0) {  // no device: a generous stand-in (used only for sizing)
        cudaGetLastError();
        return 256;
    }
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 256;
        }
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

namespace {
struct KernelShape {
    int device;
    const void *fn;
    int threads;
    int smem;
    int ctas_per_sm;
};
constexpr int kKernelCache = 128;
KernelShape g_kernel_cache[kKernelCache];
int g_kernel_cache_used = 0;
std::mutex g_kernel_cache_mutex;
}  // namespace

int prepare_kernel(const void *fn, int threads, int smem, int *ctas_per_sm) {
    const int dev = current_device();
    if (dev < 0) return cuda_failure(cudaGetLastError(), "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_kernel_cache_mutex);
    int opened = -1;  // the largest dynamic shared memory this kernel is opened to
    for (int i = 0; i < g_kernel_cache_used; ++i) {
        const KernelShape &k = g_kernel_cache[i];
        if (k.device != dev || k.fn != fn) continue;
        if (k.threads == threads && k.smem == smem) {
            if (ctas_per_sm) *ctas_per_sm = k.ctas_per_sm;
            return PKV_OK;
        }
        opened = opened > k.smem ? opened : k.smem;
    }
    cudaError_t e = cudaSuccess;
    if (smem > opened)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_failure(e, "cudaFuncSetAttribute");
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
    if (e != cudaSuccess) return cuda_failure(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (g_kernel_cache_used < kKernelCache)
        g_kernel_cache[g_kernel_cache_used++] = KernelShape{dev, fn, threads, smem, per_sm};
    if (ctas_per_sm) *ctas_per_sm = per_sm;
    return PKV_OK;
}

}  // namespace pkv

extern "C" {

int pkv_get_device_error(int32_t *kind, int64_t *index, pkv_stream_t stream) {
    if (kind) *kind = PKV_DEVERR_NONE;
    if (index) *index = -1;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pkv::cuda_failure(e, "cudaStreamSynchronize");
    pkv::ErrorRecord *rec = pkv::device_error_record();
    if (rec == nullptr) return PKV_ERR_CUDA;
    unsigned long long word = 0;
    e = cudaMemcpy(&word, rec, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return pkv::cuda_failure(e, "cudaMemcpy(error record)");
    if (word != 0) {
        const unsigned long long zero = 0;
        e = cudaMemcpy(rec, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return pkv::cuda_failure(e, "cudaMemcpy(clear error record)");
        if (kind) *kind = static_cast<int32_t>(word >> 56);
        if (index) *index = static_cast<int64_t>(word & ((1ull << 56) - 1));
    }
    return PKV_OK;
}

const char *pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "PKV_OK: success";
        case PKV_ERR_NULL: return "PKV_ERR_NULL: a required pointer is NULL";
        case PKV_ERR_INVALID: return "PKV_ERR_INVALID: a size, stride or count is out of range";
        case PKV_ERR_UNSUPPORTED:
            return "PKV_ERR_UNSUPPORTED: shape not supported (head_dim, group size, block size)";
        case PKV_ERR_ALIGNMENT: return "PKV_ERR_ALIGNMENT: a pointer or stride is misaligned";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE: split-KV needs a larger workspace";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA: a CUDA call failed (see pkv_last_error_string)";
        default: return "unknown pkv status";
    }
}

const char *pkv_last_error_string(void) { return pkv::g_last_error; }

int pkv_version(void) { return 10000; }

}  // extern "C"
