// mla_static.cu -- dsa_sparse_mla_static: sparse MLA attention that performs
// no device-memory allocation and takes no workspace.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocating API)
// around the attention call.  Examples are code that runs where an allocation
// would be unsafe or too slow -- a latency-critical serving step that must not
// take the implicit device synchronisation an allocation can cause, a plug-in
// running under a host framework that owns all device memory through its own
// pool and forbids raw allocations, or a caller that simply has no workspace
// buffer to hand over.  Such callers still own their inputs and outputs.
//
// How: the split-K partial results live in one file-scope __device__ array of
// fixed size, kStaticScratchBytes, which every GPU that loads this library
// holds until the process exits.  Host code obtains the array's device address
// with cudaGetSymbolAddress once per device (the host-side name of the array
// is only a stand-in, not a device address); the first call on each device
// does that set-up, so make that first call before any stream capture.
//
// Limits and sharing: requests whose split-K partials would not fit in the
// array are rejected with DSA_ERR_UNSUPPORTED (and a message on stderr).
// Every call on a device uses the same array and leaves its contents behind;
// the call clears the array's error word itself and overwrites every partial
// it later reads; dsa_sparse_mla_static_get_error reads (and clears) the
// error word of the last call.  Calls whose kernels overlap on the GPU (e.g. on two
// streams without ordering) race on the array and must be avoided.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "dsa.h"
#include "kernels.h"

namespace {

// 256 bytes of error word, then partial outputs and (max, sum) pairs.
constexpr size_t kStaticErrBytes = 256;
constexpr size_t kStaticScratchBytes = 32u << 20;  // 32 MiB per device

static __device__ __align__(256) unsigned char g_mla_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_mla_scratch on the current device (set up on first use).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_mla_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" dsa_status dsa_sparse_mla_static(const void *q, const void *kv_cache, const void *kv_rope,
                                            const float *kv_scale, int64_t num_pages, const int32_t *page_table,
                                            int32_t max_pages_per_seq, const int32_t *seq_lens, const int32_t *cu_q,
                                            const int32_t *indices, int32_t B, int32_t T, int32_t H, int32_t K,
                                            float scale, int32_t page_size, dsa_kv_dtype dtype, void *out,
                                            float *lse, void *stream) {
    // the same split choice as dsa_sparse_mla, so both give the same result
    const size_t need = dsa::mla_split_workspace_size(T, H, K);
    if (need > kStaticScratchBytes) {
        fprintf(stderr,
                "[dsa] dsa_sparse_mla_static: %zu bytes of split partials needed, the static scratch holds %zu; "
                "use dsa_sparse_mla with a workspace\n",
                need, kStaticScratchBytes);
        return DSA_ERR_UNSUPPORTED;
    }
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        fprintf(stderr, "[dsa] dsa_sparse_mla_static: cudaGetSymbolAddress failed: %s\n", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    // the error word must start at zero; the partials are rewritten by the call
    e = cudaMemsetAsync(scratch, 0, kStaticErrBytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        fprintf(stderr, "[dsa] dsa_sparse_mla_static: %s\n", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    return dsa_sparse_mla(q, kv_cache, kv_rope, kv_scale, num_pages, page_table, max_pages_per_seq, seq_lens, cu_q,
                          indices, B, T, H, K, scale, page_size, dtype, out, lse, scratch, kStaticScratchBytes,
                          stream);
}

extern "C" dsa_status dsa_sparse_mla_static_get_error(void *stream) {
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        fprintf(stderr, "[dsa] dsa_sparse_mla_static_get_error: cudaGetSymbolAddress failed: %s\n",
                cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    // the array's first 256 bytes are an ordinary workspace error block
    return dsa_get_error(scratch, stream);
}
