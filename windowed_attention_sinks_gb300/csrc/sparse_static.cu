// Gathered attention for callers that cannot allocate device memory.
//
// sattn_sparse_fwd splits short index lists across CTAs and needs a scratch
// buffer for the per-split partial outputs, which its caller allocates. Some
// callers cannot: a plug-in running inside a host application that has
// reserved all device memory for its own pool, a latency-critical loop whose
// policy forbids cudaMalloc/cudaFree after start-up (both can synchronise the
// device), or plain C code that is handed tensor pointers and a stream but no
// allocator. sattn_sparse_fwd_static_scratch serves them with a fixed array
// compiled into this library instead of a caller-provided workspace.
//
// Every GPU that loads the library holds this array until the process exits.
// All calls share it and it keeps the last call's contents; nothing in it
// needs to start at zero, because each split writes its whole partial result
// before the merge reads it. Calls whose work overlaps on the GPU (two
// streams, or two host threads on different streams) race on the array:
// issue them on one stream, or use sattn_sparse_fwd with separate buffers.
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace sattn {
namespace {

static __device__ __align__(256) unsigned char g_sparse_scratch[SATTN_SPARSE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device. The host-side
// name g_sparse_scratch is only a stand-in; the address is fetched once per
// device, with that device current, and cached.
cudaError_t scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_sparse_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace sattn

extern "C" sattn_status sattn_sparse_fwd_static_scratch(
    const void *q, const void *kv_cache, const int32_t *topk_idxs, const float *sinks,
    sattn_sink_mode sink_mode, float scale, void *o, float *lse, int32_t B, int32_t M, int32_t H,
    int32_t d, int32_t N, int32_t K, sattn_dtype dtype, void *cuda_stream) {
    // only the tensor-core path (bf16, 32 heads, d = 128) splits lists and
    // uses the scratch; the other shapes run without it
    const bool uses_scratch = dtype == SATTN_BF16 && H == 32 && d == 128;
    const size_t need = uses_scratch ? sattn_sparse_workspace_bytes(B, M, H, d, K) : 0;
    if (need > (size_t)SATTN_SPARSE_STATIC_SCRATCH_BYTES) {
        if (sattn::verbose())
            fprintf(stderr,
                    "sattn: sattn_sparse_fwd_static_scratch needs %zu bytes of scratch, more than "
                    "the built-in %zu; use sattn_sparse_fwd with a workspace\n",
                    need, (size_t)SATTN_SPARSE_STATIC_SCRATCH_BYTES);
        return SATTN_ERR_INVALID_ARG;
    }
    void *scratch = nullptr;
    if (sattn::scratch_address(&scratch) != cudaSuccess) return SATTN_ERR_CUDA;
    return sattn_sparse_fwd(q, kv_cache, topk_idxs, sinks, sink_mode, scale, o, lse, B, M, H, d, N,
                            K, scratch, (size_t)SATTN_SPARSE_STATIC_SCRATCH_BYTES, dtype,
                            cuda_stream);
}
