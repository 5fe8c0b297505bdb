// C ABI of libsattn.so: argument validation, per-device set-up and dispatch
// to the kernel launchers. No exception crosses this boundary and nothing is
// allocated: the only device memory the library owns is the error word below,
// a module-scope variable.
#include <stdio.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>
#include <new>

#include "common.cuh"
#include <algorithm>

#include "internal.h"

namespace sattn {

__device__ unsigned g_error_word;
// Item-claim counters of the persistent kernels, one per launch in turn, each
// on its own 128-byte line.
constexpr unsigned kClaimStride = 32;
__device__ unsigned g_claims[kClaimCounters * kClaimStride];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
DevInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices];
std::atomic<int> g_debug{0};
std::atomic<uint64_t> g_wait_ns{1000000000ull};
std::atomic<int> g_test_stall{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

cudaStream_t as_stream(void *s) {
    return s ? static_cast<cudaStream_t>(s) : cudaStreamPerThread;
}

sattn_status finish(cudaError_t e, cudaStream_t s) {
    if (e != cudaSuccess) {
        if (verbose()) fprintf(stderr, "sattn: CUDA error: %s\n", cudaGetErrorString(e));
        return SATTN_ERR_CUDA;
    }
    if (g_debug.load()) return sattn_check_device(s);
    return SATTN_OK;
}

bool is_device_ptr(const void *p) { return p != nullptr; }

}  // namespace

const DevInfo *device_info(cudaError_t *e) {
    int dev = -1;
    *e = cudaGetDevice(&dev);
    if (*e != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *e = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_ready[dev]) {
        DevInfo d;
        d.device = dev;
        if ((*e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) !=
            cudaSuccess)
            return nullptr;
        if ((*e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) !=
            cudaSuccess)
            return nullptr;
        if ((*e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
            cudaSuccess)
            return nullptr;
        void *p = nullptr;
        if ((*e = cudaGetSymbolAddress(&p, g_error_word)) != cudaSuccess) return nullptr;
        d.err = static_cast<unsigned *>(p);
        if ((*e = cudaGetSymbolAddress(&p, g_claims)) != cudaSuccess) return nullptr;
        d.claims = static_cast<unsigned *>(p);
        if ((*e = cudaMemset(d.err, 0, sizeof(unsigned))) != cudaSuccess) return nullptr;
        if ((*e = cudaDeviceSynchronize()) != cudaSuccess) return nullptr;
        g_dev[dev] = d;
        g_dev_ready[dev] = true;
    }
    return &g_dev[dev];
}

uint64_t wait_limit_ns() { return g_wait_ns.load(); }

DevCtx make_ctx(const DevInfo &dev) { return DevCtx{dev.err, g_wait_ns.load(), g_test_stall.load()}; }

unsigned *launch_claim_counter(const DevInfo &dev, cudaStream_t s, cudaError_t *e) {
    static std::atomic<unsigned> next{0};
    unsigned *c = dev.claims + (size_t)(next.fetch_add(1) % kClaimCounters) * kClaimStride;
    *e = cudaMemsetAsync(c, 0, sizeof(*c), s);
    return *e == cudaSuccess ? c : nullptr;
}

cudaError_t ensure_smem_attr(const void *kernel, size_t bytes, const DevInfo &dev) {
    struct Entry {
        const void *fn;
        int device;
        size_t bytes;
    };
    static std::mutex mu;
    static Entry done[256];
    static int ndone = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < ndone; ++i)
        if (done[i].fn == kernel && done[i].device == dev.device && done[i].bytes >= bytes)
            return cudaSuccess;
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    if (ndone < 256) done[ndone++] = Entry{kernel, dev.device, bytes};
    return cudaSuccess;
}

bool verbose() {
    static const bool v = getenv("SATTN_VERBOSE") != nullptr;
    return v;
}

CUresult encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t rank, void *base,
                           const uint64_t *dims, const uint64_t *strides_bytes,
                           const uint32_t *box, CUtensorMapSwizzle swizzle) {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    if (!g_encode) return CUDA_ERROR_NOT_FOUND;
    cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    return g_encode(map, dtype, rank, base, reinterpret_cast<const cuuint64_t *>(dims),
                    reinterpret_cast<const cuuint64_t *>(strides_bytes),
                    reinterpret_cast<const cuuint32_t *>(box), estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace sattn

using namespace sattn;

namespace {

bool valid_dtype(sattn_dtype t) { return t == SATTN_F32 || t == SATTN_BF16; }
bool valid_sink(sattn_sink_mode m, const float *sinks) {
    if (m == SATTN_SINK_NONE) return true;
    if (m != SATTN_SINK_KEY0_BIAS && m != SATTN_SINK_NULL_LOGIT) return false;
    return sinks != nullptr;
}
// The softmax scale must be finite and positive.
bool finite_scale(float s) { return s == s && s - s == 0.0f && s > 0.0f; }
// TMA tiles need 16-byte aligned base addresses.
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// sm_103 only: the fatbin carries sm_103a code and nothing else.
sattn_status check_arch(const DevInfo *dev) {
    if (dev->cc_major != 10 || dev->cc_minor != 3) return SATTN_ERR_UNSUPPORTED;
    return SATTN_OK;
}

}  // namespace

extern "C" {

int32_t sattn_version(void) { return 103; }

const char *sattn_status_str(sattn_status s) {
    switch (s) {
    case SATTN_OK: return "ok";
    case SATTN_ERR_INVALID_ARG: return "invalid argument";
    case SATTN_ERR_UNSUPPORTED: return "unsupported device or argument combination";
    case SATTN_ERR_CUDA: return "CUDA error";
    case SATTN_ERR_DEVICE_CHECK: return "device-side index or sequence check failed";
    case SATTN_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

void sattn_set_debug(int on) { g_debug.store(on ? 1 : 0); }

void sattn_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns ? ns : 1000000000ull); }

void sattn_set_test_wait_stall(int on) { g_test_stall.store(on ? 1 : 0); }

sattn_status sattn_check_device(void *cuda_stream) {
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    cudaStream_t s = as_stream(cuda_stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return SATTN_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, dev->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SATTN_ERR_CUDA;
    if (word) {
        unsigned zero = 0;
        if (cudaMemcpy(dev->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return SATTN_ERR_CUDA;
    }
    if (word & DEVERR_TIMEOUT) return SATTN_ERR_TIMEOUT;
    if (word) return SATTN_ERR_DEVICE_CHECK;
    return SATTN_OK;
}

sattn_status sattn_window_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                              const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                              int32_t max_seqlen, int32_t H, int32_t Hkv, int32_t d,
                              int32_t window_left, int32_t window_right, int32_t causal,
                              const float *sinks, sattn_sink_mode sink_mode, float scale,
                              sattn_dtype dtype, void *cuda_stream) {
    if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0) return SATTN_ERR_INVALID_ARG;
    if (H <= 0 || Hkv <= 0 || H % Hkv != 0) return SATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return SATTN_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || !valid_sink(sink_mode, sinks) || !finite_scale(scale))
        return SATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return SATTN_ERR_INVALID_ARG;
    if (total_tokens == 0 || num_seqs == 0) return SATTN_OK;
    if (max_seqlen == 0) return SATTN_ERR_INVALID_ARG;
    if (!is_device_ptr(q) || !is_device_ptr(k) || !is_device_ptr(v) || !is_device_ptr(o) ||
        !is_device_ptr(cu_seqlens))
        return SATTN_ERR_INVALID_ARG;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    WindowArgs a{q, k, v, o, lse, cu_seqlens, num_seqs, total_tokens, max_seqlen, H, Hkv, d,
                 window_left < 0 ? -1 : window_left, window_right < 0 ? -1 : window_right,
                 causal, sink_mode == SATTN_SINK_NONE ? nullptr : sinks, (int)sink_mode, scale,
                 (int)dtype};
    cudaStream_t s = as_stream(cuda_stream);
    if (dtype == SATTN_BF16 && d == 128) {
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
            return SATTN_ERR_INVALID_ARG;
        return finish(launch_window_tc(a, *dev, s), s);
    }
    return finish(launch_window_simt(a, *dev, s), s);
}

size_t sattn_sparse_workspace_bytes(int32_t B, int32_t M, int32_t H, int32_t d, int32_t K) {
    if (B <= 0 || M <= 0 || H <= 0 || d <= 0 || K <= 0) return 0;
    return sparse_tc_workspace_bytes(B, M, H, d, K);
}

sattn_status sattn_sparse_fwd(const void *q, const void *kv_cache, const int32_t *topk_idxs,
                              const float *sinks, sattn_sink_mode sink_mode, float scale, void *o,
                              float *lse, int32_t B, int32_t M, int32_t H, int32_t d, int32_t N,
                              int32_t K, void *workspace, size_t workspace_bytes,
                              sattn_dtype dtype, void *cuda_stream) {
    if (B < 0 || M < 0 || H <= 0 || N < 0 || K < 0) return SATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return SATTN_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || !valid_sink(sink_mode, sinks) || !finite_scale(scale))
        return SATTN_ERR_INVALID_ARG;
    if (B == 0 || M == 0) return SATTN_OK;
    if (N == 0) return SATTN_ERR_INVALID_ARG;
    if (!q || !kv_cache || !o || (K > 0 && !topk_idxs)) return SATTN_ERR_INVALID_ARG;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return SATTN_ERR_INVALID_ARG;
    if (dtype == SATTN_BF16 && d != 128) return SATTN_ERR_UNSUPPORTED;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    SparseArgs a{q, kv_cache, nullptr, nullptr, nullptr, topk_idxs,
                 sink_mode == SATTN_SINK_NONE ? nullptr : sinks, (int)sink_mode, scale, o, lse,
                 B, M, H, d, N, K, workspace, workspace_bytes, (int)dtype};
    cudaStream_t s = as_stream(cuda_stream);
    if (dtype == SATTN_BF16) {
        if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(o)) return SATTN_ERR_INVALID_ARG;
        return finish(launch_sparse_tc(a, *dev, s), s);
    }
    return finish(launch_sparse_simt(a, *dev, s), s);
}

sattn_status sattn_sparse_fp8_fwd(const void *q, const uint8_t *kv_nope, const void *kv_rope,
                                  const float *kv_scale, const int32_t *topk_idxs,
                                  const float *sinks, sattn_sink_mode sink_mode, float scale,
                                  void *o, float *lse, int32_t B, int32_t M, int32_t H, int32_t d,
                                  int32_t rd, int32_t N, int32_t K, void *workspace,
                                  size_t workspace_bytes, void *cuda_stream) {
    if (B < 0 || M < 0 || H <= 0 || N < 0 || K < 0 || d <= 0 || rd < 0 || rd > d)
        return SATTN_ERR_INVALID_ARG;
    if (!valid_sink(sink_mode, sinks) || !finite_scale(scale)) return SATTN_ERR_INVALID_ARG;
    if (B == 0 || M == 0) return SATTN_OK;
    if (N == 0) return SATTN_ERR_INVALID_ARG;
    if (!q || !kv_nope || !kv_rope || !kv_scale || !o || (K > 0 && !topk_idxs))
        return SATTN_ERR_INVALID_ARG;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return SATTN_ERR_INVALID_ARG;
    if (H != 32 || d != 128 || rd != 64) return SATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(kv_nope) || !aligned16(kv_rope) || !aligned16(o))
        return SATTN_ERR_INVALID_ARG;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    SparseArgs a{q, nullptr, kv_nope, kv_rope, kv_scale, topk_idxs,
                 sink_mode == SATTN_SINK_NONE ? nullptr : sinks, (int)sink_mode, scale, o, lse,
                 B, M, H, d, N, K, workspace, workspace_bytes, (int)SATTN_BF16};
    cudaStream_t s = as_stream(cuda_stream);
    return finish(launch_sparse_tc(a, *dev, s), s);
}

sattn_status sattn_quantize_kv_fp8(const void *kv, uint8_t *kv_nope, void *kv_rope,
                                   float *kv_scale, int64_t rows, int32_t d, int32_t rd,
                                   sattn_dtype dtype, void *cuda_stream) {
    if (rows < 0 || d <= 0 || rd < 0 || rd > d || d % 4 != 0 || rd % 4 != 0 || !valid_dtype(dtype))
        return SATTN_ERR_INVALID_ARG;
    if (rows == 0) return SATTN_OK;
    if (!kv || !kv_nope || !kv_rope || !kv_scale) return SATTN_ERR_INVALID_ARG;
    if (!aligned16(kv) || !aligned16(kv_nope) || !aligned16(kv_rope) || !aligned16(kv_scale))
        return SATTN_ERR_INVALID_ARG;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    cudaStream_t s = as_stream(cuda_stream);
    return finish(launch_quantize_kv_fp8(kv, kv_nope, kv_rope, kv_scale, rows, d, rd, (int)dtype,
                                         *dev, s),
                  s);
}

// shared validation of the two estimate passes
static sattn_status xattn_check(const void *q, const void *k, int32_t M, int32_t Nctx, int32_t H,
                                int32_t Hkv, int32_t d, int32_t q_pos0, int32_t kv_begin,
                                int32_t kv_end, int32_t causal, float scale) {
    if (M < 0 || Nctx < 0 || H <= 0 || H > 65535 || Hkv <= 0 || H % Hkv != 0 || q_pos0 < 0)
        return SATTN_ERR_INVALID_ARG;
    if (kv_begin < 0 || kv_end > Nctx || kv_begin > kv_end || (causal != 0 && causal != 1))
        return SATTN_ERR_INVALID_ARG;
    // chunks cover whole key blocks, so that each block sum comes from one chunk
    if (kv_begin % 128 != 0 || (kv_end % 128 != 0 && kv_end != Nctx)) return SATTN_ERR_INVALID_ARG;
    if (!finite_scale(scale)) return SATTN_ERR_INVALID_ARG;
    if (M > 0 && (!q || (Nctx > 0 && !k))) return SATTN_ERR_INVALID_ARG;
    if (M > 0 && (!aligned16(q) || (Nctx > 0 && !aligned16(k)))) return SATTN_ERR_INVALID_ARG;
    if (d != 128) return SATTN_ERR_UNSUPPORTED;
    return SATTN_OK;
}

sattn_status sattn_xattn_partial_stats(const void *q, const void *k, int32_t M, int32_t Nctx,
                                       int32_t H, int32_t Hkv, int32_t d, int32_t q_pos0,
                                       int32_t kv_begin, int32_t kv_end, int32_t causal,
                                       float scale, float *m, float *l, void *cuda_stream) {
    if (sattn_status st = xattn_check(q, k, M, Nctx, H, Hkv, d, q_pos0, kv_begin, kv_end, causal,
                                      scale))
        return st;
    if (M == 0) return SATTN_OK;
    if (!m || !l) return SATTN_ERR_INVALID_ARG;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    cudaStream_t s = as_stream(cuda_stream);
    XattnArgs a{q, k, M, Nctx, H, Hkv, q_pos0, kv_begin, kv_end, causal, scale, m, l, nullptr};
    return finish(launch_xattn_stats(a, *dev, s), s);
}

sattn_status sattn_xattn_merge_stats(const float *m_parts, const float *l_parts, int32_t C,
                                     int64_t R, float *m, float *l, void *cuda_stream) {
    if (C < 0 || R < 0) return SATTN_ERR_INVALID_ARG;
    if (R == 0) return SATTN_OK;
    if (!m || !l || (C > 0 && (!m_parts || !l_parts))) return SATTN_ERR_INVALID_ARG;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    cudaStream_t s = as_stream(cuda_stream);
    return finish(launch_xattn_merge_stats(m_parts, l_parts, C, R, m, l, s), s);
}

sattn_status sattn_xattn_block_sum(const void *q, const void *k, const float *m, const float *l,
                                   int32_t M, int32_t Nctx, int32_t H, int32_t Hkv, int32_t d,
                                   int32_t q_pos0, int32_t kv_begin, int32_t kv_end,
                                   int32_t causal, float scale, float *block_sum,
                                   void *cuda_stream) {
    if (sattn_status st = xattn_check(q, k, M, Nctx, H, Hkv, d, q_pos0, kv_begin, kv_end, causal,
                                      scale))
        return st;
    if (M == 0 || kv_begin == kv_end) return SATTN_OK;
    if (!m || !l || !block_sum) return SATTN_ERR_INVALID_ARG;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    cudaStream_t s = as_stream(cuda_stream);
    XattnArgs a{q, k, M, Nctx, H, Hkv, q_pos0, kv_begin, kv_end, causal, scale,
                const_cast<float *>(m), const_cast<float *>(l), block_sum};
    return finish(launch_xattn_block_sum(a, *dev, s), s);
}

sattn_status sattn_xattn_find_blocks(const float *block_sum, int32_t H, int32_t QB, int32_t KB,
                                     float threshold, uint8_t *mask, void *cuda_stream) {
    if (H < 0 || QB < 0 || KB < 0 || KB > 4096 || !(threshold >= 0.f && threshold <= 1.f))
        return SATTN_ERR_INVALID_ARG;
    if ((int64_t)H * QB * KB == 0) return SATTN_OK;
    if ((int64_t)H * QB > 0x7fffffff) return SATTN_ERR_INVALID_ARG;
    if (!block_sum || !mask) return SATTN_ERR_INVALID_ARG;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    cudaStream_t s = as_stream(cuda_stream);
    return finish(launch_xattn_find_blocks(block_sum, H * QB, KB, threshold, mask, s), s);
}

size_t sattn_xattn_select_workspace_bytes(int32_t M, int32_t H, int32_t Nctx, int32_t chunk) {
    if (M <= 0 || H <= 0 || Nctx <= 0 || chunk <= 0) return 0;
    const size_t C = ((size_t)Nctx + (size_t)chunk - 1) / (size_t)chunk;
    return (2 * C + 2) * (size_t)M * (size_t)H * sizeof(float);
}

sattn_status sattn_xattn_select_blocks(const void *q, const void *k, int32_t M, int32_t Nctx,
                                       int32_t H, int32_t Hkv, int32_t d, int32_t q_pos0,
                                       int32_t causal, float scale, int32_t chunk,
                                       float threshold, void *workspace, size_t workspace_bytes,
                                       float *block_sum, uint8_t *mask, void *cuda_stream) {
    if (sattn_status st = xattn_check(q, k, M, Nctx, H, Hkv, d, q_pos0, 0, Nctx, causal, scale))
        return st;
    if (chunk <= 0 || chunk % 128 != 0 || !(threshold >= 0.f && threshold <= 1.f))
        return SATTN_ERR_INVALID_ARG;
    const int64_t C = ((int64_t)Nctx + chunk - 1) / chunk;
    const int64_t QB = ((int64_t)M + 127) / 128, KB = ((int64_t)Nctx + 127) / 128;
    if (C > 65535 || KB > 4096 || (int64_t)H * QB > 0x7fffffff) return SATTN_ERR_INVALID_ARG;
    if (M == 0 || Nctx == 0) return SATTN_OK;
    if (!workspace || !block_sum || !mask || !aligned16(workspace) ||
        workspace_bytes < sattn_xattn_select_workspace_bytes(M, H, Nctx, chunk))
        return SATTN_ERR_INVALID_ARG;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    cudaStream_t s = as_stream(cuda_stream);
    const int64_t R = (int64_t)M * H;
    float *mp = static_cast<float *>(workspace), *lp = mp + C * R, *m = lp + C * R, *l = m + R;
    XattnArgs a1{q, k, M, Nctx, H, Hkv, q_pos0, 0, Nctx, causal, scale, mp, lp, nullptr, chunk};
    e = launch_xattn_stats(a1, *dev, s);
    if (e == cudaSuccess) e = launch_xattn_merge_stats(mp, lp, (int)C, R, m, l, s);
    XattnArgs a3{q, k, M, Nctx, H, Hkv, q_pos0, 0, Nctx, causal, scale, m, l, block_sum, 0};
    if (e == cudaSuccess) e = launch_xattn_block_sum(a3, *dev, s);
    if (e == cudaSuccess)
        e = launch_xattn_find_blocks(block_sum, (int)(H * QB), (int)KB, threshold, mask, s);
    return finish(e, s);
}

sattn_status sattn_merge_lse(const float *o_parts, const float *lse_parts, int32_t C, int64_t R,
                             int32_t d, int32_t H, const float *sinks, void *o, float *lse,
                             sattn_dtype dtype, void *cuda_stream) {
    if (C < 0 || R < 0 || d <= 0 || d > 1024 || H <= 0 || !valid_dtype(dtype))
        return SATTN_ERR_INVALID_ARG;
    if (R == 0) return SATTN_OK;
    if ((C > 0 && (!o_parts || !lse_parts)) || !o) return SATTN_ERR_INVALID_ARG;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    MergeArgs a{o_parts, lse_parts, C, R, d, H, sinks, o, lse, (int)dtype};
    cudaStream_t s = as_stream(cuda_stream);
    return finish(launch_merge(a, *dev, s), s);
}

sattn_status sattn_build_topk_idxs(int32_t *topk_idxs, const int32_t *start_pos, int32_t B,
                                   int32_t M, int32_t K, int32_t win, int32_t ratio,
                                   void *cuda_stream) {
    if (B < 0 || M < 0 || K < 0 || win < 1 || ratio < 0) return SATTN_ERR_INVALID_ARG;
    if ((long long)B * M * K == 0) return SATTN_OK;
    if (!topk_idxs || !start_pos) return SATTN_ERR_INVALID_ARG;
    if ((K & 3) == 0 && (reinterpret_cast<uintptr_t>(topk_idxs) & 15u)) return SATTN_ERR_INVALID_ARG;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    cudaStream_t s = as_stream(cuda_stream);
    return finish(launch_topk_idxs(topk_idxs, start_pos, B, M, K, win, ratio, *dev, s), s);
}

sattn_status sattn_kv_ring_write(void *kv_cache, const void *kv_new, const int32_t *start_pos,
                                 int32_t B, int32_t S, int32_t N, int32_t d, int32_t win,
                                 sattn_dtype dtype, void *cuda_stream) {
    if (B < 0 || S < 0 || d <= 0 || win < 1 || N < win || !valid_dtype(dtype))
        return SATTN_ERR_INVALID_ARG;
    const int elem = dtype == SATTN_BF16 ? 2 : 4;
    if ((d * elem) % 16 != 0) return SATTN_ERR_INVALID_ARG;
    if ((long long)B * S == 0) return SATTN_OK;
    if (!kv_cache || !kv_new || !start_pos) return SATTN_ERR_INVALID_ARG;
    if (!aligned16(kv_cache) || !aligned16(kv_new)) return SATTN_ERR_INVALID_ARG;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    cudaStream_t s = as_stream(cuda_stream);
    return finish(launch_kv_ring_write(kv_cache, kv_new, start_pos, B, S, N, d, win, elem, *dev, s),
                  s);
}

sattn_status sattn_compress_kv(const void *kv, const void *score, const float *ape, void *out,
                               int64_t out_batch_stride, int32_t B, int32_t S, int32_t d,
                               int32_t ratio, int32_t overlap, sattn_dtype in_dtype,
                               sattn_dtype out_dtype, void *cuda_stream) {
    if (B < 0 || S < 0 || ratio < 1 || (overlap != 0 && overlap != 1)) return SATTN_ERR_INVALID_ARG;
    if (d <= 0 || d % 4 != 0 || !valid_dtype(in_dtype) || !valid_dtype(out_dtype))
        return SATTN_ERR_INVALID_ARG;
    const int64_t nwin = S / ratio;
    if (out_batch_stride < nwin * d || out_batch_stride % 4 != 0) return SATTN_ERR_INVALID_ARG;
    if ((int64_t)B * nwin == 0) return SATTN_OK;
    if (!kv || !score || !ape || !out) return SATTN_ERR_INVALID_ARG;
    if (!aligned16(kv) || !aligned16(score) || !aligned16(ape) || !aligned16(out))
        return SATTN_ERR_INVALID_ARG;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    cudaStream_t s = as_stream(cuda_stream);
    CompressArgs a{kv, score, ape, out, out_batch_stride, B, S, d, ratio, overlap,
                   (int)in_dtype, (int)out_dtype};
    return finish(launch_compress_kv(a, *dev, s), s);
}

sattn_status sattn_block_sparse_fwd(const void *q, const void *k, const void *v,
                                    const uint8_t *block_mask, int32_t M, int32_t Nctx, int32_t H,
                                    int32_t Hkv, int32_t d, int32_t q_pos0, int32_t kv_begin,
                                    int32_t kv_end, int32_t causal, float scale, float *o_part,
                                    float *lse_part, sattn_dtype dtype, void *cuda_stream) {
    if (M < 0 || Nctx < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0) return SATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return SATTN_ERR_INVALID_ARG;
    if (q_pos0 < 0 || kv_begin < 0 || kv_end > Nctx || kv_begin > kv_end)
        return SATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return SATTN_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || !finite_scale(scale)) return SATTN_ERR_INVALID_ARG;
    if (M == 0) return SATTN_OK;
    if (!q || !o_part || !lse_part || (Nctx > 0 && (!k || !v || !block_mask)))
        return SATTN_ERR_INVALID_ARG;
    if (dtype == SATTN_BF16 && d != 128) return SATTN_ERR_UNSUPPORTED;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    BlockArgs a{q, k, v, block_mask, M, Nctx, H, Hkv, d, q_pos0, kv_begin, kv_end, causal, scale,
                o_part, lse_part, (int)dtype};
    cudaStream_t s = as_stream(cuda_stream);
    if (dtype == SATTN_BF16) {
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_part))
            return SATTN_ERR_INVALID_ARG;
        return finish(launch_block_tc(a, *dev, s), s);
    }
    return finish(launch_block_simt(a, *dev, s), s);
}

sattn_status sattn_block_sparse_chunks_fwd(const void *q, const void *k, const void *v,
                                           const uint8_t *block_mask, int32_t M, int32_t Nctx,
                                           int32_t H, int32_t Hkv, int32_t d, int32_t q_pos0,
                                           int32_t kv_begin, int32_t kv_end, int32_t chunk,
                                           int32_t causal, float scale, float *o_parts,
                                           float *lse_parts, sattn_dtype dtype,
                                           void *cuda_stream) {
    if (M < 0 || Nctx < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0) return SATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return SATTN_ERR_INVALID_ARG;
    if (q_pos0 < 0 || kv_begin < 0 || kv_end > Nctx || kv_begin > kv_end || chunk <= 0)
        return SATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return SATTN_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || !finite_scale(scale)) return SATTN_ERR_INVALID_ARG;
    const int64_t C = ((int64_t)kv_end - kv_begin + chunk - 1) / chunk;
    if (M == 0 || C == 0) return SATTN_OK;
    if (!q || !o_parts || !lse_parts || !k || !v || !block_mask) return SATTN_ERR_INVALID_ARG;
    if (dtype == SATTN_BF16 && d != 128) return SATTN_ERR_UNSUPPORTED;
    cudaError_t e;
    const DevInfo *dev = device_info(&e);
    if (!dev) return SATTN_ERR_CUDA;
    if (sattn_status st = check_arch(dev)) return st;
    cudaStream_t s = as_stream(cuda_stream);
    if (dtype == SATTN_BF16) {
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_parts))
            return SATTN_ERR_INVALID_ARG;
        BlockArgs a{q, k, v, block_mask, M, Nctx, H, Hkv, d, q_pos0, kv_begin, kv_end, causal,
                    scale, o_parts, lse_parts, (int)dtype, chunk};
        return finish(launch_block_tc(a, *dev, s), s);
    }
    // F32: one launch per chunk
    const size_t rows = (size_t)M * H;
    for (int64_t c = 0; c < C; ++c) {
        const int b0 = kv_begin + (int)(c * chunk);
        const int b1 = (int)std::min<int64_t>(kv_end, (int64_t)b0 + chunk);
        BlockArgs a{q, k, v, block_mask, M, Nctx, H, Hkv, d, q_pos0, b0, b1, causal, scale,
                    o_parts + (size_t)c * rows * d, lse_parts + (size_t)c * rows, (int)dtype, 0};
        e = launch_block_simt(a, *dev, s);
        if (e != cudaSuccess) break;
    }
    return finish(e, s);
}

}  // extern "C"
