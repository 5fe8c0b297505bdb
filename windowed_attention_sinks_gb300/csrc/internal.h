// Host-side interface between the C ABI (api.cu) and the kernel launchers.
// Arguments reaching a launcher have already been validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "sattn.h"
#include "common.cuh"

namespace sattn {

struct DevInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    unsigned *err = nullptr;                 // device address of the error word
    unsigned *claims = nullptr;              // device address of the claim-counter ring
};

// Per-device facts, initialised once per device (thread-safe).
const DevInfo *device_info(cudaError_t *e);
uint64_t wait_limit_ns();
// The device context of one launch: error word, wait limit, test stall flag.
struct DevCtx make_ctx(const DevInfo &dev);

// The item-claim counter of one launch of a persistent kernel that hands
// out work items dynamically: the next of a ring of kClaimCounters built into
// the library (each on its own 128-byte line), zeroed by an asynchronous
// memset on `s`. Two launches that get the same counter (kClaimCounters
// launches apart in issue order) must not overlap on the GPU; the header
// states this limit. Returns nullptr (and sets *e) if the memset cannot be
// issued.
constexpr unsigned kClaimCounters = 256;
unsigned *launch_claim_counter(const DevInfo &dev, cudaStream_t s, cudaError_t *e);

// cudaFuncSetAttribute(kernel, MaxDynamicSharedMemorySize, bytes) once per
// (kernel, device, size), thread-safe.
cudaError_t ensure_smem_attr(const void *kernel, size_t bytes, const DevInfo &dev);
// True when the environment variable SATTN_VERBOSE is set (launch reports on stderr).
bool verbose();

// cuTensorMapEncodeTiled through the driver entry point (no libcuda link).
CUresult encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t rank,
                           void *base, const uint64_t *dims, const uint64_t *strides_bytes,
                           const uint32_t *box, CUtensorMapSwizzle swizzle);

struct WindowArgs {
    const void *q, *k, *v;
    void *o;
    float *lse;
    const int32_t *cu_seqlens;
    int num_seqs, T, max_seqlen, H, Hkv, d, wl, wr, causal;
    const float *sinks;
    int sink_mode;
    float scale;
    int dtype;
};

struct SparseArgs {
    const void *q, *kv;
    // FP8 cache (kv == nullptr): e4m3 codes [B, N, d - 64], one fp32 scale per
    // row, bf16 RoPE part [B, N, 64]
    const uint8_t *kv_nope;
    const void *kv_rope;
    const float *kv_scale;
    const int32_t *idx;
    const float *sinks;
    int sink_mode;
    float scale;
    void *o;
    float *lse;
    int B, M, H, d, N, K;
    void *workspace;
    size_t workspace_bytes;
    int dtype;
};

struct BlockArgs {
    const void *q, *k, *v;
    const uint8_t *mask;
    int M, Nctx, H, Hkv, d, q_pos0, kv_begin, kv_end, causal;
    float scale;
    float *o_part, *lse_part;  // [C, M, H, d], [C, M, H]
    int dtype;
    int chunk;  // > 0: [kv_begin, kv_end) in C chunks of this many keys; 0: one chunk
};

struct MergeArgs {
    const float *o_parts, *lse_parts;
    int C;
    int64_t R;
    int d, H;
    const float *sinks;
    void *o;
    float *lse;
    int dtype;
};

// Compressor gated pooling: kv / score [B, S, coff*d] (in_dtype), ape fp32
// [ratio, coff*d], rows to out + b * out_batch_stride + w * d (out_dtype).
struct CompressArgs {
    const void *kv, *score;
    const float *ape;
    void *out;
    int64_t out_batch_stride;
    int B, S, d, ratio, overlap;
    int in_dtype, out_dtype;
};

// Block selection estimate: q [M, H, 128], k [Nctx, Hkv, 128] (bf16).
struct XattnArgs {
    const void *q, *k;
    int M, Nctx, H, Hkv, q_pos0, kv_begin, kv_end, causal;
    float scale;
    float *m, *l;      // [M, H]
    float *block_sum;  // [H, ceil(M/128), ceil(Nctx/128)]
    int chunk;         // stage 1: keys per (m, l) output, outputs [C, M, H]; 0: one output
};

// SIMT kernels: any dtype, d in {64, 128}.
cudaError_t launch_window_simt(const WindowArgs &a, const DevInfo &dev, cudaStream_t s);
cudaError_t launch_sparse_simt(const SparseArgs &a, const DevInfo &dev, cudaStream_t s);
cudaError_t launch_block_simt(const BlockArgs &a, const DevInfo &dev, cudaStream_t s);
cudaError_t launch_topk_idxs(int32_t *out, const int32_t *start_pos, int B, int M, int K, int win,
                             int ratio, const DevInfo &dev, cudaStream_t s);
cudaError_t launch_kv_ring_write(void *cache, const void *src, const int32_t *start_pos, int B,
                                 int S, int N, int d, int win, int elem_bytes, const DevInfo &dev,
                                 cudaStream_t s);
cudaError_t launch_compress_kv(const CompressArgs &a, const DevInfo &dev, cudaStream_t s);
cudaError_t launch_xattn_stats(const XattnArgs &a, const DevInfo &dev, cudaStream_t s);
cudaError_t launch_xattn_block_sum(const XattnArgs &a, const DevInfo &dev, cudaStream_t s);
cudaError_t launch_xattn_merge_stats(const float *m_parts, const float *l_parts, int C, long long R,
                                     float *m_out, float *l_out, cudaStream_t s);
cudaError_t launch_xattn_find_blocks(const float *block_sum, int rows, int KB, float threshold,
                                     uint8_t *mask, cudaStream_t s);
cudaError_t launch_quantize_kv_fp8(const void *kv, uint8_t *nope, void *rope, float *row_scale,
                                   long long rows, int d, int rd, int dtype, const DevInfo &dev,
                                   cudaStream_t s);
// after_primary: launched as a programmatic dependent of the kernel just
// issued on `s` (that kernel triggers early; the merge waits for its results).
cudaError_t launch_merge(const MergeArgs &a, const DevInfo &dev, cudaStream_t s,
                         bool after_primary = false);

// tcgen05 kernels: bf16, d = 128.
cudaError_t launch_window_tc(const WindowArgs &a, const DevInfo &dev, cudaStream_t s);
cudaError_t launch_block_tc(const BlockArgs &a, const DevInfo &dev, cudaStream_t s);
cudaError_t launch_sparse_tc(const SparseArgs &a, const DevInfo &dev, cudaStream_t s);
// Few queries: each query's list cut into C segments, one per CTA of a
// cluster, merged through distributed shared memory. Returns the cluster
// size C for a shape this kernel takes (H = 32, d = 128; bf16 or FP8 cache), else 0.
int sparse_decode_cluster(int B, int M, int K, int sm_count);
cudaError_t launch_sparse_decode(const SparseArgs &a, int C, const DevInfo &dev, cudaStream_t s);
size_t sparse_tc_workspace_bytes(int B, int M, int H, int d, int K);

}  // namespace sattn
