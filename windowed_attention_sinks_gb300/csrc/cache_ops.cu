// Cache bookkeeping around the gathered path ("DeepSeek-V4 CSA/HCA
// walkthrough", section 2.3 steps 5-6 and section 3.3): the per-query index
// lists over a [window ring | compressed] cache, and the ring write of new
// KV rows. Both are pure data movement: coalesced stores of int32 entries,
// 16-byte row copies.
#include "common.cuh"
#include "internal.h"

namespace sattn {
namespace {

// A warp writes 512 consecutive entries of one query's list: lane l takes
// the groups of four entries l, l + 32, l + 64, l + 96 of that span, so every
// store instruction of the warp covers 512 contiguous bytes (int4 stores when
// K % 4 == 0). Integer work is hoisted out of the entries: with
// base = (p + 1) mod win, window slot k (token t = p - win + 1 + k >= 0) sits
// at ring row (base + k) mod win, a single conditional subtraction.
constexpr int GROUPS = 4;              // groups of four entries per thread
constexpr int SPAN = 32 * 4 * GROUPS;  // entries per warp

__global__ void topk_idxs_kernel(int32_t *__restrict__ out, const int32_t *__restrict__ start_pos,
                                 int M, int K, int win, int ratio, int warps_per_row, int total,
                                 DevCtx ctx) {
    const int g = blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= total) return;
    const int w = g >> 5, lane = g & 31;
    const int row = w / warps_per_row;  // (b, m)
    const int kw = (w - row * warps_per_row) * SPAN;
    const int b = row / M, m = row - b * M;
    const int sp = __ldg(start_pos + b);
    // positions are 0 .. 2^31 - 2 (32-bit arithmetic below); others leave the
    // lists at -1 and are reported
    const bool ok = sp >= 0 && sp <= 0x7ffffffe - m;
    if (!ok && kw == 0 && lane == 0) record_error(ctx, DEVERR_INDEX);
    const unsigned p = ok ? (unsigned)(sp + m) : 0u;  // absolute position
    const int base = (int)((p + 1u) % (unsigned)win);
    const long long first_t = (long long)p - win + 1;  // token of window slot 0
    // compressed rows visible at p: 0 .. p / ratio; the most recent K - win of them
    const int visible = ratio > 0 ? (int)(p / (unsigned)ratio) + 1 : 0;
    const int room = K - win;
    const int first_c = visible > room ? visible - room : 0;
    const int ncomp = visible - first_c;
    int32_t *dst = out + (long long)row * K;
#pragma unroll
    for (int j = 0; j < GROUPS; ++j) {
        const int k0 = kw + 4 * (lane + 32 * j);
        int v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k = k0 + e;
            int x = -1;
            if (ok) {
                if (k < win) {
                    if (first_t + k >= 0) x = base + k < win ? base + k : base + k - win;
                } else if (k - win < ncomp) {
                    x = win + first_c + (k - win);
                }
            }
            v[e] = x;
        }
        if ((K & 3) == 0) {
            if (k0 < K) *reinterpret_cast<int4 *>(dst + k0) = make_int4(v[0], v[1], v[2], v[3]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (k0 + e < K) dst[k0 + e] = v[e];
        }
    }
}

// One thread per 16-byte unit of the rows written: row i of the last
// min(S, win) new rows of request b goes to ring row (start_pos[b] + S - n + i) % win.
__global__ void ring_write_kernel(uint8_t *__restrict__ cache, const uint8_t *__restrict__ src,
                                  const int32_t *__restrict__ start_pos, int S, int N, int n,
                                  int win, int row_bytes, long long total16, DevCtx ctx) {
    const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= total16) return;
    const int units = row_bytes / 16;
    const long long r = g / units;  // (b, i)
    const int u = (int)(g % units);
    const int b = (int)(r / n), i = (int)(r % n);
    const int sp = __ldg(start_pos + b);
    if (sp < 0) {  // positions start at 0: nothing is written, the error is reported
        if (i == 0 && u == 0) record_error(ctx, DEVERR_INDEX);
        return;
    }
    const long long pos = (long long)sp + (S - n) + i;
    const int slot = (int)(pos % win);
    const uint4 val =
        *reinterpret_cast<const uint4 *>(src + ((long long)b * S + (S - n) + i) * row_bytes + u * 16);
    *reinterpret_cast<uint4 *>(cache + ((long long)b * N + slot) * row_bytes + u * 16) = val;
}

}  // namespace

cudaError_t launch_topk_idxs(int32_t *out, const int32_t *start_pos, int B, int M, int K, int win,
                             int ratio, const DevInfo &dev, cudaStream_t s) {
    const int warps_per_row = (K + SPAN - 1) / SPAN;
    const long long total = (long long)B * M * warps_per_row * 32;
    if (total == 0) return cudaSuccess;
    if (total > 0x7fffffffLL - 256) return cudaErrorInvalidValue;  // 32-bit thread index
    const int threads = 256;
    const int blocks = (int)((total + threads - 1) / threads);
    const DevCtx ctx = make_ctx(dev);
    topk_idxs_kernel<<<blocks, threads, 0, s>>>(out, start_pos, M, K, win, ratio, warps_per_row,
                                                (int)total, ctx);
    return cudaGetLastError();
}

cudaError_t launch_kv_ring_write(void *cache, const void *src, const int32_t *start_pos, int B,
                                 int S, int N, int d, int win, int elem_bytes, const DevInfo &dev,
                                 cudaStream_t s) {
    const int n = S < win ? S : win;
    const int row_bytes = d * elem_bytes;
    const long long total16 = (long long)B * n * (row_bytes / 16);
    if (total16 == 0) return cudaSuccess;
    const int threads = 256;
    const long long blocks = (total16 + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const DevCtx ctx = make_ctx(dev);
    ring_write_kernel<<<(unsigned)blocks, threads, 0, s>>>(
        static_cast<uint8_t *>(cache), static_cast<const uint8_t *>(src), start_pos, S, N, n, win,
        row_bytes, total16, ctx);
    return cudaGetLastError();
}

}  // namespace sattn
