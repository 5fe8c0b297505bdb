// SIMT kernels: one warp per attention row (query token, head).
//
// These serve every dtype and head size in {64, 128}: the fp32 window path
// (vLLM PR #49815 report, the 5/37-token window-8 test), and the fp32 forms of
// the gathered and block-sparse paths. Each lane holds d/32 elements of the
// query and of the output accumulator; the row walks its key set in order
// with an online softmax in the log2 domain:
//   s = <q, k> * scale * log2(e)           (+ sink*log2(e) on key 0, key-0 mode)
//   m' = max(m, s), l = l*2^(m-m') + 2^(s-m'), acc = acc*2^(m-m') + 2^(s-m') v
// Null-logit sinks start from m = sink*log2(e), l = 1 ("PR #49815 report",
// `_fwd_kernel` listing, USE_SINKS); key-0 mode and no sinks start empty.
// The LSE merge kernel ("XAttention Offload Stream Synchronization Fix",
// three-stage KV chunking) is here as well.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace sattn {
namespace {

constexpr int kWarps = 4;

template <typename T, int D> struct RowAcc {
    static constexpr int E = D / 32;
    float acc[E];
    float m, l;

    __device__ void init(bool null_sink, float sink_l2) {
        m = null_sink ? sink_l2 : -INFINITY;
        l = null_sink ? 1.0f : 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.0f;
    }

    // s: logit already in log2 units.
    __device__ void add(float s, const T *vrow, int lane) {
        float mn = fmaxf(m, s);
        float alpha = (m == -INFINITY) ? 0.0f : ex2(m - mn);
        float p = ex2(s - mn);
        l = l * alpha + p;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = acc[e] * alpha + p * to_f32(vrow[lane + 32 * e]);
        m = mn;
    }

    template <typename TO>
    __device__ void store(TO *orow, float *lse_out, int lane) const {
        float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) orow[lane + 32 * e] = from_f32<TO>(acc[e] * inv);
        if (lse_out && lane == 0) *lse_out = l > 0.0f ? (m + log2f(l)) * LN2 : -INFINITY;
    }
};

template <typename T, int D>
__device__ __forceinline__ float dot_row(const float (&qv)[D / 32], const T *krow, int lane) {
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) s += qv[e] * to_f32(krow[lane + 32 * e]);
    return warp_sum(s);
}

// --------------------------------------------------------------- window

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) window_simt_kernel(WindowArgs a, DevCtx ctx) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (row >= (int64_t)a.T * a.H) return;
    const int t = (int)(row / a.H), h = (int)(row % a.H);
    const int g = h / (a.H / a.Hkv);
    // sequence containing token t: last s with cu[s] <= t
    int lo = 0, hi = a.num_seqs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(a.cu_seqlens + mid) <= t) lo = mid; else hi = mid - 1;
    }
    const int start = __ldg(a.cu_seqlens + lo), end = __ldg(a.cu_seqlens + lo + 1);
    T *orow = static_cast<T *>(a.o) + row * D;
    float *lse_out = a.lse ? a.lse + row : nullptr;
    RowAcc<T, D> r;
    const float sink_l2 = a.sinks ? __ldg(a.sinks + h) * LOG2E : 0.0f;
    r.init(a.sink_mode == 2, sink_l2);
    if (!(start <= t && t < end && end <= a.T && __ldg(a.cu_seqlens) == 0)) {
        if (lane == 0) record_error(ctx, DEVERR_SEQLENS);
        r.init(false, 0.0f);
        r.template store<T>(orow, lse_out, lane);
        return;
    }
    const int L = end - start, i = t - start;
    int jlo = a.wl < 0 ? 0 : max(0, i - a.wl);
    int jhi = a.wr < 0 ? L - 1 : min(L - 1, i + a.wr);
    if (a.causal) jhi = min(jhi, i);
    const float qs = a.scale * LOG2E;
    float qv[D / 32];
    const T *qrow = static_cast<const T *>(a.q) + row * D;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) qv[e] = to_f32(qrow[lane + 32 * e]) * qs;
    const T *kbase = static_cast<const T *>(a.k);
    const T *vbase = static_cast<const T *>(a.v);
    for (int j = jlo; j <= jhi; ++j) {
        const int64_t kr = ((int64_t)(start + j) * a.Hkv + g) * D;
        float s = dot_row<T, D>(qv, kbase + kr, lane);
        if (a.sink_mode == 1 && j == 0) s += sink_l2;
        r.add(s, vbase + kr, lane);
    }
    r.template store<T>(orow, lse_out, lane);
}

// --------------------------------------------------------------- gathered (shared KV head)

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) sparse_simt_kernel(SparseArgs a, DevCtx ctx) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (row >= (int64_t)a.B * a.M * a.H) return;
    const int64_t bm = row / a.H;
    const int h = (int)(row % a.H);
    const int64_t b = bm / a.M;
    const float sink_l2 = a.sinks ? __ldg(a.sinks + h) * LOG2E : 0.0f;
    RowAcc<T, D> r;
    r.init(a.sink_mode == 2, sink_l2);
    const float qs = a.scale * LOG2E;
    float qv[D / 32];
    const T *qrow = static_cast<const T *>(a.q) + row * D;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) qv[e] = to_f32(qrow[lane + 32 * e]) * qs;
    const T *kvb = static_cast<const T *>(a.kv) + b * (int64_t)a.N * D;
    const int32_t *list = a.idx + bm * a.K;
    bool bad = false;
    for (int t0 = 0; t0 < a.K; t0 += 32) {
        const int mine = t0 + lane < a.K ? __ldg(list + t0 + lane) : -1;
        const int cnt = min(32, a.K - t0);
        for (int u = 0; u < cnt; ++u) {
            const int e = __shfl_sync(0xffffffffu, mine, u);
            if (e == -1) continue;
            if (e < -1 || e >= a.N) { bad = true; continue; }
            const T *krow = kvb + (int64_t)e * D;
            float s = dot_row<T, D>(qv, krow, lane);
            if (a.sink_mode == 1 && e == 0) s += sink_l2;
            r.add(s, krow, lane);
        }
    }
    if (bad && lane == 0) record_error(ctx, DEVERR_INDEX);
    r.template store<T>(static_cast<T *>(a.o) + row * D, a.lse ? a.lse + row : nullptr, lane);
}

// --------------------------------------------------------------- block-sparse chunk

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) block_simt_kernel(BlockArgs a, DevCtx ctx) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (row >= (int64_t)a.M * a.H) return;
    const int i = (int)(row / a.H), h = (int)(row % a.H);
    const int g = h / (a.H / a.Hkv);
    const int QB = (a.M + SATTN_BLOCK - 1) / SATTN_BLOCK;
    const int KB = (a.Nctx + SATTN_BLOCK - 1) / SATTN_BLOCK;
    const int64_t pos = (int64_t)a.q_pos0 + i;
    int jend = a.kv_end;
    if (a.causal && pos + 1 < (int64_t)jend) jend = (int)(pos + 1);
    const uint8_t *mrow = a.mask + ((int64_t)h * QB + i / SATTN_BLOCK) * KB;
    RowAcc<T, D> r;
    r.init(false, 0.0f);
    const float qs = a.scale * LOG2E;
    float qv[D / 32];
    const T *qrow = static_cast<const T *>(a.q) + row * D;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) qv[e] = to_f32(qrow[lane + 32 * e]) * qs;
    const T *kb_ = static_cast<const T *>(a.k);
    const T *vb_ = static_cast<const T *>(a.v);
    for (int kb = a.kv_begin / SATTN_BLOCK; kb * SATTN_BLOCK < jend; ++kb) {
        if (!__ldg(mrow + kb)) continue;
        const int j0 = max(a.kv_begin, kb * SATTN_BLOCK);
        const int j1 = min(jend, (kb + 1) * SATTN_BLOCK);
        for (int j = j0; j < j1; ++j) {
            const int64_t kr = ((int64_t)j * a.Hkv + g) * D;
            r.add(dot_row<T, D>(qv, kb_ + kr, lane), vb_ + kr, lane);
        }
    }
    r.template store<float>(a.o_part + row * D, a.lse_part + row, lane);
}

// --------------------------------------------------------------- LSE merge

template <typename TO>
__global__ void __launch_bounds__(kWarps * 32) merge_kernel(MergeArgs a) {
    // When launched as a programmatic dependent, wait until the producing grid
    // has finished and its writes are visible (returns at once otherwise).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (r >= a.R) return;
    const float sink_v = a.sinks ? __ldg(a.sinks + r % a.H) : -INFINITY;
    TO *orow_v = static_cast<TO *>(a.o) + r * a.d;
    if (a.C <= 32 && (a.d & 3) == 0 && a.d <= 128 &&
        (reinterpret_cast<uintptr_t>(a.o_parts) & 15u) == 0) {
        // lane c holds split c's lse (one load); each lane owns four
        // consecutive columns and reads them from every split with one
        // 16-byte load; splits with nothing (lse = -inf) are skipped
        const float lc = lane < a.C ? __ldg(a.lse_parts + (int64_t)lane * a.R + r) : -INFINITY;
        const int col = 4 * lane;
        // up to eight splits: their rows are loaded together with the lse, so
        // the merge waits for one round of loads instead of two
        constexpr int PRE = 8;
        float4 pre[PRE];
        const bool prefetch = a.C <= PRE && col < a.d;
        if (prefetch) {
#pragma unroll
            for (int c = 0; c < PRE; ++c)
                if (c < a.C)
                    pre[c] = __ldg(reinterpret_cast<const float4 *>(
                        a.o_parts + ((int64_t)c * a.R + r) * a.d + col));
        }
        const float m = fmaxf(warp_max(lc), sink_v);
        if (m == -INFINITY) {
            if (col < a.d) {
#pragma unroll
                for (int k = 0; k < 4; ++k) orow_v[col + k] = from_f32<TO>(0.0f);
            }
            if (a.lse && lane == 0) a.lse[r] = -INFINITY;
            return;
        }
        float z = warp_sum(lc == -INFINITY ? 0.f : ex2((lc - m) * LOG2E));
        if (a.sinks) z += ex2((sink_v - m) * LOG2E);
        const float L = m + logf(z);
        const float w = lc == -INFINITY ? 0.f : ex2((lc - L) * LOG2E);
        const unsigned live = __ballot_sync(0xffffffffu, lc != -INFINITY);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (a.C <= PRE) {
#pragma unroll
            for (int c = 0; c < PRE; ++c) {
                if (c >= a.C) break;
                const float wc = __shfl_sync(0xffffffffu, w, c);
                if (!((live >> c) & 1u) || !prefetch) continue;
                acc[0] += wc * pre[c].x;
                acc[1] += wc * pre[c].y;
                acc[2] += wc * pre[c].z;
                acc[3] += wc * pre[c].w;
            }
        }
#pragma unroll 8
        for (int c = 0; c < a.C && a.C > PRE; ++c) {
            const float wc = __shfl_sync(0xffffffffu, w, c);
            if (!((live >> c) & 1u) || col >= a.d) continue;
            const float4 v = __ldg(
                reinterpret_cast<const float4 *>(a.o_parts + ((int64_t)c * a.R + r) * a.d + col));
            acc[0] += wc * v.x;
            acc[1] += wc * v.y;
            acc[2] += wc * v.z;
            acc[3] += wc * v.w;
        }
        if (col < a.d) {
#pragma unroll
            for (int k = 0; k < 4; ++k) orow_v[col + k] = from_f32<TO>(acc[k]);
        }
        if (a.lse && lane == 0) a.lse[r] = L;
        return;
    }
    float m = -INFINITY;
    for (int c = lane; c < a.C; c += 32) m = fmaxf(m, __ldg(a.lse_parts + (int64_t)c * a.R + r));
    m = warp_max(m);
    const float sink = a.sinks ? __ldg(a.sinks + r % a.H) : -INFINITY;
    m = fmaxf(m, sink);
    TO *orow = static_cast<TO *>(a.o) + r * a.d;
    if (m == -INFINITY) {
        for (int e = lane; e < a.d; e += 32) orow[e] = from_f32<TO>(0.0f);
        if (a.lse && lane == 0) a.lse[r] = -INFINITY;
        return;
    }
    float z = 0.0f;
    for (int c = lane; c < a.C; c += 32)
        z += ex2((__ldg(a.lse_parts + (int64_t)c * a.R + r) - m) * LOG2E);
    z = warp_sum(z);
    if (a.sinks) z += ex2((sink - m) * LOG2E);
    const float L = m + logf(z);
    if (a.d <= 128) {
        // up to four columns per lane (lane, lane+32, ...), accumulated over
        // the splits; loads of different splits are independent
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int c = 0; c < a.C; ++c) {
            const float lc = __ldg(a.lse_parts + (int64_t)c * a.R + r);
            if (lc == -INFINITY) continue;  // the same for every lane
            const float w = ex2((lc - L) * LOG2E);
            const float *src = a.o_parts + ((int64_t)c * a.R + r) * a.d;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (lane + 32 * k < a.d) acc[k] += w * __ldg(src + lane + 32 * k);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (lane + 32 * k < a.d) orow[lane + 32 * k] = from_f32<TO>(acc[k]);
    } else {
        for (int e = lane; e < a.d; e += 32) {
            float acc = 0.0f;
            for (int c = 0; c < a.C; ++c) {
                const float lc = __ldg(a.lse_parts + (int64_t)c * a.R + r);
                if (lc == -INFINITY) continue;
                acc += ex2((lc - L) * LOG2E) * __ldg(a.o_parts + ((int64_t)c * a.R + r) * a.d + e);
            }
            orow[e] = from_f32<TO>(acc);
        }
    }
    if (a.lse && lane == 0) a.lse[r] = L;
}

inline dim3 rows_grid(int64_t rows) { return dim3((unsigned)((rows + kWarps - 1) / kWarps)); }

}  // namespace

cudaError_t launch_window_simt(const WindowArgs &a, const DevInfo &dev, cudaStream_t s) {
    const DevCtx ctx = make_ctx(dev);
    dim3 g = rows_grid((int64_t)a.T * a.H), b(kWarps * 32);
    if (a.dtype == SATTN_F32) {
        if (a.d == 64) window_simt_kernel<float, 64><<<g, b, 0, s>>>(a, ctx);
        else window_simt_kernel<float, 128><<<g, b, 0, s>>>(a, ctx);
    } else {
        if (a.d == 64) window_simt_kernel<__nv_bfloat16, 64><<<g, b, 0, s>>>(a, ctx);
        else window_simt_kernel<__nv_bfloat16, 128><<<g, b, 0, s>>>(a, ctx);
    }
    return cudaGetLastError();
}

cudaError_t launch_sparse_simt(const SparseArgs &a, const DevInfo &dev, cudaStream_t s) {
    const DevCtx ctx = make_ctx(dev);
    dim3 g = rows_grid((int64_t)a.B * a.M * a.H), b(kWarps * 32);
    if (a.dtype == SATTN_F32) {
        if (a.d == 64) sparse_simt_kernel<float, 64><<<g, b, 0, s>>>(a, ctx);
        else sparse_simt_kernel<float, 128><<<g, b, 0, s>>>(a, ctx);
    } else {
        if (a.d == 64) sparse_simt_kernel<__nv_bfloat16, 64><<<g, b, 0, s>>>(a, ctx);
        else sparse_simt_kernel<__nv_bfloat16, 128><<<g, b, 0, s>>>(a, ctx);
    }
    return cudaGetLastError();
}

cudaError_t launch_block_simt(const BlockArgs &a, const DevInfo &dev, cudaStream_t s) {
    const DevCtx ctx = make_ctx(dev);
    dim3 g = rows_grid((int64_t)a.M * a.H), b(kWarps * 32);
    if (a.dtype == SATTN_F32) {
        if (a.d == 64) block_simt_kernel<float, 64><<<g, b, 0, s>>>(a, ctx);
        else block_simt_kernel<float, 128><<<g, b, 0, s>>>(a, ctx);
    } else {
        if (a.d == 64) block_simt_kernel<__nv_bfloat16, 64><<<g, b, 0, s>>>(a, ctx);
        else block_simt_kernel<__nv_bfloat16, 128><<<g, b, 0, s>>>(a, ctx);
    }
    return cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs &a, const DevInfo &dev, cudaStream_t s,
                         bool after_primary) {
    (void)dev;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = rows_grid(a.R);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_primary ? 1 : 0;
    if (a.dtype == SATTN_F32) return cudaLaunchKernelEx(&cfg, merge_kernel<float>, a);
    return cudaLaunchKernelEx(&cfg, merge_kernel<__nv_bfloat16>, a);
}

}  // namespace sattn
