// Compressor gated pooling ("DeepSeek-V4 CSA/HCA walkthrough", sections 5.1
// and 5.2): every `ratio` consecutive tokens become one compressed KV row,
// out[w, j] = sum_e kv_e[j] * softmax_e(score_e[j] + ape_e[j]) over the
// window's entries e (with overlap also the previous window's tokens, on the
// first d columns of the projections).
//
// Pure streaming: every kv / score element is read once, each row written
// once. One thread owns four consecutive columns of one window (a warp covers
// 128 columns of a token row with 16-byte loads, fully coalesced) and runs an
// online softmax over the window's entries in the log2 domain, so nothing is
// staged.
#include "common.cuh"
#include "internal.h"

namespace sattn {
namespace {

template <typename T> struct Vec4;
template <> struct Vec4<float> {
    __device__ static void load(const float *p, float (&v)[4]) {
        const float4 x = __ldg(reinterpret_cast<const float4 *>(p));
        v[0] = x.x;
        v[1] = x.y;
        v[2] = x.z;
        v[3] = x.w;
    }
    __device__ static void store(float *p, const float (&v)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <> struct Vec4<__nv_bfloat16> {
    __device__ static void load(const __nv_bfloat16 *p, float (&v)[4]) {
        const uint2 x = __ldg(reinterpret_cast<const uint2 *>(p));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.y));
        v[0] = a.x;
        v[1] = a.y;
        v[2] = b.x;
        v[3] = b.y;
    }
    __device__ static void store(__nv_bfloat16 *p, const float (&v)[4]) {
        uint2 x;
        x.x = pack_bf16x2(v[0], v[1]);
        x.y = pack_bf16x2(v[2], v[3]);
        *reinterpret_cast<uint2 *>(p) = x;
    }
};

struct Online4 {
    float m[4], l[4], acc[4];
    __device__ Online4() {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            m[c] = -INFINITY;
            l[c] = 0.f;
            acc[c] = 0.f;
        }
    }
    // one entry: scores in log2 units, values
    __device__ void add(const float (&s2)[4], const float (&v)[4]) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (s2[c] > m[c]) {  // the first entry always lands here (m = -inf)
                const float a = ex2(m[c] - s2[c]);
                l[c] *= a;
                acc[c] *= a;
                m[c] = s2[c];
            }
            const float p = ex2(s2[c] - m[c]);
            l[c] += p;
            acc[c] = fmaf(p, v[c], acc[c]);
        }
    }
};

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) compress_kernel(const Tin *__restrict__ kv,
                                                       const Tin *__restrict__ score,
                                                       const float *__restrict__ ape,
                                                       Tout *__restrict__ out, long long out_bstride,
                                                       int S, int d, int ratio, int coff, int nwin,
                                                       long long total) {
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (tid >= total) return;
    const int qd = d >> 2;  // threads per window
    const long long win = tid / qd;
    const int j0 = (int)(tid - win * qd) * 4;
    const int b = (int)(win / nwin), w = (int)(win - (long long)b * nwin);
    const size_t W = (size_t)coff * d;  // projection width
    const Tin *kvb = kv + (size_t)b * S * W;
    const Tin *scb = score + (size_t)b * S * W;
    Online4 st;
    auto entries = [&](int t0, int c) {  // tokens t0 .. t0 + ratio - 1, columns c .. c + 3
#pragma unroll 4
        for (int i = 0; i < ratio; ++i) {
            const size_t off = (size_t)(t0 + i) * W + c;
            float v[4], s[4];
            Vec4<Tin>::load(kvb + off, v);
            Vec4<Tin>::load(scb + off, s);
            const float4 a = __ldg(reinterpret_cast<const float4 *>(ape + (size_t)i * W + c));
            float s2[4] = {(s[0] + a.x) * LOG2E, (s[1] + a.y) * LOG2E, (s[2] + a.z) * LOG2E,
                           (s[3] + a.w) * LOG2E};
            st.add(s2, v);
        }
    };
    // overlap: the previous window's tokens on the first d columns
    if (coff == 2 && w > 0) entries((w - 1) * ratio, j0);
    entries(w * ratio, (coff - 1) * d + j0);
    float o[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) o[c] = st.acc[c] / st.l[c];
    Vec4<Tout>::store(out + (size_t)b * out_bstride + (size_t)w * d + j0, o);
}

template <typename Tin, typename Tout>
cudaError_t launch_typed(const CompressArgs &a, cudaStream_t s) {
    const int nwin = a.S / a.ratio;
    const long long total = (long long)a.B * nwin * (a.d / 4);
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    compress_kernel<Tin, Tout><<<(unsigned)blocks, threads, 0, s>>>(
        static_cast<const Tin *>(a.kv), static_cast<const Tin *>(a.score), a.ape,
        static_cast<Tout *>(a.out), a.out_batch_stride, a.S, a.d, a.ratio, a.overlap ? 2 : 1, nwin,
        total);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compress_kv(const CompressArgs &a, const DevInfo &, cudaStream_t s) {
    const bool in_bf = a.in_dtype == SATTN_BF16, out_bf = a.out_dtype == SATTN_BF16;
    if (in_bf) {
        return out_bf ? launch_typed<__nv_bfloat16, __nv_bfloat16>(a, s)
                      : launch_typed<__nv_bfloat16, float>(a, s);
    }
    return out_bf ? launch_typed<float, __nv_bfloat16>(a, s) : launch_typed<float, float>(a, s);
}

}  // namespace sattn
