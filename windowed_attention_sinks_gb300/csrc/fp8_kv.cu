// FP8 KV rows ("DeepSeek-V4 CSA/HCA walkthrough", section 2.3 step 4 and
// section 5.3: the non-RoPE part of a KV row is quantised to FP8, the RoPE
// part keeps a wider type). Layout: the first d - rd columns as e4m3 codes
// with one fp32 scale per row (amax / 448, 1 for an all-zero part; code =
// e4m3(x / scale), nearest even, saturating), the last rd columns as bf16.
//
// One warp per row; a lane holds four consecutive columns, so the row's
// amax is a warp max and every store is a 4-code or 4-value vector.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace sattn {
namespace {

template <typename T>
__device__ __forceinline__ void load4(const T *p, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float *p, float (&v)[4]) {
    const float4 x = __ldg(reinterpret_cast<const float4 *>(p));
    v[0] = x.x;
    v[1] = x.y;
    v[2] = x.z;
    v[3] = x.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16 *p, float (&v)[4]) {
    const uint2 x = __ldg(reinterpret_cast<const uint2 *>(p));
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.y));
    v[0] = a.x;
    v[1] = a.y;
    v[2] = b.x;
    v[3] = b.y;
}

template <typename T>
__global__ void __launch_bounds__(256)
quantize_kernel(const T *__restrict__ kv, uint8_t *__restrict__ nope, __nv_bfloat16 *__restrict__ rope,
                float *__restrict__ row_scale, long long rows, int d, int rd) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;  // whole warps leave together
    const int lane = threadIdx.x & 31;
    const int dn = d - rd;
    const T *src = kv + row * d;
    // amax of the non-RoPE part
    float amax = 0.f;
    for (int c = lane * 4; c < dn; c += 128) {
        float v[4];
        load4(src + c, v);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
    }
    amax = warp_max(amax);
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    if (lane == 0) row_scale[row] = s;
    for (int c = lane * 4; c < dn; c += 128) {
        float v[4];
        load4(src + c, v);
        uint32_t packed = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __nv_fp8_storage_t code =
                __nv_cvt_float_to_fp8(__fdiv_rn(v[k], s), __NV_SATFINITE, __NV_E4M3);
            packed |= (uint32_t)code << (8 * k);
        }
        *reinterpret_cast<uint32_t *>(nope + row * dn + c) = packed;
    }
    for (int c = lane * 4; c < rd; c += 128) {
        float v[4];
        load4(src + dn + c, v);
        uint2 x;
        x.x = pack_bf16x2(v[0], v[1]);
        x.y = pack_bf16x2(v[2], v[3]);
        *reinterpret_cast<uint2 *>(rope + row * rd + c) = x;
    }
}

}  // namespace

cudaError_t launch_quantize_kv_fp8(const void *kv, uint8_t *nope, void *rope, float *row_scale,
                                   long long rows, int d, int rd, int dtype, const DevInfo &,
                                   cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    auto *r = static_cast<__nv_bfloat16 *>(rope);
    if (dtype == SATTN_BF16)
        quantize_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(kv), nope, r, row_scale, rows, d, rd);
    else
        quantize_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const float *>(kv), nope,
                                                                 r, row_scale, rows, d, rd);
    return cudaGetLastError();
}

}  // namespace sattn
