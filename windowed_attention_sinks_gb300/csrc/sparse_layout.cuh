// Shared-memory layout of the gathered attention kernels ("DeepSeek-V4
// CSA/HCA walkthrough", sections 4.2-4.3: index-gathered KV rows staged in
// shared memory so that Q K^T and P V become dense contractions), and the
// tcgen05 descriptors that read it. One KV head is shared by NH = 32 query
// heads; rows are HD = 128 bf16 values (256 bytes).
//
// With R = 128 gathered rows per tile the operand roles are swapped so that
// the rows fill the 128-row MMA:
//   S^T [R x NH]  = KV [R x HD] . Q^T        A = KV tile (K-major), B = Q
//   O^T [HD x NH] += KV^T [HD x R] . P^T     A = the same tile (MN-major), B = P
// KV tile: two 64-column halves of R rows x 128 bytes, 128B-swizzled.
// Q and P: [NH rows x 128 columns] bf16 K-major, two 64-column halves of
// QP_HALF bytes each, 128B-swizzled.
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace sattn {
namespace gather {

constexpr int R = 128;   // gathered rows per tile
constexpr int HD = 128;  // head dim
constexpr int NH = 32;   // query heads sharing the KV head
constexpr uint32_t KV_TILE = R * HD * 2;   // 32 KB
constexpr uint32_t KV_HALF = KV_TILE / 2;  // 64 columns of d
constexpr uint32_t QP_HALF = NH * 128;     // 4 KB: one 64-column half of Q or P
// Per-warp transpose buffer: head h, key i of the warp at h * TB_STRIDE + i.
// Writes (one head, 32 keys) are consecutive; the 16-byte reads of the 8
// lanes sharing an LDS.128 phase fall in distinct bank groups (9h + k mod 8).
constexpr int TB_STRIDE = 36;
// Copy warps per tile: warp g copies rows 32 g .. 32 g + 31.
constexpr int COPY_WARPS = 4;
constexpr int PAIRS = R / 2 / COPY_WARPS;  // row pairs per copy warp (multiple of 4)

constexpr uint32_t IDESC_S = idesc_bf16_f32(128, NH, 0, 0);
constexpr uint32_t IDESC_O = idesc_bf16_f32(128, NH, 1, 0);

// Shared-memory descriptors are built once per buffer; the K step kk (16
// elements) only moves the start address, whose field holds address >> 4 in
// the low bits (no carry: shared addresses stay below 256 KB).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t base, uint32_t lbo) {
    return smem_desc_sw128(base, lbo, 1024u);
}
// K-major operand split in 64-element halves `half_stride` bytes apart
__host__ __device__ constexpr uint32_t koff(int kk, uint32_t half_stride) {
    return ((uint32_t)(kk >> 2) * half_stride + (uint32_t)(kk & 3) * 32u) >> 4;
}
// MN-major operand: 16 K rows of 128 bytes per step
__host__ __device__ constexpr uint32_t mnoff(int kk) { return (uint32_t)kk * 2048u >> 4; }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (counts as one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Copy warp g of a tile copies rows 2i + hi, i in [PAIRS g, PAIRS (g+1)).
// Lane = (hi, unit) copies 16-byte unit `unit` of rows 2i + hi. In the 128B
// swizzle, unit u of row r sits at r * 128 + ((u ^ (r & 7)) << 4), and
// (unit & 7) ^ (r & 7) = ((unit & 7) ^ hi) ^ (2i & 6): four lane offsets
// cover every i. Entries that are not valid rows (-1) are zero-filled so
// that P V stays finite.
struct RowCopier {
    uint32_t dofs[4];
    int hi, unit;
    __device__ explicit RowCopier(int lane) {
        hi = lane >> 4;
        unit = lane & 15;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            dofs[c] = (uint32_t)(unit >> 3) * KV_HALF + (uint32_t)hi * 128u +
                      ((((uint32_t)(unit & 7) ^ (uint32_t)hi) ^ (uint32_t)(2 * c)) << 4);
    }
    // entries of the tile's rows read from shared memory (ids[row], -1 = none)
    __device__ void issue(uint32_t kv_s, const int *ids, const __nv_bfloat16 *rows, int g) const {
        const __nv_bfloat16 *src0 = rows + unit * 8;
#pragma unroll
        for (int i2 = 0; i2 < PAIRS; ++i2) {
            const int i = PAIRS * g + i2;
            const int e = ids[2 * i + hi];
            cp_async16(kv_s + dofs[i2 & 3] + (uint32_t)i * 256u,
                       src0 + (size_t)(e >= 0 ? e : 0) * HD, e >= 0 ? 16u : 0u);
        }
    }
    // the same with the warp's 32 entries held one per lane: lane l has the
    // entry of row 32 g + l (any negative value = none)
    __device__ void issue_lanes(uint32_t kv_s, int e_lane, const __nv_bfloat16 *rows, int g) const {
        const __nv_bfloat16 *src0 = rows + unit * 8;
#pragma unroll
        for (int i2 = 0; i2 < PAIRS; ++i2) {
            const int i = PAIRS * g + i2;
            const int e = __shfl_sync(0xffffffffu, e_lane, 2 * i2 + hi);
            cp_async16(kv_s + dofs[i2 & 3] + (uint32_t)i * 256u,
                       src0 + (size_t)(e >= 0 ? e : 0) * HD, e >= 0 ? 16u : 0u);
        }
    }
};

// FP8 cache rows: the RoPE part (bf16, the stage's second 64-column half) is
// copied by cp.async like the bf16 rows; the DN e4m3 codes are loaded to
// registers before the stage is free, then dequantised (code value x row
// scale, rounded to bf16) and stored into the first half with the same 128B
// swizzle.
constexpr int DN = HD / 2;  // non-RoPE columns

struct Fp8Copier {
    uint32_t rope_dofs[2];
    int rsub, ru, rn, cu;
    // RoPE: lane = (rsub, ru) copies unit ru of rows 4k + rsub (four rows per
    // instruction); codes: lane = (rn, cu) handles codes 16 cu .. 16 cu + 15 of
    // rows 8k + rn. A warp's rows start at a multiple of 8, so the swizzle
    // term of row 4k + rsub is rsub | 4 (k & 1), that of row 8k + rn is rn.
    __device__ explicit Fp8Copier(int lane) {
        rsub = lane >> 3;
        ru = lane & 7;
        rn = lane >> 2;
        cu = lane & 3;
#pragma unroll
        for (int j = 0; j < 2; ++j)
            rope_dofs[j] = KV_HALF + (uint32_t)rsub * 128u +
                           (((uint32_t)ru ^ ((uint32_t)rsub | (4u * j))) << 4);
    }
    // codes and scales of this warp's rows (32 g .. 32 g + 31) to registers
    __device__ void load_codes(const int *ids, const uint8_t *nope, const float *scl, int g,
                               uint4 (&q)[4], float (&sc)[4]) const {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int e = ids[32 * g + 8 * k + rn];
            if (e >= 0) {
                q[k] = __ldg(reinterpret_cast<const uint4 *>(nope + (size_t)e * DN) + cu);
                sc[k] = __ldg(scl + e);
            } else {  // -1 entry: a zero row keeps P V finite
                q[k] = make_uint4(0u, 0u, 0u, 0u);
                sc[k] = 0.f;
            }
        }
    }
    __device__ void issue_rope(uint32_t kv_s, const int *ids, const __nv_bfloat16 *rope,
                               int g) const {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int e = ids[32 * g + 4 * k + rsub];
            cp_async16(kv_s + (uint32_t)(32 * g + 4 * k) * 128u + rope_dofs[k & 1],
                       rope + (size_t)(e >= 0 ? e : 0) * (HD - DN) + ru * 8, e >= 0 ? 16u : 0u);
        }
    }
    // codes -> bf16 (e4m3 value x scale, rounded to nearest even) into the
    // stage's first half
    __device__ void store_codes(uint32_t kv_s, int g, const uint4 (&q)[4],
                                const float (&sc)[4]) const {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t w[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const __nv_fp8x2_storage_t two =
                        (__nv_fp8x2_storage_t)((w[i] >> (16 * hh)) & 0xffffu);
                    const __half2 h2 = __half2(__nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3));
                    const float2 f = __half22float2(h2);
                    o[2 * i + hh] = pack_bf16x2(f.x * sc[k], f.y * sc[k]);
                }
            }
            const uint32_t row = kv_s + (uint32_t)(32 * g + 8 * k + rn) * 128u;
            const uint32_t a0 = row + ((((uint32_t)(2 * cu)) ^ (uint32_t)rn) << 4);
            const uint32_t a1 = row + ((((uint32_t)(2 * cu + 1)) ^ (uint32_t)rn) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "r"(o[0]),
                         "r"(o[1]), "r"(o[2]), "r"(o[3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a1), "r"(o[4]),
                         "r"(o[5]), "r"(o[6]), "r"(o[7])
                         : "memory");
        }
    }
};

}  // namespace gather
}  // namespace sattn
