// XAttention block selection ("XAttention Offload Stream Synchronization
// Fix", technical details): stage 1 computes per-chunk softmax stats (m, l) of
// every query row, stage 2 merges them, stage 3 sums the normalised
// probabilities exp(s - m) / l over 128 x 128 blocks, step 4 selects, per
// query block, the shortest run of key blocks by descending mass that reaches
// threshold x the total. The estimate is the exact softmax at full
// resolution.
//
// Stages 1 and 3 are one tcgen05 kernel (MODE 1 / MODE 3): a CTA owns one
// (query block of 128 rows, head); a producer warp loads the Q tile once and
// the key tiles of the chunk into a 3-stage ring (2-D boxes of a 3-D tensor
// map, 128B swizzle); one thread issues S = Q K^T (M = N = 128, K = 128 in
// eight K = 16 steps) into a double-buffered TMEM accumulator; four warps, one
// per TMEM lane quarter, own one query row per thread and reduce its 128
// scores in the log2 domain. The exponentials (one MUFU ex2 per score) bound
// the kernel, not the tensor pipe.
#include <math.h>
#include <stdio.h>

#include "common.cuh"
#include "internal.h"

namespace sattn {
namespace {

constexpr int BM = 128;  // query rows per CTA
constexpr int BN = 128;  // keys per tile (= the block size)
constexpr int HD = 128;
constexpr int KST = 2;   // key-tile stages (two CTAs fit on an SM)
constexpr int NRED = 8;  // reduction warps: two per TMEM lane quarter, 64 columns each
constexpr int NTHREADS = 32 * (2 + NRED);  // producer, MMA, reduction warps
constexpr uint32_t TILE = BM * HD * 2;  // 32 KB
constexpr uint32_t HALF = TILE / 2;     // one 64-column half
constexpr int PART = 256;  // tiles whose block partials are kept before a flush

struct Bars {
    uint64_t q_full, k_full[KST], k_empty[KST], s_full[2], s_empty[2], drain;
};

struct alignas(1024) Smem {
    uint8_t q[TILE];
    uint8_t k[KST][TILE];
    float part[NRED][PART];  // MODE 3: per reduction warp, per tile: its rows' mass
    Bars b;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Smem) <= 227 * 1024, "shared memory of one CTA");

struct XParams {
    int M, Nctx, H, Hkv, q_pos0, kv_begin, kv_end, causal;
    float scale_l2;      // scale * log2(e)
    float *m, *l;        // MODE 1: written; MODE 3: the merged stats
    float *block_sum;    // MODE 3: [H, QB, KB]
    int QB, KB;
};

constexpr uint32_t IDESC = idesc_bf16_f32(128, 128, 0, 0);

__host__ __device__ constexpr uint32_t koff(int kk) {
    return ((uint32_t)(kk >> 2) * HALF + (uint32_t)(kk & 3) * 32u) >> 4;
}

// key tiles of a CTA: [kb_lo, kb_hi)
struct Range {
    int kb_lo, kb_hi;
};
__device__ __forceinline__ Range tile_range(const XParams &p, int qb) {
    Range r;
    r.kb_lo = p.kv_begin / BN;
    int hi = (p.kv_end + BN - 1) / BN;
    if (p.causal) {
        const int i_last = min(p.M, (qb + 1) * BM) - 1;
        const int j_last = p.q_pos0 + i_last;  // the last key any row of the block sees
        hi = min(hi, j_last / BN + 1);
    }
    r.kb_hi = max(hi, r.kb_lo);
    return r;
}

__device__ __forceinline__ bool wait_warp(uint64_t &bar, uint32_t parity, const DevCtx &ctx,
                                          volatile int *abort) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(smem_u32(&bar), parity, ctx, abort) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
}

__device__ void producer(const XParams &p, Smem &sm, const CUtensorMap *tq, const CUtensorMap *tk,
                         int qb, int h, Range rg, const DevCtx &ctx) {
    Bars &b = sm.b;
    const int lane = threadIdx.x & 31;
    const int g = h / (p.H / p.Hkv);
    if (lane == 0) {
        prefetch_tmap(tq);
        prefetch_tmap(tk);
        mbar_arrive_expect_tx(smem_u32(&b.q_full), TILE);
        tma_load_3d(smem_u32(sm.q), tq, smem_u32(&b.q_full), 0, h, qb * BM);
        tma_load_3d(smem_u32(sm.q) + HALF, tq, smem_u32(&b.q_full), 64, h, qb * BM);
    }
    int t = 0;
    for (int kb = rg.kb_lo; kb < rg.kb_hi; ++kb, ++t) {
        const int st = t % KST, use = t / KST;
        if (use >= 1 && !wait_warp(b.k_empty[st], (use - 1) & 1, ctx, &sm.abort)) break;
        if (lane == 0) {
            const uint32_t bar = smem_u32(&b.k_full[st]);
            mbar_arrive_expect_tx(bar, TILE);
            tma_load_3d(smem_u32(sm.k[st]), tk, bar, 0, g, kb * BN);
            tma_load_3d(smem_u32(sm.k[st]) + HALF, tk, bar, 64, g, kb * BN);
        }
    }
    // the loads in flight land before the CTA may leave (matters after an abort)
    if (lane == 0) {
        int zero = 0;
        mbar_wait(smem_u32(&b.q_full), 0, ctx, &zero);
        for (int u = t > KST ? t - KST : 0; u < t; ++u)
            mbar_wait(smem_u32(&b.k_full[u % KST]), (u / KST) & 1, ctx, &zero);
    }
    __syncwarp();
}

// one thread: S of every tile in order
__device__ void mma_issue(Smem &sm, uint32_t tmem, int ntiles, const DevCtx &ctx) {
    Bars &b = sm.b;
    volatile int *abort = &sm.abort;
    const uint64_t dq = smem_desc_sw128(smem_u32(sm.q), 16u, 1024u);
    const uint64_t dk0 = smem_desc_sw128(smem_u32(sm.k[0]), 16u, 1024u);
    if (!mbar_wait(smem_u32(&b.q_full), 0, ctx, abort)) return;
    for (int t = 0; t < ntiles; ++t) {
        const int st = t % KST, sb = t & 1;
        if (!mbar_wait(smem_u32(&b.k_full[st]), (t / KST) & 1, ctx, abort)) return;
        if (t >= 2 && !mbar_wait(smem_u32(&b.s_empty[sb]), ((t >> 1) - 1) & 1, ctx, abort)) return;
        tc_fence_after();
        const uint64_t dk = dk0 + (uint64_t)(st * (TILE >> 4));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
            tc_mma_f16(tmem + 128u * (uint32_t)sb, dq + koff(kk), dk + koff(kk), IDESC,
                       kk > 0 ? 1u : 0u);
        tc_commit(smem_u32(&b.s_full[sb]));
        tc_commit(smem_u32(&b.k_empty[st]));
    }
}

__device__ void mma_thread(Smem &sm, uint32_t tmem, int ntiles, const DevCtx &ctx) {
    mma_issue(sm, tmem, ntiles, ctx);
    // every MMA issued completes before TMEM is released (also after an abort)
    tc_commit(smem_u32(&sm.b.drain));
    int zero = 0;
    mbar_wait(smem_u32(&sm.b.drain), 0, ctx, &zero);
}

// Named barrier over the reduction threads, OR-reducing a predicate.
__device__ __forceinline__ int red_bar_or(int pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.s32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred), "r"(32 * NRED)
        : "memory");
    return r;
}

// A query row (TMEM lane) per thread and half-tile: warp w handles lane
// quarter w % 4 and columns 64 (w / 4) .. +63 of each S tile. MODE 1: online
// (max, sum of exp) of the row's visible scores, the two halves merged at the
// end through shared memory; MODE 3: the row's mass exp(s - m) / l per tile,
// summed over the warp's 32 rows, then over the eight warps per key block.
template <int MODE>
__device__ void reduce_rows(const XParams &p, Smem &sm, uint32_t tmem, int qb, int h, Range rg,
                            const DevCtx &ctx) {
    Bars &b = sm.b;
    volatile int *abort = &sm.abort;
    const int lane = threadIdx.x & 31, quarter = (threadIdx.x >> 5) & 3;
    const int rw = (threadIdx.x >> 5) - 2;  // reduction warp 0 .. NRED-1
    const int half = rw >> 2;               // column half of the tiles
    const int rt = quarter * 32 + lane;     // row within the tile = TMEM lane
    const int i = qb * BM + rt;
    const bool row_ok = i < p.M;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    // last key the row may see
    const int jmax = p.causal ? min(p.kv_end - 1, p.q_pos0 + i) : p.kv_end - 1;
    const size_t st_idx = (size_t)(row_ok ? i : 0) * p.H + h;
    float neg_lse2 = 0.f;
    bool has_mass = false;
    if (MODE == 3 && row_ok) {
        const float m = p.m[st_idx], l = p.l[st_idx];
        has_mass = l > 0.f && m != -INFINITY;
        neg_lse2 = has_mass ? -(m * LOG2E + log2f(l)) : 0.f;
    }
    const uint64_t c2 = f2_pack(p.scale_l2, p.scale_l2);
    float m2 = -INFINITY, lsum = 0.f;
    const int ntiles = rg.kb_hi - rg.kb_lo;
    bool failed = false;
    int batch0 = 0;  // first tile of the current partial batch
    for (int t = 0; t < ntiles; ++t) {
        const int sb = t & 1, kb = rg.kb_lo + t, j0 = kb * BN;
        if (!failed)
            failed = !wait_warp(b.s_full[sb], (t >> 1) & 1, ctx, abort);
        float rowsum = 0.f;
        if (!failed) {
            tc_fence_after();
            uint32_t v[2][32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
                tmem_ld32(tmem + 128u * sb + 64u * half + 32u * cc + lane_off, v[cc]);
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&b.s_empty[sb]));
            // visible columns of this row within the warp's half: [clo, chi]
            const int jh = j0 + 64 * half;
            const int clo = max(0, p.kv_begin - jh), chi = min(63, jmax - jh);
            const bool any = row_ok && chi >= clo && (MODE == 1 || has_mass);
            if (any) {
                if (clo != 0 || chi != 63) {
                    // a boundary tile: invisible scores become -inf once, so
                    // that the loops below need no tests (ex2(-inf) = 0)
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int c = 32 * cc + e;
                            if (c < clo || c > chi) v[cc][e] = 0xff800000u;
                        }
                }
                if (MODE == 1) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                        for (int e = 0; e < 32; e += 2)
                            mx = max3(mx, __uint_as_float(v[cc][e]), __uint_as_float(v[cc][e + 1]));
                    const float mnew = fmaxf(m2, mx * p.scale_l2);  // scale > 0
                    if (mnew > m2) {
                        lsum *= ex2(m2 - mnew);  // ex2(-inf) = 0 on the first tile
                        m2 = mnew;
                    }
                }
                const float off = MODE == 1 ? -m2 : neg_lse2;
                const uint64_t off2 = f2_pack(off, off);
                uint64_t acc_a = f2_pack(0.f, 0.f), acc_b = acc_a;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(v[cc][e]),
                                                 __uint_as_float(v[cc][e + 1])),
                                         c2, off2),
                                  x0, x1);
                        const uint64_t e2 = f2_pack(ex2(x0), ex2(x1));
                        if (e & 2) acc_b = f2_add(acc_b, e2);
                        else acc_a = f2_add(acc_a, e2);
                    }
                float s0, s1;
                f2_unpack(f2_add(acc_a, acc_b), s0, s1);
                rowsum = s0 + s1;
                if (MODE == 1) lsum += rowsum;
            }
        } else {
            __syncwarp();
        }
        if (MODE == 3) {
            float w = rowsum;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
            if (lane == 0) sm.part[rw][t - batch0] = w;
            if (t - batch0 == PART - 1 || t == ntiles - 1) {
                // every warp reaches this at the same t: the flush is uniform
                if (red_bar_or(failed)) failed = true;
                if (!failed) {
                    for (int tt = rw * 32 + lane; tt <= t - batch0; tt += 32 * NRED) {
                        float s = 0.f;
#pragma unroll
                        for (int w2 = 0; w2 < NRED; ++w2) s += sm.part[w2][tt];
                        p.block_sum[((size_t)h * p.QB + qb) * p.KB + rg.kb_lo + batch0 + tt] = s;
                    }
                }
                red_bar_or(0);  // the partials are read before the next batch writes them
                batch0 = t + 1;
            }
        }
    }
    if (MODE == 1) {
        // the two column halves of each row: half 1 hands (m, l) to half 0
        // (the partial-sum area is free in this mode)
        float *xm = &sm.part[0][0], *xl = &sm.part[2][0];
        if (half == 1) {
            xm[rt] = m2;
            xl[rt] = lsum;
        }
        red_bar_or(0);
        if (half == 0 && row_ok) {
            const float mo = xm[rt], lo = xl[rt];
            const float mn = fmaxf(m2, mo);
            float l = 0.f;
            if (mn != -INFINITY) {
                if (m2 != -INFINITY) l += lsum * ex2(m2 - mn);
                if (mo != -INFINITY) l += lo * ex2(mo - mn);
            }
            p.m[st_idx] = mn == -INFINITY ? -INFINITY : mn * LN2;
            p.l[st_idx] = l;
        }
    }
    if (MODE == 3) {
        // key blocks of the chunk that no row of this query block sees
        const int chunk_hi = min(p.KB, (p.kv_end + BN - 1) / BN);
        for (int kb = rg.kb_hi + rw * 32 + lane; kb < chunk_hi; kb += 32 * NRED)
            p.block_sum[((size_t)h * p.QB + qb) * p.KB + kb] = 0.f;
    }
}

template <int MODE>
__global__ void __launch_bounds__(NTHREADS, 2)
xattn_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const XParams p, const DevCtx ctx) {
    extern __shared__ __align__(1024) uint8_t dsmem[];
    Smem &sm = *reinterpret_cast<Smem *>(dsmem);
    const int warp = threadIdx.x >> 5;
    const int qb = blockIdx.x, h = blockIdx.y;
    if (smem_u32(dsmem) & 1023u) {  // the 128B swizzle needs an aligned base
        if (threadIdx.x == 0) record_error(ctx, DEVERR_LAYOUT);
        return;
    }
    const Range rg = tile_range(p, qb);
    if (threadIdx.x == 0) {
        Bars &b = sm.b;
        mbar_init(smem_u32(&b.q_full), 1);
        for (int i = 0; i < KST; ++i) {
            mbar_init(smem_u32(&b.k_full[i]), 1);
            mbar_init(smem_u32(&b.k_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&b.s_full[i]), 1);
            mbar_init(smem_u32(&b.s_empty[i]), NRED);
        }
        mbar_init(smem_u32(&b.drain), 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sm.tmem_base), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    if (warp == 0) {
        producer(p, sm, &tq, &tk, qb, h, rg, ctx);
    } else if (warp == 1) {
        if ((threadIdx.x & 31) == 0) mma_thread(sm, tmem, rg.kb_hi - rg.kb_lo, ctx);
        __syncwarp();
    } else {
        reduce_rows<MODE>(p, sm, tmem, qb, h, rg, ctx);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// Stage 2: m = max_c m_c, l = sum_c l_c exp(m_c - m), one thread per row.
__global__ void merge_stats_kernel(const float *__restrict__ m_parts,
                                   const float *__restrict__ l_parts, int C, long long R,
                                   float *__restrict__ m_out, float *__restrict__ l_out) {
    const long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= R) return;
    float m = -INFINITY;
    for (int c = 0; c < C; ++c) m = fmaxf(m, m_parts[(size_t)c * R + r]);
    float l = 0.f;
    if (m != -INFINITY) {
        for (int c = 0; c < C; ++c) {
            const float mc = m_parts[(size_t)c * R + r];
            if (mc != -INFINITY) l += l_parts[(size_t)c * R + r] * ex2((mc - m) * LOG2E);
        }
    }
    m_out[r] = m;
    l_out[r] = l;
}

// Step 4: one CTA per (head, query block). The key blocks are sorted by
// (mass descending, block ascending) with a bitonic sort of 64-bit keys in
// shared memory (masses are >= 0, so their bit patterns order like the
// values); one thread then walks them in that order with float64 sums.
constexpr int FB_THREADS = 256;
constexpr int FB_MAX = 4096;  // key blocks per row supported

__global__ void __launch_bounds__(FB_THREADS)
find_blocks_kernel(const float *__restrict__ block_sum, int KB, float threshold,
                   uint8_t *__restrict__ mask) {
    extern __shared__ unsigned long long keys[];
    const size_t row = blockIdx.x;  // h * QB + qb
    const float *v = block_sum + row * KB;
    uint8_t *out = mask + row * KB;
    int n = 1;
    while (n < KB) n <<= 1;
    for (int i = threadIdx.x; i < n; i += FB_THREADS) {
        unsigned long long key = ~0ull;  // padding sorts last
        if (i < KB) {
            const float x = fmaxf(v[i], 0.f);
            key = ((unsigned long long)(0xffffffffu - __float_as_uint(x)) << 32) | (unsigned)i;
        }
        keys[i] = key;
        if (i < KB) out[i] = 0;
    }
    __syncthreads();
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += FB_THREADS) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long a = keys[i], b2 = keys[ixj];
                    const bool up = (i & k) == 0;
                    if ((a > b2) == up) {
                        keys[i] = b2;
                        keys[ixj] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    if (threadIdx.x == 0) {
        double total = 0.0;
        for (int i = 0; i < KB; ++i) total += (double)__uint_as_float(0xffffffffu - (unsigned)(keys[i] >> 32));
        if (total > 0.0) {
            const double target = (double)threshold * total;
            double cum = 0.0;
            for (int i = 0; i < KB; ++i) {
                const unsigned long long key = keys[i];
                cum += (double)__uint_as_float(0xffffffffu - (unsigned)(key >> 32));
                out[(unsigned)(key & 0xffffffffu)] = 1;
                if (cum >= target) break;
            }
        }
    }
}

CUresult make_map(CUtensorMap *m, const void *base, int rows, int heads) {
    const uint64_t dims[3] = {(uint64_t)HD, (uint64_t)heads, (uint64_t)rows};
    const uint64_t strides[2] = {(uint64_t)HD * 2, (uint64_t)HD * 2 * heads};
    const uint32_t box[3] = {64, 1, (uint32_t)BM};
    return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                             strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int MODE>
cudaError_t launch_tc(const XattnArgs &a, const DevInfo &dev, cudaStream_t s) {
    XParams p{};
    p.M = a.M;
    p.Nctx = a.Nctx;
    p.H = a.H;
    p.Hkv = a.Hkv;
    p.q_pos0 = a.q_pos0;
    p.kv_begin = a.kv_begin;
    p.kv_end = a.kv_end;
    p.causal = a.causal;
    p.scale_l2 = a.scale * LOG2E;
    p.m = a.m;
    p.l = a.l;
    p.block_sum = a.block_sum;
    p.QB = (a.M + BM - 1) / BM;
    p.KB = (a.Nctx + BN - 1) / BN;
    if (a.M == 0) return cudaSuccess;
    CUtensorMap tq, tk;
    if (make_map(&tq, a.q, a.M, a.H) != CUDA_SUCCESS ||
        make_map(&tk, a.k, a.Nctx > 0 ? a.Nctx : 1, a.Hkv) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(Smem);
    static bool attr_set[64] = {};
    if (!attr_set[dev.device & 63]) {
        cudaError_t e = cudaFuncSetAttribute(xattn_tc_kernel<MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set[dev.device & 63] = true;
    }
    DevCtx ctx{dev.err, wait_limit_ns()};
    const dim3 grid(p.QB, a.H);
    xattn_tc_kernel<MODE><<<grid, NTHREADS, smem, s>>>(tq, tk, p, ctx);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_xattn_stats(const XattnArgs &a, const DevInfo &dev, cudaStream_t s) {
    return launch_tc<1>(a, dev, s);
}

cudaError_t launch_xattn_block_sum(const XattnArgs &a, const DevInfo &dev, cudaStream_t s) {
    return launch_tc<3>(a, dev, s);
}

cudaError_t launch_xattn_merge_stats(const float *m_parts, const float *l_parts, int C, long long R,
                                     float *m_out, float *l_out, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    const long long blocks = (R + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    merge_stats_kernel<<<(unsigned)blocks, 256, 0, s>>>(m_parts, l_parts, C, R, m_out, l_out);
    return cudaGetLastError();
}

cudaError_t launch_xattn_find_blocks(const float *block_sum, int rows, int KB, float threshold,
                                     uint8_t *mask, cudaStream_t s) {
    if (rows == 0 || KB == 0) return cudaSuccess;
    if (KB > FB_MAX) return cudaErrorInvalidValue;
    int n = 1;
    while (n < KB) n <<= 1;
    find_blocks_kernel<<<rows, FB_THREADS, (size_t)n * 8, s>>>(block_sum, KB, threshold, mask);
    return cudaGetLastError();
}

}  // namespace sattn
