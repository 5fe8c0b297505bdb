// XAttention block selection ("XAttention Offload Stream Synchronization
// Fix", technical details): stage 1 computes per-chunk softmax stats (m, l) of
// every query row, stage 2 merges them, stage 3 sums the normalised
// probabilities exp(s - m) / l over 128 x 128 blocks, step 4 selects, per
// query block, the shortest run of key blocks by descending mass that reaches
// threshold x the total. The estimate is the exact softmax at full
// resolution.
//
// Stages 1 and 3 are one persistent tcgen05 kernel (MODE 1 / MODE 3), one CTA
// per SM looping over work items. An item is two work units that read the
// same key tiles, each a (query block of 128 rows, head): two heads of one KV
// group when the group has an even number of heads, else two consecutive
// query blocks of one head; and one piece of the key range (a chunk in stage
// 1, at most 4096 keys in stage 3). A producer warp loads each item's two Q
// tiles and streams its key tiles into a 4-stage ring (2-D boxes of a 3-D
// tensor map, 128B swizzle) that runs on across items; one thread issues
// S = Q K^T per unit and tile (M = N = 128, K = 128 in eight K = 16 steps)
// into two TMEM accumulators per unit; eight warps per unit, two per TMEM
// lane quarter with 64 columns each, own one query row per thread and reduce
// its scores in the log2 domain (one MUFU ex2 per score). The MMAs of one
// tile overlap the exponentials of the one before, and an item's first tiles
// load while the previous item ends.
#include <math.h>
#include <stdio.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace sattn {
namespace {

constexpr int BM = 128;  // query rows per unit
constexpr int BN = 128;  // keys per tile (= the block size)
constexpr int HD = 128;
constexpr int NU = 2;    // work units per item
constexpr int NRED = 8;  // reduction warps per unit: two per TMEM lane quarter, 64 columns each
constexpr int KST = 4;   // key-tile stages
constexpr int NTHREADS = 32 * (2 + NU * NRED);  // producer, MMA, reduction warps
constexpr uint32_t TMEM_COLS = 512;            // two 128-column S accumulators per unit
constexpr uint32_t TILE = BN * HD * 2;         // 32 KB
constexpr uint32_t HALF = TILE / 2;            // one 64-column half
constexpr int PART = 64;     // tiles whose block partials are kept before a flush
constexpr int PIECE = 4096;  // keys per item in stage 3

struct Bars {
    uint64_t q_full, q_empty, k_full[KST], k_empty[KST], s_full[NU][2], s_empty[2], drain;
};

struct alignas(1024) Smem {
    uint8_t q[NU][TILE];
    uint8_t k[KST][TILE];
    float part[NU * NRED][PART];  // MODE 3: per reduction warp, per tile: its rows' mass
    float xch[NU][2][BM];         // MODE 1: (m, l) of the second column half of each row
    Bars b;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Smem) <= 227 * 1024, "shared memory of one CTA");

struct XParams {
    int M, Nctx, H, Hkv, q_pos0, kv_begin, kv_end, causal;
    int piece;           // keys per piece of [kv_begin, kv_end)
    int pair_heads;      // units: heads 2y, 2y+1 of query block x; else query blocks 2x, 2x+1 of head y
    int GX, GY, n_items;  // unit pairs along x and y; items = GX * GY * pieces
    long long m_stride;  // MODE 1: elements between the (m, l) outputs of consecutive pieces
    float scale_l2;      // scale * log2(e)
    float *m, *l;        // MODE 1: written; MODE 3: the merged stats
    float *block_sum;    // MODE 3: [H, QB, KB]
    int QB, KB;
};

constexpr uint32_t IDESC = idesc_bf16_f32(128, 128, 0, 0);

__host__ __device__ constexpr uint32_t koff(int kk) {
    return ((uint32_t)(kk >> 2) * HALF + (uint32_t)(kk & 3) * 32u) >> 4;
}

// One work item: its piece of the key range, [kv_begin, kv_end), the key
// tiles [kb_lo, kb_hi) that some row of its units may see, and the units.
struct Item {
    int kv_begin, kv_end, kb_lo, kb_hi, z;
    int qb[NU], h[NU];
    bool ok[NU];  // qb < QB (the second unit of an odd number of query blocks is empty)
};
__device__ __forceinline__ Item item_of(const XParams &p, int it) {
    Item w;
    const int x = it % p.GX, rest = it / p.GX;
    const int y = rest % p.GY, z = rest / p.GY;
    int qb_last = 0;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
        w.qb[u] = p.pair_heads ? x : 2 * x + u;
        w.h[u] = p.pair_heads ? 2 * y + u : y;
        w.ok[u] = w.qb[u] < p.QB;
        if (w.ok[u]) qb_last = max(qb_last, w.qb[u]);
    }
    w.z = z;
    w.kv_begin = p.kv_begin + z * p.piece;
    w.kv_end = (int)min((long long)p.kv_end, (long long)w.kv_begin + p.piece);
    w.kb_lo = w.kv_begin / BN;
    int hi = (w.kv_end + BN - 1) / BN;
    if (p.causal) {
        const int i_last = min(p.M, (qb_last + 1) * BM) - 1;
        hi = min(hi, (p.q_pos0 + i_last) / BN + 1);  // the last key any row of the units sees
    }
    w.kb_hi = max(hi, w.kb_lo);
    return w;
}

__device__ __forceinline__ bool wait_warp(uint64_t &bar, uint32_t parity, const DevCtx &ctx,
                                          volatile int *abort) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(smem_u32(&bar), parity, ctx, abort) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
}

// Producer warp. Per item: the first key tiles that the ring has room for,
// then (once the previous item's MMAs are done with the Q buffers) the two Q
// tiles, then the rest of the key tiles. The next item's Q is prefetched
// into L2 meanwhile.
__device__ void producer(const XParams &p, Smem &sm, const CUtensorMap *tq, const CUtensorMap *tk,
                         const DevCtx &ctx) {
    Bars &b = sm.b;
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        prefetch_tmap(tq);
        prefetch_tmap(tk);
    }
    int kt = 0;  // key tiles issued so far
    int nq = 0;  // items whose Q was issued
    bool failed = false;
    for (int it = blockIdx.x; it < p.n_items && !failed; it += gridDim.x) {
        const Item w = item_of(p, it);
        const int g = w.h[0] / (p.H / p.Hkv);  // both units read the same KV head
        const int ntiles = w.kb_hi - w.kb_lo;
        const int nfirst = min(ntiles, KST);
        if (lane == 0 && it + (int)gridDim.x < p.n_items) {
            const Item nx = item_of(p, it + gridDim.x);
#pragma unroll
            for (int u = 0; u < NU; ++u)
                if (nx.ok[u]) {
                    tma_prefetch_l2_3d(tq, 0, nx.h[u], nx.qb[u] * BM);
                    tma_prefetch_l2_3d(tq, 64, nx.h[u], nx.qb[u] * BM);
                }
        }
        for (int j = 0; j <= ntiles; ++j) {
            if (j == nfirst) {
                // Q of this item, once the previous item's last MMA has read its Q
                if (nq >= 1 && !wait_warp(b.q_empty, (nq - 1) & 1, ctx, &sm.abort)) {
                    failed = true;
                    break;
                }
                if (lane == 0) {
                    const uint32_t bar = smem_u32(&b.q_full);
                    mbar_arrive_expect_tx(bar, (uint32_t)((int)w.ok[0] + (int)w.ok[1]) * TILE);
#pragma unroll
                    for (int u = 0; u < NU; ++u)
                        if (w.ok[u]) {  // an empty unit's S is never read
                            tma_load_3d(smem_u32(sm.q[u]), tq, bar, 0, w.h[u], w.qb[u] * BM);
                            tma_load_3d(smem_u32(sm.q[u]) + HALF, tq, bar, 64, w.h[u], w.qb[u] * BM);
                        }
                }
                ++nq;
            }
            if (j == ntiles) break;
            const int st = kt % KST, use = kt / KST;
            if (use >= 1 && !wait_warp(b.k_empty[st], (use - 1) & 1, ctx, &sm.abort)) {
                failed = true;
                break;
            }
            if (lane == 0) {
                const uint32_t bar = smem_u32(&b.k_full[st]);
                mbar_arrive_expect_tx(bar, TILE);
                tma_load_3d(smem_u32(sm.k[st]), tk, bar, 0, g, (w.kb_lo + j) * BN);
                tma_load_3d(smem_u32(sm.k[st]) + HALF, tk, bar, 64, g, (w.kb_lo + j) * BN);
            }
            ++kt;
        }
    }
    // the loads in flight land before the CTA may leave (matters after an abort)
    if (lane == 0) {
        int zero = 0;
        for (int u = kt > KST ? kt - KST : 0; u < kt; ++u)
            mbar_wait(smem_u32(&b.k_full[u % KST]), (u / KST) & 1, ctx, &zero);
        if (nq >= 1) mbar_wait(smem_u32(&b.q_full), (nq - 1) & 1, ctx, &zero);
    }
    __syncwarp();
}

// One thread: per item, S of every tile and unit in order (unit u's tiles
// alternate between its two accumulators); the Q buffers are released after
// the item's last MMA. A tile's two waits (its key stage, the accumulators
// of both units) come before its sixteen MMAs: a shared-memory access by
// this thread stalls the MMAs already queued, so the accesses are few and
// grouped.
__device__ void mma_issue(const XParams &p, Smem &sm, uint32_t tmem, const DevCtx &ctx) {
    Bars &b = sm.b;
    volatile int *abort = &sm.abort;
    const uint64_t dk0 = smem_desc_sw128(smem_u32(sm.k[0]), 16u, 1024u);
    const uint64_t dq0 = smem_desc_sw128(smem_u32(sm.q[0]), 16u, 1024u);
    int kt = 0, ut = 0, k = 0;  // key tiles, tiles per unit, items so far
    for (int it = blockIdx.x; it < p.n_items; it += gridDim.x, ++k) {
        const Item w = item_of(p, it);
        const int ntiles = w.kb_hi - w.kb_lo;
        if (!mbar_wait(smem_u32(&b.q_full), k & 1, ctx, abort)) return;
        for (int t = 0; t < ntiles; ++t, ++kt, ++ut) {
            const int st = kt % KST, sb = ut & 1;
            if (!mbar_wait(smem_u32(&b.k_full[st]), (kt / KST) & 1, ctx, abort)) return;
            // accumulator sb of both units, released by all their reduction warps
            if (ut >= 2 && !mbar_wait(smem_u32(&b.s_empty[sb]), ((ut >> 1) - 1) & 1, ctx, abort))
                return;
            tc_fence_after();
            const uint64_t dk = dk0 + (uint64_t)(st * (TILE >> 4));
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                const uint64_t dq = dq0 + (uint64_t)(u * (TILE >> 4));
                const uint32_t acc = tmem + 128u * (uint32_t)(2 * u + sb);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    tc_mma_f16(acc, dq + koff(kk), dk + koff(kk), IDESC, kk > 0 ? 1u : 0u);
                tc_commit(smem_u32(&b.s_full[u][sb]));
            }
            tc_commit(smem_u32(&b.k_empty[st]));
        }
        tc_commit(smem_u32(&b.q_empty));
    }
}

__device__ void mma_thread(const XParams &p, Smem &sm, uint32_t tmem, const DevCtx &ctx) {
    if (ctx.stall) mbar_wait(smem_u32(&sm.b.drain), 0, ctx, &sm.abort);  // test hook: runs out
    mma_issue(p, sm, tmem, ctx);
    // every MMA issued completes before TMEM is released (also after an abort)
    tc_commit(smem_u32(&sm.b.drain));
    int zero = 0;
    mbar_wait(smem_u32(&sm.b.drain), 0, ctx, &zero);
}

// Named barrier (id 1 + unit) over the reduction threads of one unit,
// OR-reducing a predicate.
__device__ __forceinline__ int red_bar_or(int id, int pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.s32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred), "r"(id), "r"(32 * NRED)
        : "memory");
    return r;
}

// A query row (TMEM lane) per thread and half-tile: reduction warp w of unit
// u handles lane quarter (warp index % 4) and columns 64 (w / 4) .. +63 of
// each S tile. MODE 1: online (max, sum of exp) of the row's visible scores,
// the two halves merged at the end of the item through shared memory; MODE 3:
// the row's mass exp(s - m) / l per tile, summed over the warp's 32 rows,
// then over the unit's eight warps per key block.
template <int MODE>
__device__ void reduce_rows(const XParams &p, Smem &sm, uint32_t tmem, const DevCtx &ctx) {
    Bars &b = sm.b;
    volatile int *abort = &sm.abort;
    const int lane = threadIdx.x & 31, quarter = (threadIdx.x >> 5) & 3;
    const int rwg = (threadIdx.x >> 5) - 2;  // reduction warp 0 .. NU*NRED-1
    const int u = rwg / NRED, rw = rwg % NRED;
    const int half = rw >> 2;            // column half of the tiles
    const int rt = quarter * 32 + lane;  // row within the tile = TMEM lane
    const uint32_t s_base = tmem + 256u * (uint32_t)u + 64u * (uint32_t)half +
                            ((uint32_t)(quarter * 32) << 16);
    const uint64_t c2 = f2_pack(p.scale_l2, p.scale_l2);
    bool failed = false;
    int ut = 0;  // tiles of this unit so far (all items)
    for (int it = blockIdx.x; it < p.n_items; it += gridDim.x) {
        const Item w = item_of(p, it);
        const int qb = u ? w.qb[1] : w.qb[0], h = u ? w.h[1] : w.h[0];
        const bool unit_ok = u ? w.ok[1] : w.ok[0];
        const int i = qb * BM + rt;
        const bool row_ok = unit_ok && i < p.M;
        // last key the row may see
        const int jmax = p.causal ? min(w.kv_end - 1, p.q_pos0 + i) : w.kv_end - 1;
        const size_t st_idx = (size_t)(row_ok ? i : 0) * p.H + h;
        float neg_lse2 = 0.f;
        bool has_mass = false;
        if (MODE == 3 && row_ok) {
            const float m = p.m[st_idx], l = p.l[st_idx];
            has_mass = l > 0.f && m != -INFINITY;
            neg_lse2 = has_mass ? -(m * LOG2E + log2f(l)) : 0.f;
        }
        float m2 = -INFINITY, lsum = 0.f;
        const int ntiles = w.kb_hi - w.kb_lo;
        int batch0 = 0;  // first tile of the current partial batch
        for (int t = 0; t < ntiles; ++t, ++ut) {
            const int sb = ut & 1, j0 = (w.kb_lo + t) * BN;
            if (!failed) failed = !wait_warp(b.s_full[u][sb], (ut >> 1) & 1, ctx, abort);
            float rowsum = 0.f;
            if (!failed) {
                tc_fence_after();
                uint32_t v[2][32];
#pragma unroll
                for (int cc = 0; cc < 2; ++cc)
                    tmem_ld32(s_base + 128u * (uint32_t)sb + 32u * (uint32_t)cc, v[cc]);
                tc_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&b.s_empty[sb]));
                // visible columns of this row within the warp's half: [clo, chi]
                const int jh = j0 + 64 * half;
                const int clo = max(0, w.kv_begin - jh), chi = min(63, jmax - jh);
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
                float ws = rowsum;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
                if (lane == 0) sm.part[rwg][t - batch0] = ws;
                if (t - batch0 == PART - 1 || t == ntiles - 1) {
                    // every warp of the unit reaches this at the same t: the flush is uniform
                    if (red_bar_or(1 + u, failed)) failed = true;
                    if (!failed && unit_ok) {
                        for (int tt = rw * 32 + lane; tt <= t - batch0; tt += 32 * NRED) {
                            float s = 0.f;
#pragma unroll
                            for (int w2 = 0; w2 < NRED; ++w2) s += sm.part[u * NRED + w2][tt];
                            p.block_sum[((size_t)h * p.QB + qb) * p.KB + w.kb_lo + batch0 + tt] = s;
                        }
                    }
                    red_bar_or(1 + u, 0);  // the partials are read before the next batch writes them
                    batch0 = t + 1;
                }
            }
        }
        if (MODE == 1) {
            // the two column halves of each row: half 1 hands (m, l) to half 0
            float *xm = sm.xch[u][0], *xl = sm.xch[u][1];
            if (half == 1) {
                xm[rt] = m2;
                xl[rt] = lsum;
            }
            red_bar_or(1 + u, 0);
            if (half == 0 && row_ok && !failed) {
                const float mo = xm[rt], lo = xl[rt];
                const float mn = fmaxf(m2, mo);
                float l = 0.f;
                if (mn != -INFINITY) {
                    if (m2 != -INFINITY) l += lsum * ex2(m2 - mn);
                    if (mo != -INFINITY) l += lo * ex2(mo - mn);
                }
                const size_t o_idx = (size_t)w.z * (size_t)p.m_stride + st_idx;
                p.m[o_idx] = mn == -INFINITY ? -INFINITY : mn * LN2;
                p.l[o_idx] = l;
            }
            red_bar_or(1 + u, 0);  // read before the next item writes the exchange area
        }
        if (MODE == 3 && unit_ok) {
            // key blocks of the piece that no row of this unit sees
            const int piece_hi = min(p.KB, (w.kv_end + BN - 1) / BN);
            for (int kb = w.kb_hi + rw * 32 + lane; kb < piece_hi; kb += 32 * NRED)
                p.block_sum[((size_t)h * p.QB + qb) * p.KB + kb] = 0.f;
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(NTHREADS, 1)
xattn_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const XParams p, const DevCtx ctx) {
    extern __shared__ __align__(1024) uint8_t dsmem[];
    Smem &sm = *reinterpret_cast<Smem *>(dsmem);
    const int warp = threadIdx.x >> 5;
    if (smem_u32(dsmem) & 1023u) {  // the 128B swizzle needs an aligned base
        if (threadIdx.x == 0) record_error(ctx, DEVERR_LAYOUT);
        return;
    }
    if (threadIdx.x == 0) {
        Bars &b = sm.b;
        mbar_init(smem_u32(&b.q_full), 1);
        mbar_init(smem_u32(&b.q_empty), 1);
        for (int i = 0; i < KST; ++i) {
            mbar_init(smem_u32(&b.k_full[i]), 1);
            mbar_init(smem_u32(&b.k_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            for (int u = 0; u < NU; ++u) mbar_init(smem_u32(&b.s_full[u][i]), 1);
            mbar_init(smem_u32(&b.s_empty[i]), NU * NRED);
        }
        mbar_init(smem_u32(&b.drain), 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sm.tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    if (warp == 0) {
        producer(p, sm, &tq, &tk, ctx);
    } else if (warp == 1) {
        if ((threadIdx.x & 31) == 0) mma_thread(p, sm, tmem, ctx);
        __syncwarp();
    } else {
        reduce_rows<MODE>(p, sm, tmem, ctx);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
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
// shared memory (masses are taken as >= 0, so their bit patterns order like
// the values); the selection then takes the shortest leading run whose
// float64 running sum, taken in that order, reaches threshold x the total.
//
// Fast path (at most FB_THREADS blocks, nonzero masses within 2^21 of each
// other): every mass is an integer multiple of 2^(emin - 150), emin the
// smallest biased exponent among them, below 2^(24 + 21); a running sum of
// at most 256 of them stays below 2^53 units, so each float64 running sum is
// exact and equals the integer prefix sum, which the CTA computes with a
// parallel scan. Otherwise one thread walks the blocks with float64 sums.
// Both give the same decisions.
constexpr int FB_THREADS = 256;
constexpr int FB_MAX = 4096;  // key blocks per row supported
constexpr int FB_SPAN = 53 - 24 - 8;  // exponent span of the fast path (256 terms)

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
            // a negative, -0 or NaN mass counts as +0 (whose bits sort last)
            const float x = v[i] > 0.f ? v[i] : 0.f;
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
    // ---- fast path: integer prefix sums (thread t holds sorted position t)
    __shared__ int s_emin, s_emax, s_first;
    __shared__ long long s_warp[FB_THREADS / 32];
    if (threadIdx.x == 0) {
        s_emin = 1 << 30;
        s_emax = -1;
        s_first = KB;
    }
    __syncthreads();
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const uint32_t u = t < KB ? 0xffffffffu - (uint32_t)(keys[t] >> 32) : 0u;  // mass bits
    const int be = (int)(u >> 23);                                            // biased exponent
    if (KB <= FB_THREADS && u != 0u) {
        atomicMin(&s_emin, be > 0 ? be : 1);
        atomicMax(&s_emax, be);
    }
    __syncthreads();
    const int emin = s_emin, emax = s_emax;
    if (KB <= FB_THREADS && emax < 0) return;  // no mass: nothing selected
    if (KB <= FB_THREADS && emax < 255 && emax - emin <= FB_SPAN) {
        // the mass in units of 2^(emin - 150): significand shifted by its exponent's excess
        const long long mant = (long long)((u & 0x7fffffu) | (be > 0 ? 0x800000u : 0u));
        long long x = u != 0u ? mant << ((be > 0 ? be : 1) - emin) : 0ll;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {  // inclusive scan within the warp
            const long long y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_warp[wid] = x;
        __syncthreads();
        long long before = 0;
        for (int w = 0; w < wid; ++w) before += s_warp[w];
        long long total = 0;
        for (int w = 0; w < FB_THREADS / 32; ++w) total += s_warp[w];
        const long long prefix = before + x;  // running sum through sorted position t
        if (total > 0) {
            const double unit = ldexp(1.0, emin - 150);
            const double target = (double)threshold * ((double)total * unit);
            if (t < KB && (double)prefix * unit >= target) atomicMin(&s_first, t);
            __syncthreads();
            // all blocks up to the first position that reaches the target
            // (all of them if none does)
            const int last = s_first < KB ? s_first : KB - 1;
            if (t <= last) out[(unsigned)(keys[t] & 0xffffffffu)] = 1;
        }
        return;
    }
    // ---- otherwise: one thread, float64 running sums in sorted order
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

// MODE 1: one (m, l) output per chunk of `chunk` keys of [kv_begin, kv_end)
// (one output for the whole range when chunk is 0); MODE 3: the range split
// into pieces of PIECE keys, which leaves the block sums unchanged.
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
    p.m_stride = (long long)a.M * a.H;
    // two heads of a KV group share each key tile when the group has an even
    // size; otherwise two consecutive query blocks of one head do
    p.pair_heads = (a.H / a.Hkv) % 2 == 0;
    p.GX = p.pair_heads ? p.QB : (p.QB + 1) / 2;
    p.GY = p.pair_heads ? a.H / 2 : a.H;
    if (a.M == 0) return cudaSuccess;
    const long long len = (long long)a.kv_end - a.kv_begin;
    long long z;
    if (MODE == 1) {
        p.piece = a.chunk > 0 ? a.chunk : (int)(len > 0 ? len : 1);
        z = len > 0 ? (len + p.piece - 1) / p.piece : 1;
    } else {
        p.piece = PIECE;
        z = (len + PIECE - 1) / PIECE;
        if (z == 0) return cudaSuccess;
    }
    const long long items = (long long)p.GX * p.GY * z;
    if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
    p.n_items = (int)items;
    CUtensorMap tq, tk;
    if (make_map(&tq, a.q, a.M, a.H) != CUDA_SUCCESS ||
        make_map(&tk, a.k, a.Nctx > 0 ? a.Nctx : 1, a.Hkv) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(Smem);
    {
        cudaError_t e = ensure_smem_attr((const void *)xattn_tc_kernel<MODE>, smem, dev);
        if (e != cudaSuccess) return e;
    }
    const DevCtx ctx = make_ctx(dev);
    const int grid = (int)std::min<long long>(items, dev.sm_count > 0 ? dev.sm_count : 1);
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
