// Gathered decode attention, the splits of each query merged inside a
// thread-block cluster ("DeepSeek-V4 CSA/HCA walkthrough", sections 4.1-4.4:
// topk_idxs per query, -1 entries masked, the gathered rows staged as dense
// tiles, a null-logit sink in the softmax denominator; "XAttention Offload
// Stream Synchronization Fix", technical details: partial (m, l) stats per
// piece of the key set, merged through the log-sum-exp).
//
// With few queries one query's list is too short to keep many SMs busy, so
// it is cut into C contiguous segments (C a power of two <= 8, chosen so
// that every CTA of the grid is resident at once), one per CTA of a cluster
// of C CTAs. A CTA
//   - loads its segment's entries and Q, and issues the cp.async copies of
//     every row of the segment at once (at most DT_MAX tiles of 128 rows, each
//     in its own stage; a -1 entry's row is zero-filled and its score masked,
//     nothing is compacted),
//   - computes S^T = KV Q^T per tile on the tensor cores (sparse_layout.cuh),
//   - takes the softmax over the whole segment: the segment's max first, then
//     P (bf16) and the row sums, no rescaling,
//   - accumulates O^T += KV^T P^T over the tiles,
//   - takes part in the merge of the cluster's partials (m, l, O^T).
// The merge through the log-sum-exp is split in two exchanges, both
// asynchronous stores into the other CTAs' shared memory whose bytes
// complete on the receiver's own mbarrier. As soon as its P is written each
// CTA sends its (m, l) of all 32 heads to every CTA of the cluster; while P V
// runs, every CTA computes each head's merged max and denominator (the
// null-logit sink added here, once), lse and its own weight. CTA r owns heads
// [r 32/C, (r+1) 32/C) of the query: every CTA scales its O^T rows of those
// heads by its weight and sends them to CTA r, which adds what it receives
// and writes o and lse. One launch, no workspace.
//
// Warps 0-3: Q copy, softmax, epilogue and merge (warp w reads TMEM lanes
// 32w .. 32w+31); warps 4-7: row copies (warp 4 + g: rows 32g .. 32g+31 of
// each tile), after which lane 0 of warp 4 issues the MMAs. With an FP8
// cache the copy warps take the bf16 RoPE half by cp.async and dequantise the
// e4m3 half into the stage (Fp8Copier); everything else is the same.
#include <math.h>
#include <stdio.h>

#include "common.cuh"
#include "internal.h"
#include "sparse_layout.cuh"

namespace sattn {
namespace {

using namespace gather;

constexpr int DT_MAX = 3;           // tiles per CTA
constexpr int MAX_CLUSTER = 8;      // CTAs per query (portable cluster size)
constexpr int DEC_THREADS = 256;
constexpr uint32_t DEC_TMEM_COLS = 128;  // S^T of DT_MAX tiles (32 columns each), O^T
constexpr uint32_t DS_COL = 0, DO_COL = 96;
// Received O^T rows: C CTAs x HD rows of hs = NH / C heads, padded to hs + 4
// floats so that 16-byte accesses of consecutive rows avoid bank conflicts;
// the most is C = 8 (8 x 128 x 8 floats).
constexpr int RECV_FLOATS = MAX_CLUSTER * HD * (NH / MAX_CLUSTER + 4);

struct DecBars {
    uint64_t q_full;
    uint64_t kv_full[DT_MAX], s_full[DT_MAX];
    uint64_t p_full;     // P of every tile written (each softmax warp arrives once)
    uint64_t o_full, drain;
    uint64_t stats_full; // every CTA's (m, l) of all heads has landed (tx bytes)
    uint64_t recv_full;  // every CTA's weighted O^T rows of this CTA's heads (tx bytes)
};

// Bytes a CTA receives: (m, l) of all NH heads from each of the C CTAs; and
// from each of them HD rows of hs = NH / C weighted O^T values (C hs = NH).
constexpr uint32_t STATS_BYTES_PER_CTA = NH * 8;
constexpr uint32_t RECV_BYTES = NH * HD * 4;

struct alignas(1024) DecSmem {
    uint8_t kv[DT_MAX][KV_TILE];
    uint8_t q[2 * QP_HALF];
    uint8_t p[DT_MAX][2 * QP_HALF];
    float tbuf[4][NH * TB_STRIDE];
    // weighted O^T rows of this CTA's heads sent by every CTA c of the
    // cluster: recv[(c HD + d) (hs + 4) + j]
    float recv[RECV_FLOATS];
    float stat_m[MAX_CLUSTER][NH], stat_l[MAX_CLUSTER][NH];  // every CTA's (m, l), log2 units
    float wself[NH];                    // this CTA's weight per head in the merged result
    float lse_h[NH];
    float sink_l2[NH];                  // null-logit sinks x log2(e), -inf without
    int ids[DT_MAX][R];                 // FP8: each tile's entries, read by the copier
    float xmax[4][NH];                  // per-warp maxima of the segment
    float lpart[4][NH];                 // per-warp row sums
    DecBars b;
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(DecSmem) <= 227 * 1024, "shared memory of one CTA");

struct DecParams {
    const __nv_bfloat16 *q, *kv;
    // FP8 cache: e4m3 codes of the first DN columns, one scale per row, bf16
    // RoPE part (the last HD - DN columns)
    const uint8_t *kv_nope;
    const __nv_bfloat16 *kv_rope;
    const float *kv_scale;
    const int32_t *idx;
    const float *sinks;
    int sink_mode;
    float scale_l2;
    __nv_bfloat16 *o;
    float *lse;
    int M, N, K;
    int C;    // CTAs per query (cluster size)
    int seg;  // list entries per CTA (<= DT_MAX * R)
};

// Named barrier of the four softmax warps.
__device__ __forceinline__ void softmax_bar() {
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

__device__ void dec_mma(const DecSmem &sm, DecBars &b, uint32_t tmem, int nt, volatile int *abort,
                        const DevCtx &ctx) {
    if (ctx.stall) mbar_wait(smem_u32(&b.drain), 0, ctx, abort);  // test hook: runs out
    bool ok = nt > 0 && mbar_wait(smem_u32(&b.q_full), 0, ctx, abort);
    const uint64_t dq = desc_sw128(smem_u32(sm.q), 16u);
    int issued = 0;
    for (int t = 0; ok && t < nt; ++t) {
        if (!(ok = mbar_wait(smem_u32(&b.kv_full[t]), 0, ctx, abort))) break;
        tc_fence_after();
        const uint64_t a = desc_sw128(smem_u32(sm.kv[t]), 16u);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
            tc_mma_f16(tmem + DS_COL + 32u * t, a + koff(kk, KV_HALF), dq + koff(kk, QP_HALF),
                       IDESC_S, kk > 0 ? 1u : 0u);
        tc_commit(smem_u32(&b.s_full[t]));
        ++issued;
    }
    // P of all tiles is written together: one wait, then every P V back to
    // back (a barrier access of this thread stalls the MMAs already queued)
    if (ok && issued > 0) ok = mbar_wait(smem_u32(&b.p_full), 0, ctx, abort);
    if (ok) tc_fence_after();
    for (int t = 0; ok && t < issued; ++t) {
        const uint64_t a = desc_sw128(smem_u32(sm.kv[t]), KV_HALF);
        const uint64_t bp = desc_sw128(smem_u32(sm.p[t]), 16u);
#pragma unroll
        for (int kk = 0; kk < R / 16; ++kk)
            tc_mma_f16(tmem + DO_COL, a + mnoff(kk), bp + koff(kk, QP_HALF), IDESC_O,
                       (t > 0 || kk > 0) ? 1u : 0u);
    }
    if (ok && issued == nt && nt > 0) tc_commit(smem_u32(&b.o_full));
    // every MMA issued completes before TMEM is released
    tc_commit(smem_u32(&b.drain));
    int zero = 0;
    mbar_wait(smem_u32(&b.drain), 0, ctx, &zero);
}

template <bool FP8>
__global__ void __launch_bounds__(DEC_THREADS, 1)
sparse_decode_kernel(const DecParams p, const DevCtx ctx) {
    extern __shared__ __align__(1024) uint8_t dsmem[];
    DecSmem &sm = *reinterpret_cast<DecSmem *>(dsmem);
    // the 128B swizzle needs an aligned base; the offset is the same in every
    // CTA, so either all CTAs of a cluster leave here or none does
    if (smem_u32(dsmem) & 1023u) {
        if (threadIdx.x == 0) record_error(ctx, DEVERR_LAYOUT);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = p.C;
    const int bm = blockIdx.x / C;                      // query (b, m)
    const uint32_t crank = cluster_ctarank();           // segment of this CTA
    const int seg0 = (int)crank * p.seg;
    const int seg_end = min(p.K, seg0 + p.seg);
    const int nt = seg_end > seg0 ? (seg_end - seg0 + R - 1) / R : 0;
    const int32_t *list = p.idx + (size_t)bm * p.K;

    // ---- loads whose latency the set-up below hides
    // softmax warp w and copy warp 4 + w both take entry 32 w + lane of each tile
    const int rsub = (warp & 3) * 32 + lane;
    int e[DT_MAX];
#pragma unroll
    for (int t = 0; t < DT_MAX; ++t) {
        const int pos = seg0 + t * R + rsub;
        e[t] = (t < nt && pos < seg_end) ? __ldg(list + pos) : -1;
    }
    if (warp < 4) {  // Q of the query: 32 heads x 256 B into the swizzled K-major buffer
        const __nv_bfloat16 *qrow = p.q + (size_t)bm * NH * HD;
        const uint32_t qs = smem_u32(sm.q);
        for (int k = threadIdx.x; k < NH * 16; k += 128) {
            const int h = k >> 4, u = k & 15;
            cp_async16(qs + (uint32_t)(u >> 3) * QP_HALF + sw128_offset(h, u & 7),
                       qrow + h * HD + u * 8, 16u);
        }
    }
    if (threadIdx.x == 0) {
        DecBars &b = sm.b;
        mbar_init(smem_u32(&b.q_full), 128);
        for (int t = 0; t < DT_MAX; ++t) {
            // FP8: each copy warp also arrives once after its dequantised stores
            mbar_init(smem_u32(&b.kv_full[t]), 32 * COPY_WARPS + (FP8 ? COPY_WARPS : 0));
            mbar_init(smem_u32(&b.s_full[t]), 1);
        }
        mbar_init(smem_u32(&b.p_full), 4);
        mbar_init(smem_u32(&b.o_full), 1);
        mbar_init(smem_u32(&b.drain), 1);
        mbar_init(smem_u32(&b.stats_full), 1);
        mbar_arrive_expect_tx(smem_u32(&b.stats_full), STATS_BYTES_PER_CTA * (uint32_t)p.C);
        mbar_init(smem_u32(&b.recv_full), 1);
        mbar_arrive_expect_tx(smem_u32(&b.recv_full), RECV_BYTES);
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&sm.tmem_base), DEC_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // first cluster phase: every CTA of the cluster has started and set up its
    // barriers (waited for before the first store into another CTA's shared
    // memory); the second, at the end, keeps every CTA alive until all the
    // cluster's stores into it have landed
    cluster_arrive_relaxed();
    const uint32_t tmem = sm.tmem_base;
    volatile int *abort = &sm.abort;
    // an entry outside [-1, N) is skipped and recorded
    bool bad = false;
#pragma unroll
    for (int t = 0; t < DT_MAX; ++t) {
        if (e[t] < -1 || e[t] >= p.N) bad = true;
        if (e[t] >= p.N) e[t] = -1;
    }
    if (bad) record_error(ctx, DEVERR_INDEX);

    if (warp >= 4) {
        // ---- row copies: all tiles at once
        const int g = warp - 4;
        const size_t row0 = (size_t)(bm / p.M) * p.N;  // first cache row of the request
        if (!FP8) {
            const RowCopier cp(lane);
            const __nv_bfloat16 *rows = p.kv + row0 * HD;
#pragma unroll
            for (int t = 0; t < DT_MAX; ++t) {
                if (t < nt) {
                    cp.issue_lanes(smem_u32(sm.kv[t]), e[t], rows, g);
                    cp_async_arrive(smem_u32(&sm.b.kv_full[t]));
                }
            }
        } else {
            const Fp8Copier fc(lane);
            // the copier reads each tile's entries by row
#pragma unroll
            for (int t = 0; t < DT_MAX; ++t)
                if (t < nt) sm.ids[t][32 * g + lane] = e[t];
            __syncwarp();
            uint4 codes[DT_MAX][4];
            float scl[DT_MAX][4];
#pragma unroll
            for (int t = 0; t < DT_MAX; ++t)
                if (t < nt)
                    fc.load_codes(sm.ids[t], p.kv_nope + row0 * DN, p.kv_scale + row0, g, codes[t],
                                  scl[t]);
#pragma unroll
            for (int t = 0; t < DT_MAX; ++t) {
                if (t < nt) {
                    fc.issue_rope(smem_u32(sm.kv[t]), sm.ids[t], p.kv_rope + row0 * (HD - DN), g);
                    cp_async_arrive(smem_u32(&sm.b.kv_full[t]));
                }
            }
#pragma unroll
            for (int t = 0; t < DT_MAX; ++t) {
                if (t < nt) {
                    fc.store_codes(smem_u32(sm.kv[t]), g, codes[t], scl[t]);
                    fence_proxy_async_smem();  // the stores are read by the tensor core
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sm.b.kv_full[t]));
                }
            }
        }
        if (warp == 4) {
            if (lane == 0) dec_mma(sm, sm.b, tmem, nt, abort, ctx);
            __syncwarp();
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        tc_fence_before();  // the MMAs drained above come before the dealloc
        cluster_wait_acquire();
        cluster_arrive_relaxed();
        cluster_wait_acquire();
    } else {
        // ---- softmax over the segment (lane = head after the transpose)
        const int quarter = warp, h = lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        cp_async_arrive(smem_u32(&sm.b.q_full));
        const float sink_h = p.sinks ? __ldg(p.sinks + h) * LOG2E : 0.0f;
        const float bias_raw = p.sink_mode == 1 ? sink_h / p.scale_l2 : 0.0f;
        if (quarter == 0) sm.sink_l2[h] = p.sink_mode == 2 ? sink_h : -INFINITY;
        uint32_t vmask[DT_MAX], zmask[DT_MAX];
#pragma unroll
        for (int t = 0; t < DT_MAX; ++t) {
            vmask[t] = __ballot_sync(0xffffffffu, e[t] >= 0);
            zmask[t] = __ballot_sync(0xffffffffu, e[t] == 0);
        }
        float *tb = sm.tbuf[quarter];
        float x[DT_MAX][32];
        bool failed = false;
        float mt = -INFINITY;
#pragma unroll
        for (int t = 0; t < DT_MAX; ++t) {
#pragma unroll
            for (int i = 0; i < 32; ++i) x[t][i] = -INFINITY;
            if (t >= nt) continue;
            if (!failed) failed = !mbar_wait(smem_u32(&sm.b.s_full[t]), 0, ctx, abort);
            failed = __any_sync(0xffffffffu, failed);  // tcgen05.ld is warp-collective
            if (failed || vmask[t] == 0u) continue;    // no entry among this warp's keys
            tc_fence_after();
            uint32_t sv[32];
            tmem_ld32(tmem + DS_COL + 32u * t + lane_off, sv);
            tc_wait_ld();
            // row (key 32 quarter + lane) -> column lane of the warp's block
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) tb[hh * TB_STRIDE + lane] = __uint_as_float(sv[hh]);
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 f = *reinterpret_cast<const float4 *>(tb + h * TB_STRIDE + 4 * k);
                x[t][4 * k] = f.x;
                x[t][4 * k + 1] = f.y;
                x[t][4 * k + 2] = f.z;
                x[t][4 * k + 3] = f.w;
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                // the key-0 sink bias in raw-score units; invalid entries masked
                const float biased = (zmask[t] >> i) & 1u ? x[t][i] + bias_raw : x[t][i];
                x[t][i] = (vmask[t] >> i) & 1u ? biased : -INFINITY;
            }
            float mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < 32; i += 2)
                mr[(i >> 1) & 3] = max3(mr[(i >> 1) & 3], x[t][i], x[t][i + 1]);
            mt = fmaxf(mt, fmaxf(max3(mr[0], mr[1], mr[2]), mr[3]));
        }
        // raw scores: scale > 0, so the max is taken before scaling
        sm.xmax[quarter][h] = mt * p.scale_l2;
        softmax_bar();
        const float m = fmaxf(fmaxf(sm.xmax[0][h], sm.xmax[1][h]),
                              fmaxf(sm.xmax[2][h], sm.xmax[3][h]));
        const float mu = m == -INFINITY ? 0.0f : m;
        const uint64_t negm2 = f2_pack(-mu, -mu);
        const uint64_t scale2 = f2_pack(p.scale_l2, p.scale_l2);
        uint64_t ls2a = f2_pack(0.f, 0.f), ls2b = ls2a;
#pragma unroll
        for (int t = 0; t < DT_MAX; ++t) {
            if (t >= nt) continue;
            // P^T: head h, keys 32 quarter .. +31 = 64 bytes of one K-major row
            const uint32_t pbase = smem_u32(sm.p[t]) + (uint32_t)(quarter >> 1) * QP_HALF;
            const bool none = vmask[t] == 0u;  // no entry among this warp's keys: P = 0
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint32_t w[4] = {0u, 0u, 0u, 0u};
                if (!none) {
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const int i = 8 * u + 2 * e2;
                    float a0, a1;
                    f2_unpack(f2_fma(f2_pack(x[t][i], x[t][i + 1]), scale2, negm2), a0, a1);
                    a0 = ex2(a0);
                    a1 = ex2(a1);
                    if (e2 & 1) ls2b = f2_add(ls2b, f2_pack(a0, a1));
                    else ls2a = f2_add(ls2a, f2_pack(a0, a1));
                    w[e2] = pack_bf16x2(a0, a1);
                }
                }
                const uint32_t addr = pbase + sw128_offset(h, (quarter & 1) * 4 + u);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]),
                             "r"(w[1]), "r"(w[2]), "r"(w[3])
                             : "memory");
            }
        }
        if (nt > 0) {  // every tile's P at once: one proxy fence
            fence_proxy_async_smem();  // P is read by the tensor core
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.b.p_full));
        }
        {
            float a0, a1;
            f2_unpack(f2_add(ls2a, ls2b), a0, a1);
            sm.lpart[quarter][h] = a0 + a1;
        }
        softmax_bar();  // lpart complete
        const float l_h = (sm.lpart[0][h] + sm.lpart[1][h]) + (sm.lpart[2][h] + sm.lpart[3][h]);
        const int hs = NH / C;
        // ---- (m, l) of every head to every CTA of the cluster, while P V runs
        cluster_wait_acquire();  // every CTA of the cluster is running, its barriers set up
        if (quarter == 0) {  // head h = lane
            const uint32_t am = smem_u32(&sm.stat_m[crank][h]), al = smem_u32(&sm.stat_l[crank][h]);
            const uint32_t sbar = smem_u32(&sm.b.stats_full);
            for (int r = 0; r < C; ++r) {
                st_async(dsmem_addr(am, (uint32_t)r), m, dsmem_addr(sbar, (uint32_t)r));
                st_async(dsmem_addr(al, (uint32_t)r), l_h, dsmem_addr(sbar, (uint32_t)r));
            }
        }
        // merged max and denominator per head (null-logit sink added once),
        // lse, and this CTA's weight; a CTA that gave up sends nothing and the
        // wait then runs out
        const bool got_stats = mbar_wait(smem_u32(&sm.b.stats_full), 0, ctx, abort);
        if (quarter == 0) {
            const float sink = sm.sink_l2[h];
            float mx = sink;
            for (int c = 0; c < C; ++c) mx = fmaxf(mx, sm.stat_m[c][h]);
            float L = 0.f;
            if (mx != -INFINITY && got_stats) {
                L = ex2(sink - mx);  // 0 without a null-logit sink
                for (int c = 0; c < C; ++c) {
                    const float mc = sm.stat_m[c][h];
                    if (mc != -INFINITY) L += sm.stat_l[c][h] * ex2(mc - mx);
                }
            }
            sm.wself[h] = (m != -INFINITY && L > 0.f) ? ex2(m - mx) * __frcp_rn(L) : 0.f;
            sm.lse_h[h] = L > 0.f ? (mx + __log2f(L)) * LN2 : -INFINITY;
        }
        if (nt > 0) {
            if (!failed) failed = !mbar_wait(smem_u32(&sm.b.o_full), 0, ctx, abort);
            failed = __any_sync(0xffffffffu, failed);
        }
        softmax_bar();  // wself complete
        // O^T row d = 32 quarter + lane: 32 heads, times this CTA's weights
        uint32_t ov[32];
        if (nt > 0 && !failed) {
            tc_fence_after();
            tmem_ld32(tmem + DO_COL + lane_off, ov);
            tc_wait_ld();
        } else {
#pragma unroll
            for (int hh = 0; hh < 32; ++hh) ov[hh] = 0u;  // nothing seen: a zero partial
        }
        tc_fence_before();  // the TMEM loads above come before the dealloc below
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 w = *reinterpret_cast<const float4 *>(&sm.wself[4 * k]);
            ov[4 * k] = __float_as_uint(__uint_as_float(ov[4 * k]) * w.x);
            ov[4 * k + 1] = __float_as_uint(__uint_as_float(ov[4 * k + 1]) * w.y);
            ov[4 * k + 2] = __float_as_uint(__uint_as_float(ov[4 * k + 2]) * w.z);
            ov[4 * k + 3] = __float_as_uint(__uint_as_float(ov[4 * k + 3]) * w.w);
        }
        // the Q copies have landed (a CTA without tiles never waited for them)
        asm volatile("cp.async.wait_all;" ::: "memory");
        // ---- weighted O^T rows: heads of CTA r go to CTA r's shared memory
        {
            const int d = quarter * 32 + lane;
            const uint32_t row = smem_u32(sm.recv) +
                                 (uint32_t)(((int)crank * HD + d) * (hs + 4)) * 4u;
            const uint32_t rbar = smem_u32(&sm.b.recv_full);
#pragma unroll
            for (int h4 = 0; h4 < NH; h4 += 4) {
                const int r = h4 / hs, j0 = h4 - r * hs;
                st_async4(dsmem_addr(row + (uint32_t)j0 * 4u, (uint32_t)r), __uint_as_float(ov[h4]),
                          __uint_as_float(ov[h4 + 1]), __uint_as_float(ov[h4 + 2]),
                          __uint_as_float(ov[h4 + 3]), dsmem_addr(rbar, (uint32_t)r));
            }
        }

        // ---- o of heads [h0, h0 + hs): the sum of what the cluster sent
        const int tid = threadIdx.x;
        const int h0 = (int)crank * hs;
        const bool got = mbar_wait(smem_u32(&sm.b.recv_full), 0, ctx, abort);
        const float *rrow = sm.recv + tid * (hs + 4);
        __nv_bfloat16 *ob = p.o + (size_t)bm * NH * HD + tid;
        if (got) {
            for (int j0 = 0; j0 < hs; j0 += 4) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int c = 0; c < C; ++c) {
                    const float4 v = *reinterpret_cast<const float4 *>(rrow + c * HD * (hs + 4) + j0);
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
                ob[(size_t)(h0 + j0) * HD] = __float2bfloat16_rn(acc.x);
                ob[(size_t)(h0 + j0 + 1) * HD] = __float2bfloat16_rn(acc.y);
                ob[(size_t)(h0 + j0 + 2) * HD] = __float2bfloat16_rn(acc.z);
                ob[(size_t)(h0 + j0 + 3) * HD] = __float2bfloat16_rn(acc.w);
            }
            if (tid < hs && p.lse) p.lse[(size_t)bm * NH + h0 + tid] = sm.lse_h[h0 + tid];
        }
        // second cluster phase: this CTA has received everything it expects
        cluster_arrive_relaxed();
        cluster_wait_acquire();  // ... and so has every other CTA of the cluster
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, DEC_TMEM_COLS);
    }
}

}  // namespace

int sparse_decode_cluster(int B, int M, int K, int sm_count) {
    const long long items = (long long)B * M;
    if (items <= 0 || items > sm_count) return 0;
    int c = 1;
    while (c * 2 <= MAX_CLUSTER && items * c * 2 <= sm_count) c *= 2;
    if ((K + c - 1) / c > DT_MAX * R) return 0;
    return c;
}

cudaError_t launch_sparse_decode(const SparseArgs &a, int C, const DevInfo &dev, cudaStream_t s) {
    const bool fp8 = a.kv == nullptr;
    DecParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.kv = static_cast<const __nv_bfloat16 *>(a.kv);
    p.kv_nope = a.kv_nope;
    p.kv_rope = static_cast<const __nv_bfloat16 *>(a.kv_rope);
    p.kv_scale = a.kv_scale;
    p.idx = a.idx;
    p.sinks = a.sinks;
    p.sink_mode = a.sink_mode;
    p.scale_l2 = a.scale * LOG2E;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.lse = a.lse;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.C = C;
    p.seg = (a.K + C - 1) / C;
    const size_t smem = sizeof(DecSmem);
    auto kernel = fp8 ? sparse_decode_kernel<true> : sparse_decode_kernel<false>;
    cudaError_t e = ensure_smem_attr((const void *)kernel, smem, dev);
    if (e != cudaSuccess) return e;
    const DevCtx ctx = make_ctx(dev);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(a.B * a.M * C));
    cfg.blockDim = dim3(DEC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (verbose())
        fprintf(stderr, "sattn: sparse_decode_kernel<%s> grid=%d cluster=%d block=%d smem=%zu seg=%d\n",
                fp8 ? "fp8" : "bf16", a.B * a.M * C, C, DEC_THREADS, smem, p.seg);
    return cudaLaunchKernelEx(&cfg, kernel, p, ctx);
}

}  // namespace sattn
