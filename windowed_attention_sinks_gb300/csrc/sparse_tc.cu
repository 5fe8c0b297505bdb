// Gathered attention over one shared KV head on tcgen05 ("DeepSeek-V4 CSA/HCA
// walkthrough", sections 4.1-4.4: topk_idxs loaded per tile, invalid -1
// entries masked, the gathered KV rows staged in shared memory so the
// scores and the output become dense contractions, a null-logit sink in the
// softmax denominator).
//
// Every query head reads the same gathered rows, so the roles of the
// operands are swapped to fill the 128-row MMA: with R = 128 gathered rows,
//   S^T [R x H]  = KV [R x d] . Q^T          (A = KV tile, K-major)
//   O^T [d x H] += KV^T [d x R] . P^T        (A = the same tile, MN-major)
// Both accumulators live in TMEM (H = 32 columns each).
//
// A work item is one query's index list (or one slice of it when short lists
// are split across CTAs). A persistent grid of one CTA per SM runs two
// independent slots, each with its own shared memory, TMEM columns,
// barriers and item stream. Each slot is warp-specialised:
//   gather warp   reads the list 128 entries ahead and compacts the valid
//                 ones (0 <= idx < N) into tiles of up to 128 rows, so -1
//                 entries cost no MMA work; the listed rows are copied with
//                 16-byte cp.async into a 128B-swizzled K-major tile (rows
//                 past the tile's count are zero-filled); two stages, each
//                 completed on an mbarrier.
//   MMA thread    S^T of tile t into one of two S buffers, then
//                 O^T += KV^T P^T for tile t-1, so the tensor core works on
//                 the next scores while the softmax runs.
//   4 warps       softmax: S^T is transposed through shared memory so that
//                 four threads own one head (two shuffles per reduction);
//                 running max / sum per head in the log2 domain, P (bf16)
//                 to a double-buffered shared tile; epilogue O^T / l.
// Summation order differs from list order (compaction); softmax does not
// depend on it. With more than one split the normalised partial output and
// its lse go to the workspace and are merged through their log-sum-exp
// (sinks added once).
#include <math.h>
#include <stdio.h>

#include "common.cuh"
#include "internal.h"

namespace sattn {
namespace {

constexpr int R = 128;         // gathered rows per tile
constexpr int HD = 128;        // head dim
constexpr int NH = 32;         // query heads handled by the kernel
constexpr int NSLOT = 2;         // independent item streams per CTA
constexpr int GATHER_WARPS = 4;  // per slot; one warp issues cp.async at ~10 B/clk at most
constexpr int SLOT_CTRL = GATHER_WARPS + 1;  // gather warps + the MMA warp of a slot
constexpr int NTHREADS = 32 * NSLOT * (SLOT_CTRL + 4);
constexpr int SOFTMAX_THREADS = 128;
constexpr uint32_t KV_TILE = R * HD * 2;   // 32 KB
constexpr uint32_t KV_HALF = KV_TILE / 2;  // 64 columns of d
constexpr uint32_t QP_HALF = NH * 128;     // 4 KB: one 64-column half of Q or P
// Transpose buffer: head h, row quarter q, entry i at h * SB_HEAD + q * SB_PART + i.
// Row writes (fixed h) are consecutive; the 16-byte reads of the 8 threads
// sharing an LDS.128 phase fall in distinct bank groups (39h + 10q mod 8).
constexpr int SB_HEAD = 156, SB_PART = 40;
constexpr float TAU = 8.0f;
constexpr int MAX_SPLITS = 64;
constexpr uint32_t SLOT_COLS = 128;  // TMEM per slot: S^T[2] (32 each), O^T (32)
constexpr uint32_t TMEM_COLS = SLOT_COLS * NSLOT;
constexpr uint32_t S_COL = 0, O_COL = 64;

struct SlotBars {
    uint64_t q_full, q_empty;
    uint64_t kv_full[2], kv_empty[2];
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full[2], p_empty[2];
    uint64_t pv_done, o_full, o_empty, drain;
};

// Shared memory of one slot; tiles first so that they stay 1024-byte aligned.
struct alignas(1024) SlotSmem {
    uint8_t kv[2][KV_TILE];
    uint8_t q[2 * QP_HALF];
    uint8_t p[2][2 * QP_HALF];
    float sbuf[NH * SB_HEAD];
    // compacted entries of the tile in each stage (-1 past the count), one
    // copy per gather warp; the softmax reads copy 0
    int idx[GATHER_WARPS][2][R];
    int tile_cnt[2];    // rows that hold entries
    int tile_last[2];   // the tile in this stage ends its item
    float alpha[NH];
    float m[NH];
    float l[NH];
    SlotBars b;
};

struct alignas(1024) Smem {
    SlotSmem slot[NSLOT];
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(Smem) <= 227 * 1024, "shared memory of one CTA");

struct SpParams {
    const __nv_bfloat16 *q, *kv;
    const int32_t *idx;
    const float *sinks;
    int sink_mode;
    float scale_l2;
    __nv_bfloat16 *o;
    float *lse;
    int B, M, N, K;
    int splits, split_len;  // entries per split (multiple of R)
    float *o_part, *lse_part;  // workspace (splits > 1)
};

constexpr uint32_t IDESC_S = idesc_bf16_f32(128, NH, 0, 0);
constexpr uint32_t IDESC_O = idesc_bf16_f32(128, NH, 1, 0);

__device__ __forceinline__ uint64_t desc_k(uint32_t base, int kk, uint32_t half_stride) {
    return smem_desc_sw128(base + (uint32_t)(kk >> 2) * half_stride + (uint32_t)(kk & 3) * 32u,
                           16u, 1024u);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int kk) {
    return smem_desc_sw128(base + (uint32_t)kk * 2048u, KV_HALF, 1024u);
}

// 2-D tiled TMA load (x = column, y = row), completion on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
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

// Barrier among the slot's four softmax warps (named barrier 1 + slot) that
// also returns whether any thread's predicate was true.
__device__ __forceinline__ int softmax_sync_or(int slot, int pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.s32 p, %2, 0;\n\t"
        "bar.red.or.pred q, %1, %3, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(1 + slot), "r"(pred), "r"(SOFTMAX_THREADS)
        : "memory");
    return r;
}

struct ItemInfo {
    int bm, split, b, e_begin, e_end;
};

__device__ __forceinline__ ItemInfo item_info(const SpParams &p, int item) {
    ItemInfo it;
    it.bm = item / p.splits;
    it.split = item % p.splits;
    it.b = it.bm / p.M;
    it.e_begin = it.split * p.split_len;
    it.e_end = min(p.K, it.e_begin + p.split_len);
    return it;
}

// ------------------------------------------------------------------ gather warp

// Every gather warp of a slot compacts the same index lists (the result is
// deterministic, so no warp waits for another); warp g copies rows
// 64g .. 64g+63 of each tile. Warp 0 also loads Q and publishes the tile's
// indices, count and last flag for the MMA and softmax roles.
__device__ void gather_role(const SpParams &p, const CUtensorMap *tq, SlotSmem &sm,
                            volatile int *abort, int g, int first, int stride,
                            const DevCtx &ctx) {
    SlotBars &b = sm.b;
    const bool lead = g == 0;
    const int lane = threadIdx.x & 31;
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int nitems = p.B * p.M * p.splits;
    int qi = 0, gt = 0;  // items started, tiles issued
    bool ok = true, bad = false;
    // Row copies: lane = (hi, unit) copies 16-byte unit `unit` of rows 2i + hi.
    // In the 128B swizzle, unit u of row r sits at r * 128 + ((u ^ (r & 7)) << 4),
    // and (unit & 7) ^ (r & 7) = ((unit & 7) ^ hi) ^ (2i & 6): four lane offsets
    // cover every i.
    const int hi = lane >> 4, unit = lane & 15;
    uint32_t dofs[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
        dofs[c] = (uint32_t)(unit >> 3) * KV_HALF + (uint32_t)hi * 128u +
                  ((((uint32_t)(unit & 7) ^ (uint32_t)hi) ^ (uint32_t)(2 * c)) << 4);
    // warp-uniform bounded wait (lane 0 polls)
    auto wwait = [&](uint64_t &bar, int parity) -> bool {
        int r = 1;
        if (lane == 0) r = mbar_wait(smem_u32(&bar), (uint32_t)parity, ctx, abort) ? 1 : 0;
        r = __shfl_sync(0xffffffffu, r, 0);
        __syncwarp();
        return r != 0;
    };
    // pull an item's slice of the index list into L2 ahead of its use
    auto prefetch_list = [&](int item) {
        if (item >= nitems) return;
        const ItemInfo ni = item_info(p, item);
        const char *base = reinterpret_cast<const char *>(p.idx + (size_t)ni.bm * p.K + ni.e_begin);
        const int bytes = (ni.e_end - ni.e_begin) * 4;
        for (int off = lane * 128; off < bytes; off += 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(base + off));
    };
    if (lead) {
        if (lane == 0) prefetch_tmap(tq);
        prefetch_list(first);
    }
    for (int item = first; ok && item < nitems; item += stride) {
        const ItemInfo it = item_info(p, item);
        const int32_t *list = p.idx + (size_t)it.bm * p.K;
        const __nv_bfloat16 *kvb = p.kv + (size_t)it.b * p.N * HD + unit * 8;
        if (lead) {
            prefetch_list(item + stride);
            // Q rows of the query (32 heads x 256 B): two 64-column boxes
            if (qi >= 1 && !wwait(b.q_empty, (qi - 1) & 1)) { ok = false; break; }
            if (lane == 0) {
                const uint32_t bar = smem_u32(&b.q_full);
                mbar_arrive_expect_tx(bar, 2 * QP_HALF);
                tma_load_2d(smem_u32(sm.q), tq, bar, 0, it.bm * NH);
                tma_load_2d(smem_u32(sm.q) + QP_HALF, tq, bar, 64, it.bm * NH);
            }
            ++qi;
        }
        auto acquire = [&]() -> bool {  // the stage of tile gt is free
            const int use = gt >> 1;
            return use == 0 || wwait(b.kv_empty[gt & 1], (use - 1) & 1);
        };
        // Issue the tile in stage gt & 1 holding `pos` compacted rows; rows past
        // the count are zero-filled so that P V stays finite.
        auto close_tile = [&](int pos, bool last) {
            const int st = gt & 1;
            int *ids = sm.idx[g][st];
            for (int r = pos + lane; r < R; r += 32) ids[r] = -1;
            if (lead && lane == 0) {
                sm.tile_cnt[st] = pos;
                sm.tile_last[st] = last ? 1 : 0;
            }
            __syncwarp();
            const uint32_t kv_s = smem_u32(sm.kv[st]);
            constexpr int PAIRS = R / 2 / GATHER_WARPS;  // row pairs per warp (multiple of 4)
#pragma unroll 16
            for (int i2 = 0; i2 < PAIRS; ++i2) {
                const int i = PAIRS * g + i2;
                const int e = ids[2 * i + hi];
                cp_async16(kv_s + dofs[i2 & 3] + (uint32_t)i * 256u,
                           kvb + (size_t)(e >= 0 ? e : 0) * HD, e >= 0 ? 16u : 0u);
            }
            const uint32_t bar = smem_u32(&b.kv_full[st]);
            cp_async_arrive(bar);
            __syncwarp();
            if (lead && lane == 0) mbar_arrive(bar);  // publishes idx, tile_cnt, tile_last
            ++gt;
        };
        auto load = [&](int (&v)[4], int e0) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int e = e0 + 32 * c + lane;
                int x = e < it.e_end ? __ldg(list + e) : -1;
                if (x < -1 || x >= p.N) {
                    bad = true;
                    x = -1;
                }
                v[c] = x;
            }
        };
        int pos = 0;
        // compact one group of 128 entries into the open tile
        auto compact = [&](const int (&v)[4]) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const bool valid = v[c] >= 0;
                const uint32_t bal = __ballot_sync(0xffffffffu, valid);
                const int cnt = __popc(bal);
                if (cnt == 0) continue;
                if (pos + cnt > R) {  // does not fit: issue this tile, open the next
                    __syncwarp();
                    close_tile(pos, false);
                    if (!acquire()) {
                        ok = false;
                        return;
                    }
                    pos = 0;
                }
                if (valid) sm.idx[g][gt & 1][pos + __popc(bal & lt_mask)] = v[c];
                pos += cnt;
            }
        };
        if (!acquire()) { ok = false; break; }
        // two groups of indices in flight: each is loaded one group ahead of use
        int va[4], vb[4];
        load(va, it.e_begin);
        load(vb, it.e_begin + R);
        for (int e0 = it.e_begin; ok && e0 < it.e_end; e0 += 2 * R) {
            compact(va);
            load(va, e0 + 2 * R);
            if (!ok || e0 + R >= it.e_end) break;
            compact(vb);
            load(vb, e0 + 3 * R);
        }
        if (!ok) break;
        __syncwarp();
        close_tile(pos, true);  // an item without valid entries still gets one (empty) tile
    }
    if (bad && lead) record_error(ctx, DEVERR_INDEX);
    // copies in flight land before the CTA may exit (on the normal path all of
    // them were consumed already; this matters after an abort)
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (lead && lane == 0 && qi >= 1) {
        int zero = 0;
        mbar_wait(smem_u32(&b.q_full), (qi - 1) & 1, ctx, &zero);
    }
    __syncwarp();
}

// ------------------------------------------------------------------ MMA thread

__device__ void mma_role(const SpParams &p, SlotSmem &sm, volatile int *abort, uint32_t tmem,
                         int first, int stride, const DevCtx &ctx) {
    SlotBars &b = sm.b;
    const int nitems = p.B * p.M * p.splits;
    const uint32_t q_base = smem_u32(sm.q), t_o = tmem + O_COL;
    int qi = 0, gt = 0;
    bool ok = true;
    for (int item = first; ok && item < nitems; item += stride) {
        if (!mbar_wait(smem_u32(&b.q_full), qi & 1, ctx, abort)) break;
        const int gt0 = gt;
        // O^T += KV^T P^T for tile jj of this item
        auto issue_pv = [&](int jj) -> bool {
            const int t = gt0 + jj, st = t & 1;
            if (!mbar_wait(smem_u32(&b.p_full[st]), (t >> 1) & 1, ctx, abort)) return false;
            if (jj == 0 && qi >= 1 &&
                !mbar_wait(smem_u32(&b.o_empty), (qi - 1) & 1, ctx, abort))
                return false;
            tc_fence_after();
            const uint32_t kv_s = smem_u32(sm.kv[st]), p_s = smem_u32(sm.p[st]);
#pragma unroll
            for (int kk = 0; kk < R / 16; ++kk)
                tc_mma_f16(t_o, desc_mn(kv_s, kk), desc_k(p_s, kk, QP_HALF), IDESC_O,
                           (jj > 0 || kk > 0) ? 1u : 0u);
            tc_commit(smem_u32(&b.kv_empty[st]));
            tc_commit(smem_u32(&b.p_empty[st]));
            tc_commit(smem_u32(&b.pv_done));
            return true;
        };
        int j = 0;
        for (bool last = false; !last; ++j) {
            const int t = gt0 + j, st = t & 1, use = t >> 1;
            if (use >= 1 && !mbar_wait(smem_u32(&b.s_empty[st]), (use - 1) & 1, ctx, abort)) {
                ok = false;
                break;
            }
            if (!mbar_wait(smem_u32(&b.kv_full[st]), use & 1, ctx, abort)) { ok = false; break; }
            tc_fence_after();
            last = sm.tile_last[st] != 0;
            const uint32_t kv_s = smem_u32(sm.kv[st]);
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk)
                tc_mma_f16(tmem + S_COL + 32u * st, desc_k(kv_s, kk, KV_HALF),
                           desc_k(q_base, kk, QP_HALF), IDESC_S, kk > 0 ? 1u : 0u);
            tc_commit(smem_u32(&b.s_full[st]));
            if (last) tc_commit(smem_u32(&b.q_empty));
            if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
        }
        if (!ok || !issue_pv(j - 1)) break;
        tc_commit(smem_u32(&b.o_full));
        gt = gt0 + j;
        ++qi;
    }
    // every MMA issued so far completes before TMEM is released
    tc_commit(smem_u32(&b.drain));
    int zero = 0;
    mbar_wait(smem_u32(&b.drain), 0, ctx, &zero);
}

// ------------------------------------------------------------------ softmax warps

__device__ void softmax_role(const SpParams &p, SlotSmem &sm, volatile int *abort, int slot,
                             uint32_t tmem, int first, int stride, const DevCtx &ctx) {
    SlotBars &b = sm.b;
    // tid: position in the slot's softmax group (head ownership, stores);
    // a warp may only access TMEM lanes 32 * (warp id mod 4) .. +31, so this
    // thread's S^T row / O^T row (head-dim index) is 32 * quarter + lane
    const int tid = threadIdx.x - 32 * NSLOT * SLOT_CTRL - SOFTMAX_THREADS * slot;
    const int lane = threadIdx.x & 31, quarter = (threadIdx.x >> 5) & 3;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_o = tmem + O_COL + lane_off;
    const int h = tid >> 2, part = tid & 3;  // head owned (with 3 siblings) and its row quarter
    const bool key0 = p.sink_mode == 1;
    const float sink_h = p.sinks ? __ldg(p.sinks + h) * LOG2E : 0.0f;
    const float bias_raw = key0 ? sink_h / p.scale_l2 : 0.0f;
    const uint64_t scale2 = f2_pack(p.scale_l2, p.scale_l2);
    const bool null_sink = p.sink_mode == 2 && p.splits == 1;
    const int nitems = p.B * p.M * p.splits;
    int qi = 0, gt = 0;
    // A failed wait is carried to the next barrier, whose OR makes the exit
    // uniform over the four warps (no thread is left behind at a barrier).
    bool failed = false;
    for (int item = first; item < nitems; item += stride) {
        const ItemInfo it = item_info(p, item);
        float m_run = null_sink ? sink_h : -INFINITY;
        float l_run = null_sink ? 1.0f : 0.0f;
        const int gt0 = gt;
        int j = 0;
        for (bool last = false; !last; ++j) {
            const int t = gt0 + j, st = t & 1, use = t >> 1;
            // S^T of this tile -> transpose buffer; the tile's indices were
            // published with its gather; P buffer st was last read by P V of tile t-2
            if (!failed) {
                failed = !mbar_wait(smem_u32(&b.s_full[st]), use & 1, ctx, abort) ||
                         !mbar_wait(smem_u32(&b.kv_full[st]), use & 1, ctx, abort) ||
                         (use >= 1 &&
                          !mbar_wait(smem_u32(&b.p_empty[st]), (use - 1) & 1, ctx, abort));
            }
            failed = __any_sync(0xffffffffu, failed);  // tcgen05.ld is warp-collective
            if (!failed) {
                tc_fence_after();
                uint32_t sv[32];
                tmem_ld32(tmem + S_COL + 32u * st + lane_off, sv);
                tc_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&b.s_empty[st]));
#pragma unroll
                for (int hh = 0; hh < NH; ++hh)
                    sm.sbuf[hh * SB_HEAD + quarter * SB_PART + lane] = __uint_as_float(sv[hh]);
            }
            if (softmax_sync_or(slot, failed)) { failed = true; break; }
            last = sm.tile_last[st] != 0;
            // head h over rows part*32 .. part*32+31 (raw scores; scale > 0, so
            // the max is taken before scaling)
            float x[32];
            {
                const float *src = &sm.sbuf[h * SB_HEAD + part * SB_PART];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float4 f = *reinterpret_cast<const float4 *>(src + 4 * k);
                    x[4 * k] = f.x;
                    x[4 * k + 1] = f.y;
                    x[4 * k + 2] = f.z;
                    x[4 * k + 3] = f.w;
                }
            }
            if (key0) {  // the sink bias on the logit of key 0, in raw-score units
                const int *ids = &sm.idx[0][st][part * 32];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int4 e = *reinterpret_cast<const int4 *>(ids + 4 * k);
                    x[4 * k] += e.x == 0 ? bias_raw : 0.f;
                    x[4 * k + 1] += e.y == 0 ? bias_raw : 0.f;
                    x[4 * k + 2] += e.z == 0 ? bias_raw : 0.f;
                    x[4 * k + 3] += e.w == 0 ? bias_raw : 0.f;
                }
            }
            const int nvalid = sm.tile_cnt[st] - part * 32;  // rows of this quarter holding entries
            if (nvalid < 32) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i >= nvalid) x[i] = -INFINITY;
            }
            float mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < 32; i += 2) mr[(i >> 1) & 3] = max3(mr[(i >> 1) & 3], x[i], x[i + 1]);
            float mt = fmaxf(max3(mr[0], mr[1], mr[2]), mr[3]);
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
            mt *= p.scale_l2;
            const bool upd = mt > m_run + TAU;
            float alpha = 1.0f;
            if (upd) {
                alpha = (m_run == -INFINITY) ? 0.0f : ex2(m_run - mt);
                l_run *= alpha;
                m_run = mt;
            }
            const float mu = m_run == -INFINITY ? 0.0f : m_run;
            const uint64_t negm2 = f2_pack(-mu, -mu);
            uint64_t ls2a = f2_pack(0.f, 0.f), ls2b = ls2a;
            const uint32_t pbase = smem_u32(sm.p[st]) + (uint32_t)(part >> 1) * QP_HALF;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint32_t w[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const int i = 8 * u + 2 * e2;
                    float a0, a1;
                    f2_unpack(f2_fma(f2_pack(x[i], x[i + 1]), scale2, negm2), a0, a1);
                    a0 = ex2(a0);
                    a1 = ex2(a1);
                    if (e2 & 1) ls2b = f2_add(ls2b, f2_pack(a0, a1));
                    else ls2a = f2_add(ls2a, f2_pack(a0, a1));
                    w[e2] = pack_bf16x2(a0, a1);
                }
                const uint32_t addr = pbase + sw128_offset(h, (part & 1) * 4 + u);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]),
                             "r"(w[1]), "r"(w[2]), "r"(w[3])
                             : "memory");
            }
            float ls;
            {
                float a0, a1;
                f2_unpack(f2_add(ls2a, ls2b), a0, a1);
                ls = a0 + a1;
            }
            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
            l_run += ls;
            if (part == 0) sm.alpha[h] = alpha;
            // also orders this tile's transpose-buffer reads before the next tile's writes
            const int any_upd = softmax_sync_or(slot, upd && j >= 1);
            if (any_upd) {  // rescale O^T columns (heads) whose max moved
                // P V of the previous tile must be complete (the one before it
                // is: P buffer st was free)
                failed = __any_sync(0xffffffffu,
                                    !mbar_wait(smem_u32(&b.pv_done), (t - 1) & 1, ctx, abort));
                if (!failed) {
                    tc_fence_after();
                    uint32_t ov[32];
                    tmem_ld32(t_o, ov);
                    tc_wait_ld();
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh)
                        ov[hh] = __float_as_uint(__uint_as_float(ov[hh]) * sm.alpha[hh]);
                    tmem_st32(t_o, ov);
                    tc_wait_st();
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&b.p_full[st]));
        }
        gt = gt0 + j;
        // epilogue: every P V of the item is complete once o_full fires; the
        // wait comes before the barrier so that a failure leaves uniformly
        if (!failed)
            failed = __any_sync(0xffffffffu, !mbar_wait(smem_u32(&b.o_full), qi & 1, ctx, abort));
        if (part == 0) {  // per head: 1 / l and the lse (natural log)
            sm.l[h] = l_run > 0.f ? 1.0f / l_run : 0.f;
            sm.m[h] = l_run > 0.f ? (m_run + log2f(l_run)) * LN2 : -INFINITY;
        }
        if (softmax_sync_or(slot, failed)) break;
        ++qi;
        tc_fence_after();
        uint32_t ov[32];
        tmem_ld32(t_o, ov);
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&b.o_empty));
        // O / l straight from registers: for each head the 128 threads of the
        // group write 128 consecutive values of d (coalesced)
        const int d = quarter * 32 + lane;
        const size_t rows = (size_t)p.B * p.M * NH;
        if (p.splits == 1) {
            __nv_bfloat16 *ob = p.o + (size_t)it.bm * NH * HD + d;
#pragma unroll
            for (int hh = 0; hh < NH; ++hh)
                ob[hh * HD] = __float2bfloat16_rn(__uint_as_float(ov[hh]) * sm.l[hh]);
            if (p.lse && tid < NH) p.lse[(size_t)it.bm * NH + tid] = sm.m[tid];
        } else {
            float *op = p.o_part + ((size_t)it.split * rows + (size_t)it.bm * NH) * HD + d;
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) op[hh * HD] = __uint_as_float(ov[hh]) * sm.l[hh];
            if (tid < NH) p.lse_part[(size_t)it.split * rows + (size_t)it.bm * NH + tid] = sm.m[tid];
        }
        // sm.l / sm.m are rewritten only after two more barriers
    }
}

__global__ void __launch_bounds__(NTHREADS, 1)
sparse_tc_kernel(const __grid_constant__ CUtensorMap tq, const SpParams p, const DevCtx ctx) {
    extern __shared__ __align__(1024) uint8_t dsmem[];
    Smem &all = *reinterpret_cast<Smem *>(dsmem);
    const int warp = threadIdx.x >> 5;
    if (smem_u32(dsmem) & 1023u) {  // the 128B swizzle needs an aligned base
        if (threadIdx.x == 0) record_error(ctx, DEVERR_LAYOUT);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            SlotBars &b = all.slot[s].b;
            for (int i = 0; i < 2; ++i) {
                mbar_init(smem_u32(&b.kv_full[i]), 32 * GATHER_WARPS + 1);  // copies + publish
                mbar_init(smem_u32(&b.kv_empty[i]), 1);
                mbar_init(smem_u32(&b.s_full[i]), 1);
                mbar_init(smem_u32(&b.s_empty[i]), 4);
                mbar_init(smem_u32(&b.p_full[i]), 4);
                mbar_init(smem_u32(&b.p_empty[i]), 1);
            }
            mbar_init(smem_u32(&b.q_full), 1);
            mbar_init(smem_u32(&b.q_empty), 1);
            mbar_init(smem_u32(&b.pv_done), 1);
            mbar_init(smem_u32(&b.o_full), 1);
            mbar_init(smem_u32(&b.o_empty), 4);
            mbar_init(smem_u32(&b.drain), 1);
        }
        all.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&all.tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the merge of split partials may be scheduled now; it waits for this
    // grid to finish before reading anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // slot s: warps SLOT_CTRL * s + g (gather g), SLOT_CTRL * s + GATHER_WARPS
    // (MMA), then NSLOT * SLOT_CTRL + 4s .. +3 (softmax: four consecutive warps
    // cover the four TMEM lane quarters)
    const int ctrl = NSLOT * SLOT_CTRL;
    const int slot = warp < ctrl ? warp / SLOT_CTRL : (warp - ctrl) >> 2;
    const uint32_t tmem = all.tmem_base + (uint32_t)slot * SLOT_COLS;
    const int first = blockIdx.x * NSLOT + slot, stride = gridDim.x * NSLOT;
    SlotSmem &sm = all.slot[slot];
    if (warp < ctrl) {
        const int role = warp % SLOT_CTRL;
        if (role < GATHER_WARPS) {
            gather_role(p, &tq, sm, &all.abort, role, first, stride, ctx);
        } else {
            if ((threadIdx.x & 31) == 0) mma_role(p, sm, &all.abort, tmem, first, stride, ctx);
            __syncwarp();
        }
    } else {
        softmax_role(p, sm, &all.abort, slot, tmem, first, stride, ctx);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(all.tmem_base, TMEM_COLS);
    }
}

int choose_splits(int B, int M, int K, int sm_count) {
    const int items = B * M;
    const int max_split = (K + R - 1) / R;
    // two items run per SM; aim for one round of items
    if (max_split <= 1 || items >= NSLOT * sm_count) return 1;
    int s = (NSLOT * sm_count) / items;
    if (s > max_split) s = max_split;
    if (s > MAX_SPLITS) s = MAX_SPLITS;
    return s < 1 ? 1 : s;
}

// Workspace needed by a given number of splits.
size_t split_bytes(int B, int M, int H, int d, int splits) {
    if (splits <= 1) return 0;
    const size_t rows = (size_t)B * M * H;
    const size_t o = (size_t)splits * rows * d * sizeof(float);
    return ((o + 255) & ~(size_t)255) + (size_t)splits * rows * sizeof(float);
}

}  // namespace

size_t sparse_tc_workspace_bytes(int B, int M, int H, int d, int K) {
    // enough for any split count the launcher may choose on any GPU (<= 256 SMs)
    return split_bytes(B, M, H, d, choose_splits(B, M, K, 256));
}

cudaError_t launch_sparse_tc(const SparseArgs &a, const DevInfo &dev, cudaStream_t s) {
    if (a.H != NH || a.d != HD) return launch_sparse_simt(a, dev, s);
    SpParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.kv = static_cast<const __nv_bfloat16 *>(a.kv);
    p.idx = a.idx;
    p.sinks = a.sinks;
    p.sink_mode = a.sink_mode;
    p.scale_l2 = a.scale * LOG2E;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.lse = a.lse;
    p.B = a.B;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    int splits = a.workspace ? choose_splits(a.B, a.M, a.K, dev.sm_count) : 1;
    while (splits > 1 && split_bytes(a.B, a.M, a.H, a.d, splits) > a.workspace_bytes) --splits;
    const int tiles = (a.K + R - 1) / R;
    const int tiles_per_split = splits > 1 ? (tiles + splits - 1) / splits : (tiles > 0 ? tiles : 1);
    splits = splits > 1 ? (tiles + tiles_per_split - 1) / tiles_per_split : 1;
    p.splits = splits;
    p.split_len = tiles_per_split * R;
    const size_t rows = (size_t)a.B * a.M * a.H;
    if (splits > 1) {
        p.o_part = static_cast<float *>(a.workspace);
        const size_t o_bytes = ((size_t)splits * rows * a.d * sizeof(float) + 255) & ~(size_t)255;
        p.lse_part = reinterpret_cast<float *>(static_cast<uint8_t *>(a.workspace) + o_bytes);
    }
    const long long nitems = (long long)a.B * a.M * splits;
    if (nitems > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (nitems == 0) return cudaSuccess;
    const long long want = (nitems + NSLOT - 1) / NSLOT;
    const int grid = (int)(want < dev.sm_count ? want : dev.sm_count);
    // row coordinates of the Q copies are 32-bit
    if ((long long)a.B * a.M * NH > 0x7fffffffLL) return cudaErrorInvalidValue;
    CUtensorMap tq;
    {
        const uint64_t q_dims[2] = {(uint64_t)HD, (uint64_t)a.B * a.M * NH};
        const uint64_t strides[1] = {(uint64_t)HD * 2};
        const uint32_t q_box[2] = {64, (uint32_t)NH};
        if (encode_tensor_map(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(a.q),
                              q_dims, strides, q_box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const size_t smem = sizeof(Smem);
    static bool attr_set[64] = {};
    if (!attr_set[dev.device & 63]) {
        cudaError_t e = cudaFuncSetAttribute(sparse_tc_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set[dev.device & 63] = true;
    }
    DevCtx ctx{dev.err, wait_limit_ns()};
    if (verbose())
        fprintf(stderr, "sattn: sparse_tc_kernel grid=%d block=%d smem=%zu items=%lld splits=%d\n",
                grid, NTHREADS, smem, nitems, splits);
    sparse_tc_kernel<<<grid, NTHREADS, smem, s>>>(tq, p, ctx);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || splits == 1) return e;
    MergeArgs m{p.o_part, p.lse_part, splits, (int64_t)rows, a.d, a.H,
                a.sink_mode == 2 ? a.sinks : nullptr, a.o, a.lse, a.dtype};
    return launch_merge(m, dev, s, true);
}

}  // namespace sattn
