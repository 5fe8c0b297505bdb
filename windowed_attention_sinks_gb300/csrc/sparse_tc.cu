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
//   lead warp     streams the index lists into shared memory (bulk copies
//                 of 256-entry chunks), compacts the valid entries
//                 (0 <= idx < N) into tiles of up to 128 rows, so -1 entries
//                 cost no MMA work, and publishes them through a 5-entry
//                 ring that every reader releases; loads Q (TMA) as soon as
//                 the slot's Q buffer is free.
//   copy warps    copy each tile's rows with 16-byte cp.async into a
//                 128B-swizzled K-major stage (rows past the count are
//                 zero-filled); two stages, completed on an mbarrier. With
//                 an FP8 cache they take the bf16 RoPE half by cp.async and
//                 dequantise the e4m3 half into the stage.
//   MMA thread    issues in readiness order: S^T of the next tile into one
//                 of two S buffers as soon as its rows have landed, and
//                 O^T += KV^T P^T of a tile as soon as its P is written.
//   4 warps       softmax, one head per lane after a per-warp transpose;
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
#include "sparse_layout.cuh"

namespace sattn {
namespace {

using namespace gather;

constexpr int NSLOT = 2;         // independent item streams per CTA
// Per slot: one warp compacts index lists, GATHER_WARPS warps copy rows (one
// warp issues cp.async at ~10 B/clk at most, and index loads queued behind a
// warp's copies would stall its compaction), one warp issues the MMAs.
constexpr int GATHER_WARPS = COPY_WARPS;
constexpr int SLOT_CTRL = GATHER_WARPS + 2;  // control warps of a slot
// Compacted-index ring depth: the lead warp runs up to IDX_RING - 1 tiles
// ahead of the slowest reader of the ring (copy warps, MMA, softmax warps),
// each of which releases an entry (idx_empty) once it has read it.
constexpr int IDX_RING = 5;
// Index lists stream into shared memory in LCHUNK-entry chunks, NLCH in flight.
constexpr int LCHUNK = 256;
constexpr int NLCH = 2;
constexpr int NTHREADS = 32 * NSLOT * (SLOT_CTRL + 4);
constexpr int SOFTMAX_THREADS = 128;
constexpr float TAU = 8.0f;
constexpr int MAX_SPLITS = 64;
constexpr uint32_t SLOT_COLS = 128;  // TMEM per slot: S^T[2] (32 each), O^T (32)
constexpr uint32_t TMEM_COLS = SLOT_COLS * NSLOT;
constexpr uint32_t S_COL = 0, O_COL = 64;

struct SlotBars {
    uint64_t idx_ready[IDX_RING];  // lead gather warp -> copy warps, MMA, softmax
    uint64_t idx_empty[IDX_RING];  // readers -> lead gather warp
    uint64_t lst_full[NLCH];       // index-list chunk landed
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
    float tbuf[4][NH * TB_STRIDE];
    int lst[NLCH][LCHUNK];   // index-list chunks, as stored
    // Ring of compacted tiles: tile t uses entry t % IDX_RING
    int idx[IDX_RING][R];    // entries (-1 past the count)
    int tile_cnt[IDX_RING];  // rows that hold entries
    int tile_last[IDX_RING]; // the tile ends its item
    int tile_row0[IDX_RING]; // first cache row of the tile's request; -1: no more tiles
    float xmax[4][NH];   // per-warp tile maxima (max update only)
    float lpart[4][NH];  // per-warp partial denominators (epilogue)
    float alpha[NH];
    float inv_l[NH];
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
    int B, M, N, K;
    int splits, split_len;  // entries per split (multiple of R)
    float *o_part, *lse_part;  // workspace (splits > 1)
};

// 2-D tiled TMA load (x = column, y = row), completion on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y)
        : "memory");
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

// Copy warp g of a slot copies rows 32 g .. 32 g + 31 of each tile (RowCopier).
// The lead warp loads Q, compacts the index lists into the ring and publishes
// each ring entry to the copy warps, the MMA and the softmax warps
// (idx_ready); after the last tile it publishes an entry with tile_row0 = -1.

// warp-uniform bounded wait (lane 0 polls)
__device__ __forceinline__ bool warp_wait(uint64_t &bar, int parity, const DevCtx &ctx,
                                          volatile int *abort) {
    int r = 1;
    if ((threadIdx.x & 31) == 0) r = mbar_wait(smem_u32(&bar), (uint32_t)parity, ctx, abort) ? 1 : 0;
    r = __shfl_sync(0xffffffffu, r, 0);
    __syncwarp();
    return r != 0;
}

template <bool FP8>
__device__ void gather_helper(const SpParams &p, SlotSmem &sm, volatile int *abort, int g,
                              const DevCtx &ctx) {
    SlotBars &b = sm.b;
    const int lane = threadIdx.x & 31;
    const RowCopier cp(lane);
    const Fp8Copier fc(lane);
    for (int t = 0;; ++t) {
        const int r = t % IDX_RING, st = t & 1, use = t >> 1;
        if (!warp_wait(b.idx_ready[r], (t / IDX_RING) & 1, ctx, abort)) break;
        const int row0 = sm.tile_row0[r];
        if (row0 < 0) break;
        if (!FP8) {
            if (use >= 1 && !warp_wait(b.kv_empty[st], (use - 1) & 1, ctx, abort)) break;
            cp.issue(smem_u32(sm.kv[st]), sm.idx[r], p.kv + (size_t)row0 * HD, g);
            cp_async_arrive(smem_u32(&b.kv_full[st]));
            __syncwarp();
        } else {
            // the codes are loaded before the stage is free (registers only)
            // the codes are loaded before the stage is free (registers only)
            uint4 q[4];
            float sc[4];
            fc.load_codes(sm.idx[r], p.kv_nope + (size_t)row0 * DN, p.kv_scale + row0, g, q, sc);
            if (use >= 1 && !warp_wait(b.kv_empty[st], (use - 1) & 1, ctx, abort)) break;
            fc.issue_rope(smem_u32(sm.kv[st]), sm.idx[r], p.kv_rope + (size_t)row0 * (HD - DN), g);
            cp_async_arrive(smem_u32(&b.kv_full[st]));
            fc.store_codes(smem_u32(sm.kv[st]), g, q, sc);
            fence_proxy_async_smem();  // the stores are read by the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&b.kv_full[st]));
        }
        if (lane == 0) mbar_arrive(smem_u32(&b.idx_empty[r]));
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global to shared memory, completion on `bar` (tx bytes).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ void gather_lead(const SpParams &p, const CUtensorMap *tq, SlotSmem &sm,
                            volatile int *abort, int first, int stride, const DevCtx &ctx) {
    SlotBars &b = sm.b;
    const int lane = threadIdx.x & 31;
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int nitems = p.B * p.M * p.splits;
    int qi = 0, gt = 0;  // items started, tiles issued
    bool ok = true, bad = false;
    // The slot's index lists stream into a ring of NLCH chunks in shared
    // memory, by bulk copies (rows of the list 16-byte aligned: K % 4 == 0 and
    // an aligned base) or else by the warp itself. The issue cursor (item,
    // offset) runs NLCH chunks ahead of compaction.
    const bool bulk = (p.K & 3) == 0 && (reinterpret_cast<uintptr_t>(p.idx) & 15u) == 0;
    int is_item = first, is_off = 0, n_iss = 0, n_con = 0;
    auto issue_chunk = [&]() {
        while (is_item < nitems) {
            const ItemInfo ni = item_info(p, is_item);
            const int e0 = ni.e_begin + is_off;
            if (e0 >= ni.e_end) {  // next item
                is_item += stride;
                is_off = 0;
                continue;
            }
            const int n = min(LCHUNK, ni.e_end - e0);
            const int slot = n_iss % NLCH;
            const int32_t *src = p.idx + (size_t)ni.bm * p.K + e0;
            const uint32_t bar = smem_u32(&b.lst_full[slot]);
            if (bulk) {
                if (lane == 0) {
                    fence_proxy_async_smem();  // earlier reads of the slot come first
                    mbar_arrive_expect_tx(bar, (uint32_t)n * 4u);
                    bulk_load(smem_u32(sm.lst[slot]), src, (uint32_t)n * 4u, bar);
                }
            } else {
                for (int i = lane; i < n; i += 32) sm.lst[slot][i] = __ldg(src + i);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar);
            }
            is_off += LCHUNK;
            ++n_iss;
            return;
        }
    };
    if (lane == 0) prefetch_tmap(tq);
    for (int k = 0; k < NLCH; ++k) issue_chunk();
    // Q rows of a query (32 heads x 256 B, two 64-column boxes) go to the
    // slot's Q buffer once the previous item's last S was issued. The lead
    // polls for that between tiles and blocks only when it is a whole item
    // ahead (or at the end).
    int q_pend = -1;  // query row (b, m) whose Q copy is still to be issued
    auto issue_q = [&](bool block) -> bool {
        if (q_pend < 0) return true;
        if (qi >= 1) {
            if (block) {
                if (!warp_wait(b.q_empty, (qi - 1) & 1, ctx, abort)) return false;
            } else {
                int r = lane == 0 ? (mbar_try_wait(smem_u32(&b.q_empty), (qi - 1) & 1) ? 1 : 0) : 0;
                if (!__shfl_sync(0xffffffffu, r, 0)) return true;  // not yet
            }
        }
        if (lane == 0) {
            const uint32_t bar = smem_u32(&b.q_full);
            mbar_arrive_expect_tx(bar, 2 * QP_HALF);
            tma_load_2d(smem_u32(sm.q), tq, bar, 0, q_pend * NH);
            tma_load_2d(smem_u32(sm.q) + QP_HALF, tq, bar, 64, q_pend * NH);
        }
        ++qi;
        q_pend = -1;
        return true;
    };
    for (int item = first; ok && item < nitems; item += stride) {
        const ItemInfo it = item_info(p, item);
        const int row0 = it.b * p.N;  // first cache row of this request
        if (!issue_q(true)) {  // the previous item's Q first
            ok = false;
            break;
        }
        q_pend = it.bm;
        issue_q(false);  // at once when the buffer is free (always for the first item)
        int ring = gt % IDX_RING;  // ring entry of the tile being compacted
        // Publish and issue the compacted tile gt holding `pos` rows.
        auto close_tile = [&](int pos, bool last) -> bool {
            int *ids = sm.idx[ring];
            for (int r = pos + lane; r < R; r += 32) ids[r] = -1;
            if (lane == 0) {
                sm.tile_cnt[ring] = pos;
                sm.tile_last[ring] = last ? 1 : 0;
                sm.tile_row0[ring] = row0;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&b.idx_ready[ring]));
            issue_q(false);
            ++gt;
            ring = gt % IDX_RING;
            // the next entry is written once its previous tile's readers let
            // go. Before blocking on that, the pending Q is issued: S of the
            // entry's previous tile may need it (the Q wait itself only needs
            // the previous item's tiles, all published).
            if (gt < IDX_RING) return true;
            const int par = ((gt / IDX_RING) - 1) & 1;
            int r = lane == 0 ? (mbar_try_wait(smem_u32(&b.idx_empty[ring]), par) ? 1 : 0) : 0;
            if (__shfl_sync(0xffffffffu, r, 0)) return true;
            return issue_q(true) && warp_wait(b.idx_empty[ring], par, ctx, abort);
        };
        int pos = 0;
        for (int c0 = it.e_begin; ok && c0 < it.e_end; c0 += LCHUNK) {
            const int slot = n_con % NLCH;
            if (!warp_wait(b.lst_full[slot], (n_con / NLCH) & 1, ctx, abort)) {
                ok = false;
                break;
            }
            const int *lst = sm.lst[slot];
            const int n = min(LCHUNK, it.e_end - c0);
            // groups of 128 entries (four consecutive ones per lane): ballot-
            // compact the valid ones into the open tile
            for (int g0 = 0; ok && g0 < n; g0 += R) {
                int v[4];
                const int i0 = g0 + 4 * lane;
                if (i0 + 4 <= n) {
                    const int4 q4 = *reinterpret_cast<const int4 *>(lst + i0);
                    v[0] = q4.x;
                    v[1] = q4.y;
                    v[2] = q4.z;
                    v[3] = q4.w;
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) v[c] = i0 + c < n ? lst[i0 + c] : -1;
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    int x = v[c];
                    if (x < -1 || x >= p.N) {
                        bad = true;
                        x = -1;
                    }
                    const bool valid = x >= 0;
                    const uint32_t bal = __ballot_sync(0xffffffffu, valid);
                    const int cnt = __popc(bal);
                    if (cnt == 0) continue;
                    if (pos + cnt > R) {  // does not fit: issue this tile, open the next
                        __syncwarp();
                        if (!close_tile(pos, false)) {
                            ok = false;
                            break;
                        }
                        pos = 0;
                    }
                    if (valid) sm.idx[ring][pos + __popc(bal & lt_mask)] = x;
                    pos += cnt;
                }
            }
            __syncwarp();  // the chunk's reads are done: refill its slot
            ++n_con;
            if (ok) {
                issue_chunk();
                issue_q(false);
            }
        }
        if (!ok) break;
        __syncwarp();
        // an item without valid entries still gets one (empty) tile
        if (!close_tile(pos, true)) { ok = false; break; }
    }
    if (ok && !issue_q(true)) ok = false;  // the last item's Q
    if (ok) {  // no more tiles (the next ring entry was opened by the last close_tile)
        const int ring = gt % IDX_RING;
        if (lane == 0) {
            sm.tile_row0[ring] = -1;
            mbar_arrive(smem_u32(&b.idx_ready[ring]));
        }
    }
    if (bad) record_error(ctx, DEVERR_INDEX);
    // the last Q load lands before the CTA may exit (on the normal path it was
    // consumed already; this matters after an abort)
    if (lane == 0) {
        int zero = 0;
        if (qi >= 1) mbar_wait(smem_u32(&b.q_full), (qi - 1) & 1, ctx, &zero);
        for (int k = n_con; k < n_iss; ++k)  // list copies still in flight
            mbar_wait(smem_u32(&b.lst_full[k % NLCH]), (k / NLCH) & 1, ctx, &zero);
    }
    __syncwarp();
}

// ------------------------------------------------------------------ MMA thread

// The MMA thread issues in readiness order: S^T of the next tile as soon as
// its rows have landed (and its S buffer and Q are free), O^T += KV^T P^T of
// the oldest pending tile as soon as its P is written. Issuing S before P V in
// program order instead would hold P V of tile t behind the gather of tile
// t+1, which itself waits for P V of tile t-1 to free its stage.
// S(t) needs kv_full(t), hence P V of tile t-2 complete: the S cursor runs at
// most two tiles ahead of the P V cursor.
__device__ void mma_role(const SpParams &p, SlotSmem &sm, volatile int *abort, uint32_t tmem,
                         int first, int stride, const DevCtx &ctx) {
    SlotBars &b = sm.b;
    const int nitems = p.B * p.M * p.splits;
    const int my_items = first < nitems ? (nitems - first + stride - 1) / stride : 0;
    const uint32_t t_o = tmem + O_COL;
    const uint64_t dq = desc_sw128(smem_u32(sm.q), 16u);
    // per stage (selected, not indexed, so that they stay in registers)
    const uint64_t dkv0 = desc_sw128(smem_u32(sm.kv[0]), 16u);
    const uint64_t dkv1 = desc_sw128(smem_u32(sm.kv[1]), 16u);
    const uint64_t dmn0 = desc_sw128(smem_u32(sm.kv[0]), KV_HALF);
    const uint64_t dmn1 = desc_sw128(smem_u32(sm.kv[1]), KV_HALF);
    const uint64_t dp0 = desc_sw128(smem_u32(sm.p[0]), 16u);
    const uint64_t dp1 = desc_sw128(smem_u32(sm.p[1]), 16u);
    int s_t = 0, s_item = 0;     // next tile / item for S
    int pv_t = 0, pv_item = 0;   // next tile / item for P V
    bool s_first = true, pv_first = true;  // the next tile opens its item
    uint32_t lastmask = 0;       // bit t & 3: tile t closes its item (known once S(t) issued)
    uint64_t stall_t0 = 0;
    uint32_t spins = 0;
    if (ctx.stall) mbar_wait(smem_u32(&b.drain), 0, ctx, abort);  // test hook: runs out
    while (pv_item < my_items) {
        bool progress = false;
        if (s_item < my_items) {
            const int st = s_t & 1, use = s_t >> 1;
            if ((!s_first || mbar_try_wait(smem_u32(&b.q_full), s_item & 1)) &&
                (use == 0 || mbar_try_wait(smem_u32(&b.s_empty[st]), (use - 1) & 1)) &&
                mbar_try_wait(smem_u32(&b.kv_full[st]), use & 1) &&
                mbar_try_wait(smem_u32(&b.idx_ready[s_t % IDX_RING]), (s_t / IDX_RING) & 1)) {
                tc_fence_after();
                const bool last = sm.tile_last[s_t % IDX_RING] != 0;
                mbar_arrive(smem_u32(&b.idx_empty[s_t % IDX_RING]));
                const uint64_t a = st ? dkv1 : dkv0;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    tc_mma_f16(tmem + S_COL + 32u * st, a + koff(kk, KV_HALF),
                               dq + koff(kk, QP_HALF), IDESC_S, kk > 0 ? 1u : 0u);
                tc_commit(smem_u32(&b.s_full[st]));
                if (last) {
                    tc_commit(smem_u32(&b.q_empty));
                    lastmask |= 1u << (s_t & 3);
                    ++s_item;
                } else {
                    lastmask &= ~(1u << (s_t & 3));
                }
                s_first = last;
                ++s_t;
                progress = true;
            }
        }
        if (pv_t < s_t) {
            const int st = pv_t & 1;
            if (mbar_try_wait(smem_u32(&b.p_full[st]), (pv_t >> 1) & 1) &&
                (!pv_first || pv_item == 0 ||
                 mbar_try_wait(smem_u32(&b.o_empty), (pv_item - 1) & 1))) {
                tc_fence_after();
                const uint64_t a = st ? dmn1 : dmn0, bp = st ? dp1 : dp0;
                const uint32_t acc0 = pv_first ? 0u : 1u;
#pragma unroll
                for (int kk = 0; kk < R / 16; ++kk)
                    tc_mma_f16(t_o, a + mnoff(kk), bp + koff(kk, QP_HALF), IDESC_O,
                               kk > 0 ? 1u : acc0);
                tc_commit(smem_u32(&b.kv_empty[st]));
                tc_commit(smem_u32(&b.p_empty[st]));
                tc_commit(smem_u32(&b.pv_done));
                const bool last = (lastmask >> (pv_t & 3)) & 1u;
                if (last) {
                    tc_commit(smem_u32(&b.o_full));
                    ++pv_item;
                }
                pv_first = last;
                ++pv_t;
                progress = true;
            }
        }
        if (progress) {
            spins = 0;
        } else if ((++spins & 63u) == 0) {  // bounded: give up after the wait limit
            if (*abort) break;
            const uint64_t now = global_timer_ns();
            if (spins == 64) stall_t0 = now;
            else if (now - stall_t0 > ctx.wait_ns) {
                *abort = 1;
                record_error(ctx, DEVERR_TIMEOUT);
                break;
            }
        }
    }
    // every MMA issued so far completes before TMEM is released
    tc_commit(smem_u32(&b.drain));
    int zero = 0;
    mbar_wait(smem_u32(&b.drain), 0, ctx, &zero);
}

// ------------------------------------------------------------------ softmax warps

// Softmax of one slot: warp w reads S^T rows (keys) 32w .. 32w+31 from TMEM and
// transposes its own 32 x 32 block through shared memory, so that lane l owns
// head l over those 32 keys. All warps share one running max per head, which
// moves only when some warp's tile max exceeds it by more than TAU (log2
// units): the common case needs a single barrier per tile (an OR over that
// condition); the max exchange, the O^T rescale and their barriers run only
// when it is true. Each warp keeps its own partial denominator per head; the
// four are added in the epilogue.
__device__ void softmax_role(const SpParams &p, SlotSmem &sm, volatile int *abort, int slot,
                             uint32_t tmem, int first, int stride, const DevCtx &ctx) {
    SlotBars &b = sm.b;
    // a warp may only access TMEM lanes 32 * (warp id mod 4) .. +31: this
    // warp's S^T rows (keys) and O^T rows (head-dim indices) are 32 * quarter + lane
    const int lane = threadIdx.x & 31, quarter = (threadIdx.x >> 5) & 3;
    const int h = lane;  // head owned after the transpose
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_o = tmem + O_COL + lane_off;
    const bool key0 = p.sink_mode == 1;
    const float sink_h = p.sinks ? __ldg(p.sinks + h) * LOG2E : 0.0f;
    const float bias_raw = key0 ? sink_h / p.scale_l2 : 0.0f;
    const uint64_t scale2 = f2_pack(p.scale_l2, p.scale_l2);
    const bool null_sink = p.sink_mode == 2 && p.splits == 1;
    const int nitems = p.B * p.M * p.splits;
    float *tb = sm.tbuf[quarter];
    int qi = 0, gt = 0;
    // A failed wait is carried to the next barrier, whose OR makes the exit
    // uniform over the four warps (no thread is left behind at a barrier).
    bool failed = false;
    for (int item = first; item < nitems; item += stride) {
        const ItemInfo it = item_info(p, item);
        float m_run = null_sink ? sink_h : -INFINITY;
        // the null logit's exp(sink - m) = 1 is counted once, in warp 0's partial
        float l_run = (null_sink && quarter == 0) ? 1.0f : 0.0f;
        const int gt0 = gt;
        int j = 0;
        for (bool last = false; !last; ++j) {
            const int t = gt0 + j, st = t & 1, use = t >> 1, ring = t % IDX_RING;
            // the tile's ring entry, S^T of the tile; P buffer st was last read
            // by P V of tile t-2
            if (!failed) {
                failed = !mbar_wait(smem_u32(&b.idx_ready[ring]), (t / IDX_RING) & 1, ctx, abort) ||
                         !mbar_wait(smem_u32(&b.s_full[st]), use & 1, ctx, abort) ||
                         (use >= 1 &&
                          !mbar_wait(smem_u32(&b.p_empty[st]), (use - 1) & 1, ctx, abort));
            }
            failed = __any_sync(0xffffffffu, failed);  // tcgen05.ld is warp-collective
            float x[32];
            float mt = -INFINITY;
            if (!failed) {
                tc_fence_after();
                uint32_t sv[32];
                tmem_ld32(tmem + S_COL + 32u * st + lane_off, sv);
                tc_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&b.s_empty[st]));
                // row (key 32 quarter + lane) -> column lane of the warp's block
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) tb[hh * TB_STRIDE + lane] = __uint_as_float(sv[hh]);
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float4 f = *reinterpret_cast<const float4 *>(tb + h * TB_STRIDE + 4 * k);
                    x[4 * k] = f.x;
                    x[4 * k + 1] = f.y;
                    x[4 * k + 2] = f.z;
                    x[4 * k + 3] = f.w;
                }
                // the ring entry is read here, then released to the lead warp
                last = sm.tile_last[ring] != 0;
                if (key0) {  // the sink bias on the logit of key 0, in raw-score units
                    const int *ids = &sm.idx[ring][quarter * 32];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int4 e = *reinterpret_cast<const int4 *>(ids + 4 * k);
                        x[4 * k] += e.x == 0 ? bias_raw : 0.f;
                        x[4 * k + 1] += e.y == 0 ? bias_raw : 0.f;
                        x[4 * k + 2] += e.z == 0 ? bias_raw : 0.f;
                        x[4 * k + 3] += e.w == 0 ? bias_raw : 0.f;
                    }
                }
                const int nvalid = sm.tile_cnt[ring] - quarter * 32;  // keys of this warp holding entries
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&b.idx_empty[ring]));
                if (nvalid < 32) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i >= nvalid) x[i] = -INFINITY;
                }
                // raw scores: scale > 0, so the max is taken before scaling
                float mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < 32; i += 2)
                    mr[(i >> 1) & 3] = max3(mr[(i >> 1) & 3], x[i], x[i + 1]);
                mt = fmaxf(max3(mr[0], mr[1], mr[2]), mr[3]) * p.scale_l2;
            }
            // one barrier per tile: does any head of any warp need a new max?
            // (also orders this tile's transpose reads before the next writes)
            if (softmax_sync_or(slot, failed || mt > m_run + TAU)) {
                if (softmax_sync_or(slot, failed)) { failed = true; break; }
                sm.xmax[quarter][h] = mt;
                softmax_sync_or(slot, 0);
                const float mall = fmaxf(fmaxf(sm.xmax[0][h], sm.xmax[1][h]),
                                         fmaxf(sm.xmax[2][h], sm.xmax[3][h]));
                const bool upd = mall > m_run + TAU;  // the same in every warp
                float alpha = 1.0f;
                if (upd) {
                    alpha = (m_run == -INFINITY) ? 0.0f : ex2(m_run - mall);
                    l_run *= alpha;
                    m_run = mall;
                }
                if (quarter == 0) sm.alpha[h] = alpha;
                if (softmax_sync_or(slot, upd && j >= 1)) {
                    // rescale the O^T columns (heads) whose max moved, once P V of
                    // the previous tile is complete (the one before it is: P
                    // buffer st was free)
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
            }
            const float mu = m_run == -INFINITY ? 0.0f : m_run;
            const uint64_t negm2 = f2_pack(-mu, -mu);
            uint64_t ls2a = f2_pack(0.f, 0.f), ls2b = ls2a;
            // P^T: head h, keys 32 quarter .. +31 = 64 bytes of one K-major row
            const uint32_t pbase = smem_u32(sm.p[st]) + (uint32_t)(quarter >> 1) * QP_HALF;
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
                const uint32_t addr = pbase + sw128_offset(h, (quarter & 1) * 4 + u);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]),
                             "r"(w[1]), "r"(w[2]), "r"(w[3])
                             : "memory");
            }
            {
                float a0, a1;
                f2_unpack(f2_add(ls2a, ls2b), a0, a1);
                l_run += a0 + a1;
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
        sm.lpart[quarter][h] = l_run;
        if (softmax_sync_or(slot, failed)) break;
        ++qi;
        const size_t rows = (size_t)p.B * p.M * NH;
        if (quarter == 0) {  // head h: total denominator, its inverse and the lse
            const float l = (sm.lpart[0][h] + sm.lpart[1][h]) + (sm.lpart[2][h] + sm.lpart[3][h]);
            sm.inv_l[h] = l > 0.f ? 1.0f / l : 0.f;
            const float lse = l > 0.f ? (m_run + log2f(l)) * LN2 : -INFINITY;
            if (p.splits == 1) {
                if (p.lse) p.lse[(size_t)it.bm * NH + h] = lse;
            } else {
                p.lse_part[(size_t)it.split * rows + (size_t)it.bm * NH + h] = lse;
            }
        }
        tc_fence_after();
        uint32_t ov[32];
        tmem_ld32(t_o, ov);
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&b.o_empty));
        softmax_sync_or(slot, 0);  // inv_l complete
        // O / l straight from registers: for each head the 128 threads of the
        // group write 128 consecutive values of d (coalesced)
        const int d = quarter * 32 + lane;
        if (p.splits == 1) {
            __nv_bfloat16 *ob = p.o + (size_t)it.bm * NH * HD + d;
#pragma unroll
            for (int hh = 0; hh < NH; ++hh)
                ob[hh * HD] = __float2bfloat16_rn(__uint_as_float(ov[hh]) * sm.inv_l[hh]);
        } else {
            float *op = p.o_part + ((size_t)it.split * rows + (size_t)it.bm * NH) * HD + d;
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) op[hh * HD] = __uint_as_float(ov[hh]) * sm.inv_l[hh];
        }
        // lpart / inv_l are rewritten only after the next item's barriers
    }
}

// FP8: the cache holds e4m3 codes + scales + bf16 RoPE columns instead of bf16
// rows (only the copy warps differ; they also arrive once per warp on kv_full
// after their shared-memory stores)
template <bool FP8>
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
                mbar_init(smem_u32(&b.kv_full[i]), 32 * GATHER_WARPS + (FP8 ? GATHER_WARPS : 0));
                mbar_init(smem_u32(&b.kv_empty[i]), 1);
                mbar_init(smem_u32(&b.s_full[i]), 1);
                mbar_init(smem_u32(&b.s_empty[i]), 4);
                mbar_init(smem_u32(&b.p_full[i]), 4);
                mbar_init(smem_u32(&b.p_empty[i]), 1);
            }
            for (int i = 0; i < IDX_RING; ++i) {
                mbar_init(smem_u32(&b.idx_ready[i]), 1);
                mbar_init(smem_u32(&b.idx_empty[i]), GATHER_WARPS + 1 + 4);  // copy, MMA, softmax
            }
            for (int i = 0; i < NLCH; ++i) mbar_init(smem_u32(&b.lst_full[i]), 1);
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
    // slot s: warps SLOT_CTRL * s + role (lead, copy warps, MMA), then
    // NSLOT * SLOT_CTRL + 4s .. +3 (softmax: four consecutive warps cover the
    // four TMEM lane quarters)
    const int ctrl = NSLOT * SLOT_CTRL;
    const int slot = warp < ctrl ? warp / SLOT_CTRL : (warp - ctrl) >> 2;
    const uint32_t tmem = all.tmem_base + (uint32_t)slot * SLOT_COLS;
    const int first = blockIdx.x * NSLOT + slot, stride = gridDim.x * NSLOT;
    SlotSmem &sm = all.slot[slot];
    if (warp < ctrl) {
        const int role = warp % SLOT_CTRL;  // 0 lead, 1 .. GATHER_WARPS copy, then MMA
        if (role <= GATHER_WARPS) {
            if (role == 0) gather_lead(p, &tq, sm, &all.abort, first, stride, ctx);
            else gather_helper<FP8>(p, sm, &all.abort, role - 1, ctx);
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
    const long long items = (long long)B * M;
    const int max_split = (K + R - 1) / R;
    // two items run per SM; aim for one round of items
    if (max_split <= 1 || items <= 0 || items >= (long long)NSLOT * sm_count) return 1;
    int s = (int)((NSLOT * sm_count) / items);
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
    const bool fp8 = a.kv == nullptr;
    if (a.H != NH || a.d != HD) return fp8 ? cudaErrorInvalidValue : launch_sparse_simt(a, dev, s);
    {  // few queries: one launch, splits merged inside clusters
        const int C = sparse_decode_cluster(a.B, a.M, a.K, dev.sm_count);
        if (C > 0) {
            const cudaError_t e = launch_sparse_decode(a, C, dev, s);
            if (e != cudaErrorInvalidClusterSize) return e;
            (void)cudaGetLastError();  // nothing was launched: take the split path
        }
    }
    SpParams p{};
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
    auto kernel = fp8 ? sparse_tc_kernel<true> : sparse_tc_kernel<false>;
    {
        cudaError_t e = ensure_smem_attr((const void *)kernel, smem, dev);
        if (e != cudaSuccess) return e;
    }
    const DevCtx ctx = make_ctx(dev);
    if (verbose())
        fprintf(stderr, "sattn: sparse_tc_kernel<%s> grid=%d block=%d smem=%zu items=%lld splits=%d\n",
                fp8 ? "fp8" : "bf16", grid, NTHREADS, smem, nitems, splits);
    kernel<<<grid, NTHREADS, smem, s>>>(tq, p, ctx);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || splits == 1) return e;
    MergeArgs m{p.o_part, p.lse_part, splits, (int64_t)rows, a.d, a.H,
                a.sink_mode == 2 ? a.sinks : nullptr, a.o, a.lse, a.dtype};
    return launch_merge(m, dev, s, true);
}

}  // namespace sattn
