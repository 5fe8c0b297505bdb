// Tensor-core attention over contiguous key tiles (tcgen05 + TMEM + TMA).
//
// Two uses share this engine:
//  * sliding-window varlen attention with sinks ("PR #49815 report": window
//    |i-j| <= w inside each sequence, key-0 bias or null-logit sink). Only
//    the key tiles that intersect a query tile's band are visited (the report
//    notes that visiting every block and masking costs O(seq_len^2));
//  * one KV chunk of block-sparse causal attention ("XAttention Offload
//    Stream Synchronization Fix": per-chunk partial stats, merged later);
//    the key tiles are the two 64-key halves of each selected 128-key block.
//
// A work item is a tile of 128 query rows: in window mode BM / G tokens x G
// query heads of one KV group (G, the largest power of two dividing H / Hkv
// up to 8, shrinks the tile's key band and lets one K/V tile serve G heads),
// in block mode 128 tokens of one head. A persistent grid of one CTA
// per SM (kernels that allocate tensor memory run one CTA per SM) walks the
// items with two independent pipeline slots, each with its own shared
// memory, barriers, 256 TMEM columns and item stream. Per slot:
//   warp 2s       TMA producer: the Q tile, then K and V tiles of 64 keys
//                 (two stages each), 128B-swizzled, rows of 256 B.
//   warp 2s+1     MMA issuer (one thread): S = Q K^T into TMEM (64
//                 columns), then O += P V into TMEM with P read from TMEM
//                 (A operand in tensor memory, two P buffers of 32 columns).
//   warps 4+4s..  softmax + epilogue (four warps): thread = query row = TMEM lane. Each
//                 row keeps its running max m and sum l in the log2 domain. An item's
//                 epilogue runs once its last P V has completed, while the MMA
//                 computes the next item's first scores.
// S of tile j+1 is computed as soon as the softmax has loaded S of tile j.
// No tensor-memory column is read by one MMA and written by a later one, so
// ordering rests only on commits and barriers; since S of tile j is issued
// after P V of tile j-2, seeing S(j) complete also frees P buffer j % 2.
// The two slots give every SM sub-partition two softmax warps and let one
// slot's MMAs overlap the other's softmax.
//
// Softmax per tile: the maximum is taken over the raw scores (the scale is
// positive), and each probability is ex2(s * scale*log2(e) - m) with the
// multiply-add done two lanes at a time (f32x2). Chunks of 32 keys that no
// row of a warp can see are skipped; chunks every row sees are not masked.
// The running max is only moved when a tile raises it by more than 2^8, so
// the accumulator in TMEM is rarely rescaled (P <= 256 otherwise).
// Null-logit sinks start from m = sink, l = 1; key-0 sinks add the sink to
// key 0's logit where it is visible.
#include <limits.h>
#include <math.h>
#include <stddef.h>
#include <stdio.h>

#include "common.cuh"
#include "internal.h"

namespace sattn {
namespace {

constexpr int BM = 128;                   // queries per tile (TMEM lanes)
constexpr int BN = 64;                    // keys per tile
constexpr int HD = 128;                   // head dim
constexpr uint32_t Q_TILE = BM * HD * 2;  // 32 KB
constexpr uint32_t Q_HALF = Q_TILE / 2;   // 64 columns of d (128-byte rows)
constexpr uint32_t KV_TILE = BN * HD * 2; // 16 KB
constexpr uint32_t KV_HALF = KV_TILE / 2;
constexpr int NSLOTS = 2;
constexpr int KSTAGES = 2;                // K tiles in flight per slot
constexpr int VSTAGES = 2;                // V tiles in flight per slot
constexpr int NTHREADS = 128 * (NSLOTS + 1);  // 2 role warps + 4 softmax warps per slot
constexpr uint32_t SLOT_COLS = 256;       // per slot: S (64) + P[2] (32 each) + O (128)
constexpr uint32_t S_COL = 0, P_COL = 64;
constexpr uint32_t TMEM_COLS = SLOT_COLS * NSLOTS;
constexpr uint32_t O_COL = 128;
constexpr float TAU = 8.0f;               // rescale threshold (log2 units)
constexpr int ITEM_RING = 4;              // items the producer may hand on ahead
constexpr unsigned FULL = 0xffffffffu;

enum : int { MODE_WINDOW = 0, MODE_BLOCK = 1 };

struct TcParams {
    int H, Hkv, groups, num_items;
    float scale_l2;  // scale * log2(e) (> 0)
    float inv_scale; // 1 / scale
    // window
    const int32_t *cu_seqlens;
    int num_seqs, T, tiles_per_seq, wl, wr, causal;
    // query heads per item: 1 << gshift heads that share a KV head fill the
    // 128 tile rows together (row r = token r >> gshift, head r & (G - 1));
    // hslots = H >> gshift items per token tile. Block mode: gshift = 0.
    int gshift, hslots;
    const float *sinks;
    int sink_mode;
    __nv_bfloat16 *o;
    float *lse;
    // block
    const uint8_t *mask;
    int M, Nctx, q_pos0, kv_begin, kv_end, QB, KB;
    int chunk_keys;        // [kv_begin, kv_end) in chunks of this many keys, one output each
    float *o_part, *lse_part;  // [chunk, M, H, d] and [chunk, M, H]
    unsigned *work;  // the launch's claim counter, zeroed on its stream: items claimed
};

struct Item {
    bool valid;
    bool seq_err;
    int h, g, nq, ntiles;
    int q_row0;    // first row of the tile in q / o (token index)
    int key_row0;  // global K/V row of key coordinate 0
    int qpos0;     // window: local index of query row 0; block: absolute position
    int lo, hi, L; // window: key band of the tile (local), sequence length;
                   // block: the chunk's keys [lo, hi) and the chunk's index
    const uint8_t *mrow;
    int kb_lo, kb_hi, kend;  // block: 128-key block range, key limit
    float sink[8];           // window: the sinks of heads h .. h + G - 1 (0 without sinks)
};

struct Bars {
    uint64_t q_full, q_empty, k_full[KSTAGES], k_empty[KSTAGES], v_full[VSTAGES], v_empty[VSTAGES];
    // p_full is per P buffer: a softmax warp may run one tile ahead of the
    // others, so arrivals for consecutive tiles must not share a barrier.
    uint64_t s_full, s_empty, p_full[2], pv_done, o_full, o_empty, drain;
    // items claimed by the producer, handed to the MMA issuer and softmax warps
    // already decoded (valid = false: no more items)
    uint64_t item_full[ITEM_RING], item_empty[ITEM_RING];
    Item item[ITEM_RING];
};

// Operand tiles and epilogue staging of one pipeline slot (112 KB).
struct Slot {
    uint8_t q[Q_TILE];
    uint8_t k[KSTAGES][KV_TILE];
    uint8_t v[VSTAGES][KV_TILE];
    // epilogue staging: each softmax warp turns its 32 output rows into
    // whole 128-byte line writes, 128 bytes of every row per pass
    uint8_t stage[4][32 * 128];
};
static_assert(offsetof(Slot, k) % 1024 == 0 && offsetof(Slot, v) % 1024 == 0 &&
                  sizeof(Slot) % 1024 == 0,
              "operand tiles must sit on 1024-byte boundaries");

// The whole shared-memory footprint (dynamic only; the base of the CTA's
// shared window is 1024-byte aligned, as the 128B swizzle needs).
struct Smem {
    Slot slot[NSLOTS];
    Bars bars[NSLOTS];
    uint32_t tmem_base;
    int abort;  // any role that gives up stops every role of the CTA
};
static_assert(sizeof(Smem) <= 227 * 1024, "shared memory of one CTA");


template <int MODE> __device__ __forceinline__ Item decode_item(const TcParams &p, int v) {
    Item it;
    it.valid = false;
    it.seq_err = false;
    it.ntiles = 0;
    const int hslots = MODE == MODE_WINDOW ? p.hslots : p.H;
    it.h = (v % hslots) << (MODE == MODE_WINDOW ? p.gshift : 0);  // first head of the item
    it.g = it.h / p.groups;
    const int rest = v / hslots;
    if (MODE == MODE_WINDOW) {
        const int TT = BM >> p.gshift;  // tokens per tile
        const int t = rest % p.tiles_per_seq, s = rest / p.tiles_per_seq;
        const int s0 = __ldg(p.cu_seqlens + s), s1 = __ldg(p.cu_seqlens + s + 1);
        if (s0 < 0 || s1 < s0 || s1 > p.T || __ldg(p.cu_seqlens) != 0 ||
            s1 - s0 > p.tiles_per_seq * TT) {
            it.seq_err = true;
            return it;
        }
        it.L = s1 - s0;
        const int qs = t * TT;
        if (qs >= it.L) return it;
        const int ntok = min(TT, it.L - qs);
        it.nq = ntok << p.gshift;  // valid rows (token-major, so a prefix)
        it.q_row0 = s0 + qs;
        it.key_row0 = s0;
        it.qpos0 = qs;
        const int last = qs + ntok - 1;
        it.lo = p.wl < 0 ? 0 : max(0, qs - p.wl);
        it.hi = p.wr < 0 ? it.L - 1 : min(it.L - 1, last + p.wr);
        if (p.causal) it.hi = min(it.hi, last);
        it.ntiles = (it.hi - it.lo + BN) / BN;
#pragma unroll
        for (int i = 0; i < 8; ++i)  // constant indices keep the item in registers
            it.sink[i] = p.sinks && i < (1 << p.gshift) ? __ldg(p.sinks + it.h + i) : 0.f;
        it.valid = true;
    } else {
        const int qb = rest % p.QB;
        it.L = rest / p.QB;  // chunk
        it.lo = p.kv_begin + it.L * p.chunk_keys;
        it.hi = (int)min((long long)p.kv_end, (long long)it.lo + p.chunk_keys);
        const int qs = qb * BM;
        it.nq = min(BM, p.M - qs);
        it.q_row0 = qs;
        it.key_row0 = 0;
        it.qpos0 = p.q_pos0 + qs;
        int end = it.hi;
        if (p.causal) end = min(end, it.qpos0 + it.nq);
        it.kend = end;
        it.kb_lo = it.lo / 128;
        it.kb_hi = end > it.lo ? (end - 1) / 128 : it.kb_lo - 1;
        it.mrow = p.mask + ((size_t)it.h * p.QB + qb) * p.KB;
        int n = 0;
        for (int kb = it.kb_lo; kb <= it.kb_hi; ++kb) {
            if (!__ldg(it.mrow + kb)) continue;
            // 64-key halves that overlap [kv_begin, end)
            for (int hh = 0; hh < 2; ++hh) {
                const int base = kb * 128 + hh * BN;
                n += (base < end && base + BN > it.lo) ? 1 : 0;
            }
        }
        it.ntiles = n;
        it.valid = true;
    }
    return it;
}

// Key coordinate of the first key of each successive tile of an item.
template <int MODE> struct TileIter {
    int j, kb, hh;
    __device__ explicit TileIter(const Item &it) : j(0), kb(it.kb_lo - 1), hh(1) {}
    __device__ int next(const TcParams &p, const Item &it) {
        if (MODE == MODE_WINDOW) return it.lo + BN * (j++);
        for (;;) {
            if (kb > it.kb_hi) return it.kb_hi * 128;  // unreachable for a fixed mask
            if (hh == 1) {
                do { ++kb; } while (kb <= it.kb_hi && __ldg(it.mrow + kb) == 0);
                hh = 0;
            } else {
                hh = 1;
            }
            const int base = kb * 128 + hh * BN;
            if (base < it.kend && base + BN > it.lo) {
                ++j;
                return base;
            }
        }
    }
};

// Shared-memory descriptors are built once per buffer; the K step kk (16
// elements) only moves the start address, whose field holds address >> 4 in
// the low bits (no carry: shared addresses stay below 256 KB).
// K-major operand with 128-byte rows split in 64-column halves `half` bytes apart
__host__ __device__ constexpr uint32_t koff(int kk, uint32_t half) {
    return ((uint32_t)(kk >> 2) * half + (uint32_t)(kk & 3) * 32u) >> 4;
}
// MN-major operand (V: rows = keys, 64-column halves of d KV_HALF bytes apart)
__host__ __device__ constexpr uint32_t mnoff(int kk) { return (uint32_t)kk * 2048u >> 4; }

// 3-D tiled TMA store from shared memory (bulk group), its commit and waits.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *m, uint32_t src, int x, int y,
                                             int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(m)),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the shared-memory sources of this thread's bulk stores have been read
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// this thread's bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BN, 0, 0);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, HD, 0, 1);

// ------------------------------------------------------------------ producer

template <int MODE>
__device__ void producer(const TcParams &p, const CUtensorMap *tq, const CUtensorMap *tk,
                         const CUtensorMap *tv, Slot &sm, Bars &b, volatile int *abort,
                         int first, int stride, const DevCtx &ctx) {
    prefetch_tmap(tq);
    prefetch_tmap(tk);
    prefetch_tmap(tv);
    // Loads are issued in the order their stages free up: S of tile t frees
    // K stage t, P V of tile t frees V stage t, and the MMA issues S(t+1)
    // before P V(t), so V runs one tile behind K.
    int qi = 0, kt = 0, vt = 0;
    auto load_k = [&](const Item &it, int row) -> bool {
        const int st = kt % KSTAGES, use = kt / KSTAGES;
        if (use >= 1 && !mbar_wait(smem_u32(&b.k_empty[st]), (use - 1) & 1, ctx, abort))
            return false;
        const uint32_t bar = smem_u32(&b.k_full[st]);
        mbar_arrive_expect_tx(bar, KV_TILE);
        tma_load_3d(smem_u32(sm.k[st]), tk, bar, 0, it.g, row);
        tma_load_3d(smem_u32(sm.k[st]) + KV_HALF, tk, bar, 64, it.g, row);
        ++kt;
        return true;
    };
    auto load_v = [&](int g, int row) -> bool {
        const int st = vt % VSTAGES, use = vt / VSTAGES;
        if (use >= 1 && !mbar_wait(smem_u32(&b.v_empty[st]), (use - 1) & 1, ctx, abort))
            return false;
        const uint32_t bar = smem_u32(&b.v_full[st]);
        mbar_arrive_expect_tx(bar, KV_TILE);
        tma_load_3d(smem_u32(sm.v[st]), tv, bar, 0, g, row);
        tma_load_3d(smem_u32(sm.v[st]) + KV_HALF, tv, bar, 64, g, row);
        ++vt;
        return true;
    };
    bool ok = true;
    // Items are claimed from the launch's counter (the slot that frees up first
    // takes the next one) and handed on through the item ring; items past the
    // end of a short sequence are skipped here and never reach the others.
    int ip = 0;  // items published
    auto publish = [&](const Item &it) -> bool {
        const int k = ip % ITEM_RING, use = ip / ITEM_RING;
        if (use >= 1 && !mbar_wait(smem_u32(&b.item_empty[k]), (use - 1) & 1, ctx, abort))
            return false;
        b.item[k] = it;
        mbar_arrive(smem_u32(&b.item_full[k]));
        ++ip;
        return true;
    };
    // Item order. Window mode: the first 7/8 of the item range is dealt out
    // round-robin (item first + k * stride): the slots of the grid then work on
    // neighbouring query tiles and adjacent heads at the same time, which share
    // K/V bands in L2 and token rows in HBM. The rest is claimed one item at a
    // time from the launch's counter, so that slots that finish early take the
    // remaining work. Block mode (few items per slot) claims every item.
    const int v_static =
        MODE == MODE_WINDOW ? (p.num_items / 8 * 7 / stride) * stride : 0;
    int v_next = first;  // next round-robin item
    for (;;) {
        int v;
        if (v_next < v_static) {
            v = v_next;
            v_next += stride;
        } else {
            v = v_static + (int)atomicAdd(p.work, 1u);
            if (v >= p.num_items) break;
        }
        const Item it = decode_item<MODE>(p, v);
        if (!it.valid) {
            if (it.seq_err) {
                record_error(ctx, DEVERR_SEQLENS);
            } else if (MODE == MODE_WINDOW && v >= v_static) {
                // every later item of this sequence lies past its end as well:
                // move the counter to the next sequence's first item
                const int per_seq = p.hslots * p.tiles_per_seq;
                atomicMax(p.work, (unsigned)((v / per_seq + 1) * per_seq - v_static));
            }
            continue;
        }
        if (!(ok = publish(it))) break;
        if (it.ntiles == 0) continue;
        if (qi >= 1) ok = mbar_wait(smem_u32(&b.q_empty), (qi - 1) & 1, ctx, abort);
        if (!ok) break;
        const uint32_t qbar = smem_u32(&b.q_full);
        mbar_arrive_expect_tx(qbar, Q_TILE);
        tma_load_3d(smem_u32(sm.q), tq, qbar, 0, it.h, it.q_row0);
        tma_load_3d(smem_u32(sm.q) + Q_HALF, tq, qbar, 64, it.h, it.q_row0);
        ++qi;
        TileIter<MODE> ti(it);
        int prev_row = 0;
        for (int j = 0; j < it.ntiles; ++j) {
            const int row = it.key_row0 + ti.next(p, it);
            if (!(ok = load_k(it, row))) break;
            if (j >= 1 && !(ok = load_v(it.g, prev_row))) break;
            prev_row = row;
        }
        if (ok) ok = load_v(it.g, prev_row);
        if (!ok) break;
    }
    if (ok) {
        Item end{};  // valid = false: no more items
        ok = publish(end);
    }
    {
        // Let copies already in flight land before the CTA leaves (bounded;
        // on the normal path every phase waited for here has completed, and
        // after an abort of another role loads may still be in flight).
        int zero = 0;
        if (qi > 0) mbar_wait(smem_u32(&b.q_full), (qi - 1) & 1, ctx, &zero);
        for (int i = 1; i <= KSTAGES && i <= kt; ++i)
            mbar_wait(smem_u32(&b.k_full[(kt - i) % KSTAGES]), ((kt - i) / KSTAGES) & 1, ctx, &zero);
        for (int i = 1; i <= VSTAGES && i <= vt; ++i)
            mbar_wait(smem_u32(&b.v_full[(vt - i) % VSTAGES]), ((vt - i) / VSTAGES) & 1, ctx, &zero);
    }
}

// ------------------------------------------------------------------ MMA issuer

template <int MODE, bool LOOK>
__device__ void mma_issuer(const TcParams &p, Slot &sm, Bars &b, volatile int *abort,
                           uint32_t tmem, int first, int stride, const DevCtx &ctx) {
    int qi = 0, kt = 0, pc = 0;
    bool ok = true;
    const uint32_t o_tmem = tmem + O_COL;
    // descriptors per buffer (two stages each, selected so they stay in registers)
    static_assert(KSTAGES == 2 && VSTAGES == 2, "descriptor selection assumes two stages");
    const uint64_t dq = smem_desc_sw128(smem_u32(sm.q), 16u, 1024u);
    const uint64_t dk0 = smem_desc_sw128(smem_u32(sm.k[0]), 16u, 1024u);
    const uint64_t dk1 = smem_desc_sw128(smem_u32(sm.k[1]), 16u, 1024u);
    const uint64_t dv0 = smem_desc_sw128(smem_u32(sm.v[0]), KV_HALF, 1024u);
    const uint64_t dv1 = smem_desc_sw128(smem_u32(sm.v[1]), KV_HALF, 1024u);
    if (ctx.stall) mbar_wait(smem_u32(&b.drain), 0, ctx, abort);  // test hook: runs out
    if constexpr (!LOOK) {
        for (int ic = 0; ok; ++ic) {
            const int slot_k = ic % ITEM_RING;
            if (!mbar_wait(smem_u32(&b.item_full[slot_k]), (ic / ITEM_RING) & 1, ctx, abort)) break;
            const Item it = b.item[slot_k];
            mbar_arrive(smem_u32(&b.item_empty[slot_k]));
            if (!it.valid) break;
            if (it.ntiles == 0) continue;
            ok = mbar_wait(smem_u32(&b.q_full), qi & 1, ctx, abort);
            const int n = it.ntiles, kt0 = kt;
            auto issue_pv = [&](int jj) -> bool {
                const int st = (kt0 + jj) % VSTAGES, use = (kt0 + jj) / VSTAGES;
                // the stage and O waits first, P (written by the softmax, the one
                // this thread usually waits for) last: each barrier access of this
                // thread stalls the MMAs in flight, so the last one should be the
                // one that releases the issue
                if (!mbar_wait(smem_u32(&b.v_full[st]), use & 1, ctx, abort)) return false;
                if (jj == 0 && qi >= 1 &&
                    !mbar_wait(smem_u32(&b.o_empty), (qi - 1) & 1, ctx, abort))
                    return false;
                if (!mbar_wait(smem_u32(&b.p_full[pc & 1]), (pc >> 1) & 1, ctx, abort)) return false;
                tc_fence_after();
                const uint64_t dv = st ? dv1 : dv0;
                const uint32_t p_tmem = tmem + P_COL + 32u * (uint32_t)(pc & 1);
                const uint32_t acc0 = jj > 0 ? 1u : 0u;
    #pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    tc_mma_f16_ts(o_tmem, p_tmem + 8u * kk, dv + mnoff(kk), IDESC_PV,
                                  kk > 0 ? 1u : acc0);
                tc_commit(smem_u32(&b.v_empty[st]));
                tc_commit(smem_u32(&b.pv_done));
                ++pc;
                return true;
            };
            for (int j = 0; ok && j < n; ++j) {
                // one S buffer: tile t may start once the softmax has loaded tile t-1
                const int t = kt0 + j, st = t % KSTAGES, use = t / KSTAGES;
                // the key stage first, the softmax's release of S last (as above)
                ok = mbar_wait(smem_u32(&b.k_full[st]), use & 1, ctx, abort);
                if (ok && t >= 1) ok = mbar_wait(smem_u32(&b.s_empty), (t - 1) & 1, ctx, abort);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dk = st ? dk1 : dk0;
                const uint32_t s_tmem = tmem + S_COL;
    #pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    tc_mma_f16(s_tmem, dq + koff(kk, Q_HALF), dk + koff(kk, KV_HALF), IDESC_S,
                               kk > 0 ? 1u : 0u);
                tc_commit(smem_u32(&b.k_empty[st]));
                tc_commit(smem_u32(&b.s_full));
                if (j == n - 1) tc_commit(smem_u32(&b.q_empty));
                if (j >= 1) ok = issue_pv(j - 1);
            }
            if (ok) ok = issue_pv(n - 1);
            if (ok) tc_commit(smem_u32(&b.o_full));
            ++qi;
            kt += n;
        }
    } else {
        // Lookahead: an item's last P V is issued after the next item's first S,
        // so that the next scores are computed while the softmax ends the item
        // (which hides the next item's Q load). The softmax then defers that
        // item's epilogue past the next item's first tile: the last P V waits for
        // this thread to have taken the next item with key tiles from the ring,
        // which the softmax must keep draining instead of waiting for O.
        auto issue_pv = [&](int kt0, int jj, int q) -> bool {
            const int st = (kt0 + jj) % VSTAGES, use = (kt0 + jj) / VSTAGES;
            if (!mbar_wait(smem_u32(&b.v_full[st]), use & 1, ctx, abort)) return false;
            if (jj == 0 && q >= 1 && !mbar_wait(smem_u32(&b.o_empty), (q - 1) & 1, ctx, abort))
                return false;
            if (!mbar_wait(smem_u32(&b.p_full[pc & 1]), (pc >> 1) & 1, ctx, abort)) return false;
            tc_fence_after();
            const uint64_t dv = st ? dv1 : dv0;
            const uint32_t p_tmem = tmem + P_COL + 32u * (uint32_t)(pc & 1);
            const uint32_t acc0 = jj > 0 ? 1u : 0u;
    #pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
                tc_mma_f16_ts(o_tmem, p_tmem + 8u * kk, dv + mnoff(kk), IDESC_PV, kk > 0 ? 1u : acc0);
            tc_commit(smem_u32(&b.v_empty[st]));
            tc_commit(smem_u32(&b.pv_done));
            ++pc;
            return true;
        };
        auto issue_s = [&](int t, bool last_of_item) -> bool {
            const int st = t % KSTAGES, use = t / KSTAGES;
            if (!mbar_wait(smem_u32(&b.k_full[st]), use & 1, ctx, abort)) return false;
            if (t >= 1 && !mbar_wait(smem_u32(&b.s_empty), (t - 1) & 1, ctx, abort)) return false;
            tc_fence_after();
            const uint64_t dk = st ? dk1 : dk0;
            const uint32_t s_tmem = tmem + S_COL;
    #pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk)
                tc_mma_f16(s_tmem, dq + koff(kk, Q_HALF), dk + koff(kk, KV_HALF), IDESC_S,
                           kk > 0 ? 1u : 0u);
            tc_commit(smem_u32(&b.k_empty[st]));
            tc_commit(smem_u32(&b.s_full));
            if (last_of_item) tc_commit(smem_u32(&b.q_empty));
            return true;
        };
        int pend_kt0 = -1, pend_j = 0, pend_q = 0;  // pending last P V (pend_kt0 < 0: none)
        auto flush = [&]() -> bool {
            if (pend_kt0 < 0) return true;
            if (!issue_pv(pend_kt0, pend_j, pend_q)) return false;
            tc_commit(smem_u32(&b.o_full));
            pend_kt0 = -1;
            return true;
        };
        for (int ic = 0; ok; ++ic) {
            const int slot_k = ic % ITEM_RING;
            if (!mbar_wait(smem_u32(&b.item_full[slot_k]), (ic / ITEM_RING) & 1, ctx, abort)) {
                ok = false;
                break;
            }
            const Item it = b.item[slot_k];
            mbar_arrive(smem_u32(&b.item_empty[slot_k]));
            if (!it.valid) break;
            if (it.ntiles == 0) continue;
            const int n = it.ntiles, kt0 = kt;
            ok = mbar_wait(smem_u32(&b.q_full), qi & 1, ctx, abort) && issue_s(kt0, n == 1) && flush();
            for (int j = 1; ok && j < n; ++j)
                ok = issue_s(kt0 + j, j == n - 1) && issue_pv(kt0, j - 1, qi);
            pend_kt0 = kt0;
            pend_j = n - 1;
            pend_q = qi;
            ++qi;
            kt += n;
        }
        if (ok) ok = flush();
    }
    // Every tcgen05 operation issued above completes before TMEM is released.
    tc_commit(smem_u32(&b.drain));
    int zero = 0;
    mbar_wait(smem_u32(&b.drain), 0, ctx, &zero);
}

// ------------------------------------------------------------------ softmax / epilogue

template <int MODE, bool LOOK>
__device__ void softmax_role(const TcParams &p, const CUtensorMap *to, Slot &slot, Bars &b,
                             volatile int *abort,
                             uint32_t tmem, int first, int stride, const DevCtx &ctx) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row within the tile == TMEM lane
    // the row's token (from the tile's first) and head (from the item's first)
    const int gs = MODE == MODE_WINDOW ? p.gshift : 0;
    const int tok = r >> gs, hl = r & ((1 << gs) - 1);
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t o_tmem = tmem + O_COL + lane_off;
    int sc = 0, pc = 0, qi = 0;  // sc: tiles seen, pc: P tiles written
    bool ok = true;
    // The epilogue of an item runs as soon as the item's last P V has
    // completed; the MMA thread issues the next item's first S right after
    // that P V, so those scores are computed while the epilogue runs.
    struct Out {
        int q_row0, nq, h;
        float m, l;
        size_t row_off;  // block: the chunk's first output row
    };
    Out pend{0, 0, 0, 0.f, 0.f, 0};
    bool pend_valid = false;  // lookahead: the epilogue waits for the next item's first tile
    auto epilogue = [&](const Out &pe) -> bool {
        if (!mbar_wait(smem_u32(&b.o_full), qi & 1, ctx, abort)) return false;
        tc_fence_after();
        const float inv = pe.l > 0.0f ? 1.0f / pe.l : 0.0f;
        // block: the chunk's rows; window: no offset (folded at compile time)
        const size_t roff = MODE == MODE_BLOCK ? pe.row_off : 0;
        const size_t orow = roff + (size_t)(pe.q_row0 + tok) * p.H + pe.h + hl;
        // Each pass covers 128 bytes of every row: this thread's row goes to
        // the warp's staging buffer (128B-swizzled, conflict-free). Window
        // warps whose 32 rows all belong to the item hand the buffer to one
        // bulk tensor store; otherwise the warp writes 4 whole rows (4 lines)
        // per store instruction, skipping rows past the item.
        {
            const bool bulk = MODE == MODE_WINDOW && quarter * 32 + 32 <= pe.nq;
            const uint32_t sb = smem_u32(slot.stage[quarter]);
            constexpr int PASSES = MODE == MODE_WINDOW ? 2 : 4;  // bf16: 64 d, fp32: 32 d per pass
            constexpr int ROW_BYTES = MODE == MODE_WINDOW ? HD * 2 : HD * 4;
            uint8_t *const obase = MODE == MODE_WINDOW ? reinterpret_cast<uint8_t *>(p.o)
                                                       : reinterpret_cast<uint8_t *>(p.o_part);
#pragma unroll 1
            for (int pass = 0; pass < PASSES; ++pass) {
                uint32_t w[32];  // this row's 128 bytes
                if (MODE == MODE_WINDOW) {
                    uint32_t ov[2][32];
                    tmem_ld32(o_tmem + 64u * pass, ov[0]);
                    tmem_ld32(o_tmem + 64u * pass + 32u, ov[1]);
                    tc_wait_ld();
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            w[16 * cc + e] = pack_bf16x2(__uint_as_float(ov[cc][2 * e]) * inv,
                                                         __uint_as_float(ov[cc][2 * e + 1]) * inv);
                } else {
                    uint32_t ov[32];
                    tmem_ld32(o_tmem + 32u * pass, ov);
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(__uint_as_float(ov[e]) * inv);
                }
                if (pass == PASSES - 1) {  // O fully read: the next item's first P V may overwrite it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&b.o_empty));
                }
                if (MODE == MODE_WINDOW) {  // an earlier bulk store may still read the buffer
                    if (lane == 0) bulk_wait_read();
                    __syncwarp();
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                     sb + (uint32_t)lane * 128u + (((uint32_t)u ^ (lane & 7u)) << 4)),
                                 "r"(w[4 * u]), "r"(w[4 * u + 1]), "r"(w[4 * u + 2]), "r"(w[4 * u + 3])
                                 : "memory");
                if (bulk) {
                    fence_proxy_async_smem();  // the rows are read by the bulk copy
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(to, sb, pass * 64, pe.h, pe.q_row0 + ((quarter * 32) >> gs));
                        bulk_commit();
                    }
                    continue;
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rw = 4 * i + (lane >> 3), unit = lane & 7;  // row in the warp, 16-B unit
                    uint4 v;
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                                 : "r"(sb + (uint32_t)rw * 128u + (((uint32_t)unit ^ ((uint32_t)rw & 7u)) << 4)));
                    const int rr = quarter * 32 + rw;
                    if (rr < pe.nq) {
                        const size_t grow = roff + (size_t)(pe.q_row0 + (rr >> gs)) * p.H + pe.h +
                                            (rr & ((1 << gs) - 1));
                        *reinterpret_cast<uint4 *>(obase + grow * ROW_BYTES + pass * 128 + unit * 16) = v;
                    }
                }
                __syncwarp();  // the buffer is rewritten by the next pass
            }
        }
        if (r < pe.nq) {
            const float lse = pe.l > 0.0f ? (pe.m + log2f(pe.l)) * LN2 : -INFINITY;
            if (MODE == MODE_WINDOW) {
                if (p.lse) p.lse[orow] = lse;
            } else {
                p.lse_part[orow] = lse;
            }
        }
        ++qi;
        return true;
    };
    for (int ic = 0; ok; ++ic) {
        const int slot_k = ic % ITEM_RING;
        if (!mbar_wait(smem_u32(&b.item_full[slot_k]), (ic / ITEM_RING) & 1, ctx, abort)) {
            ok = false;
            break;
        }
        const Item it = b.item[slot_k];
        const float sink = MODE == MODE_WINDOW ? b.item[slot_k].sink[hl] : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&b.item_empty[slot_k]));
        if (!it.valid) break;
        const bool row_valid = r < it.nq;
        if (it.ntiles == 0) {  // block mode: nothing visible in this chunk
            if (MODE == MODE_BLOCK && row_valid) {
                const size_t orow = (size_t)it.L * p.M * p.H + (size_t)(it.q_row0 + tok) * p.H + it.h + hl;
                float4 *dst = reinterpret_cast<float4 *>(p.o_part + orow * HD);
#pragma unroll 8
                for (int i = 0; i < HD / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                p.lse_part[orow] = -INFINITY;
            }
            continue;
        }
        const bool warp_all_valid = __all_sync(FULL, row_valid);
        // visible key interval of this row (window: fixed for the item)
        const int qi_loc = it.qpos0 + tok;
        constexpr int NONE_LO = 1 << 30, NONE_HI = -(1 << 30);  // empty interval
        int lo_r = NONE_LO, hi_r = NONE_HI;
        if (MODE == MODE_WINDOW && row_valid) {
            lo_r = p.wl < 0 ? 0 : max(0, qi_loc - p.wl);
            hi_r = p.wr < 0 ? it.L - 1 : min(it.L - 1, qi_loc + p.wr);
            if (p.causal) hi_r = min(hi_r, qi_loc);
        }
        const bool null_sink = MODE == MODE_WINDOW && p.sink_mode == 2;
        const bool key0 = MODE == MODE_WINDOW && p.sink_mode == 1;
        float m_run = null_sink ? sink * LOG2E : -INFINITY;
        float l = null_sink ? 1.0f : 0.0f;
        const uint64_t scale2 = f2_pack(p.scale_l2, p.scale_l2);
        // warp-level: union of the rows' intervals (for skipping) and their
        // intersection (chunks inside it need no masking); fixed per item in
        // window mode, per tile in block mode
        int wlo = __reduce_min_sync(FULL, lo_r);
        int whi = __reduce_max_sync(FULL, hi_r);
        int ilo = __reduce_max_sync(FULL, row_valid ? lo_r : INT_MIN);
        int ihi = __reduce_min_sync(FULL, row_valid ? hi_r : INT_MAX);
        TileIter<MODE> ti(it);
        for (int j = 0; j < it.ntiles; ++j) {
            const int base = ti.next(p, it);
            if (MODE == MODE_BLOCK) {
                if (row_valid) {
                    lo_r = max(base, it.lo);
                    hi_r = min(base + BN - 1, it.hi - 1);
                    if (p.causal) hi_r = min(hi_r, qi_loc);
                } else {
                    lo_r = NONE_LO;
                    hi_r = NONE_HI;
                }
                wlo = __reduce_min_sync(FULL, lo_r);
                whi = __reduce_max_sync(FULL, hi_r);
                ilo = __reduce_max_sync(FULL, row_valid ? lo_r : INT_MIN);
                ihi = __reduce_min_sync(FULL, row_valid ? hi_r : INT_MAX);
            }
            if (!mbar_wait(smem_u32(&b.s_full), sc & 1, ctx, abort)) { ok = false; break; }
            tc_fence_after();
            uint32_t x[2][32];
            unsigned live = 0, full = 0;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int k0 = base + 32 * c;
                if (!(k0 + 31 < wlo || k0 > whi)) {
                    live |= 1u << c;
                    if (warp_all_valid && k0 >= ilo && k0 + 31 <= ihi) full |= 1u << c;
                    tmem_ld32(tmem + S_COL + 32u * c + lane_off, x[c]);
                }
            }
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&b.s_empty));
            ++sc;
            // key-0 bias, in raw score units, on the sequence's first key
            if (key0 && base == 0 && (live & 1u))
                x[0][0] = __float_as_uint(__uint_as_float(x[0][0]) + sink * p.inv_scale);
            // mask partial chunks; maximum of the raw scores
            float mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // independent chains
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (!(live >> c & 1u)) continue;
                if (!(full >> c & 1u)) {
                    const int a = lo_r - (base + 32 * c), z = hi_r - (base + 32 * c);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (e < a || e > z) x[c][e] = __float_as_uint(-INFINITY);
                }
#pragma unroll
                for (int e = 0; e < 32; e += 2)
                    mr[(e >> 1) & 3] = max3(mr[(e >> 1) & 3], __uint_as_float(x[c][e]),
                                            __uint_as_float(x[c][e + 1]));
            }
            const float mraw = fmaxf(max3(mr[0], mr[1], mr[2]), mr[3]);
            const float mt = mraw * p.scale_l2;
            const bool upd = mt > m_run + TAU;
            float alpha = 1.0f;
            if (upd) {
                alpha = (m_run == -INFINITY) ? 0.0f : ex2(m_run - mt);
                l *= alpha;
                m_run = mt;
            }
            if (j >= 1 && __any_sync(FULL, upd)) {
                // O is rescaled in place: the previous P V must have finished.
                // (S of this tile complete implies the P V before that one has,
                // so this parity wait cannot alias.)
                if (!mbar_wait(smem_u32(&b.pv_done), (pc - 1) & 1, ctx, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(o_tmem + 32u * c, ov);
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                    tmem_st32(o_tmem + 32u * c, ov);
                }
                tc_wait_st();
            }
            const float mu = (m_run == -INFINITY) ? 0.0f : m_run;
            const uint64_t negm2 = f2_pack(-mu, -mu);
            uint64_t lsum = f2_pack(0.f, 0.f), lsum2 = f2_pack(0.f, 0.f);
            uint32_t pw[32];  // P as bf16 pairs: word w holds keys 2w (low half) and 2w+1
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (live >> c & 1u) {
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const uint64_t arg = f2_fma(
                            f2_pack(__uint_as_float(x[c][e]), __uint_as_float(x[c][e + 1])),
                            scale2, negm2);
                        float a0, a1;
                        f2_unpack(arg, a0, a1);
                        a0 = ex2(a0);
                        a1 = ex2(a1);
                        if (e & 2) lsum2 = f2_add(lsum2, f2_pack(a0, a1));
                        else lsum = f2_add(lsum, f2_pack(a0, a1));
                        pw[16 * c + e / 2] = pack_bf16x2(a0, a1);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) pw[16 * c + e] = 0u;
                }
            }
            {
                float s0, s1, s2, s3;
                f2_unpack(lsum, s0, s1);
                f2_unpack(lsum2, s2, s3);
                l += (s0 + s1) + (s2 + s3);
            }
            tmem_st32(tmem + P_COL + 32u * (uint32_t)(pc & 1) + lane_off, pw);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&b.p_full[pc & 1]));
            ++pc;
            if (LOOK && j == 0 && pend_valid) {
                if (!(ok = epilogue(pend))) break;
                pend_valid = false;
            }
        }
        if (!ok) break;
        const Out out{it.q_row0, it.nq, it.h, m_run, l,
                      MODE == MODE_BLOCK ? (size_t)it.L * p.M * p.H : 0};
        if (LOOK) {
            pend = out;
            pend_valid = true;
        } else {
            ok = epilogue(out);
        }
    }
    if (LOOK && ok && pend_valid) epilogue(pend);
    if (MODE == MODE_WINDOW && lane == 0) bulk_wait_all();  // before the CTA's shared memory goes
}

template <int MODE, bool LOOK>
__global__ void __launch_bounds__(NTHREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap to,
               const __grid_constant__ CUtensorMap tv, const TcParams p, const DevCtx ctx) {
    extern __shared__ __align__(1024) uint8_t dsmem[];
    Smem &sm = *reinterpret_cast<Smem *>(dsmem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The 128B swizzle pattern is anchored to 1024-byte boundaries of the
    // shared window; the layout above relies on an aligned base.
    if (smem_u32(dsmem) & 1023u) {
        if (threadIdx.x == 0) record_error(ctx, DEVERR_LAYOUT);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < NSLOTS; ++s) {
            Bars &b = sm.bars[s];
            for (int i = 0; i < KSTAGES; ++i) {
                mbar_init(smem_u32(&b.k_full[i]), 1);
                mbar_init(smem_u32(&b.k_empty[i]), 1);
            }
            for (int i = 0; i < VSTAGES; ++i) {
                mbar_init(smem_u32(&b.v_full[i]), 1);
                mbar_init(smem_u32(&b.v_empty[i]), 1);
            }
            mbar_init(smem_u32(&b.s_full), 1);
            mbar_init(smem_u32(&b.s_empty), 4);
            mbar_init(smem_u32(&b.q_full), 1);
            mbar_init(smem_u32(&b.q_empty), 1);
            mbar_init(smem_u32(&b.p_full[0]), 4);
            mbar_init(smem_u32(&b.p_full[1]), 4);
            mbar_init(smem_u32(&b.pv_done), 1);
            mbar_init(smem_u32(&b.o_full), 1);
            mbar_init(smem_u32(&b.o_empty), 4);
            mbar_init(smem_u32(&b.drain), 1);
            for (int i = 0; i < ITEM_RING; ++i) {
                mbar_init(smem_u32(&b.item_full[i]), 1);
                mbar_init(smem_u32(&b.item_empty[i]), 1 + 4);  // MMA issuer + softmax warps
            }
        }
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
    // slot s: warps 2s (producer), 2s+1 (MMA), 4+4s .. 7+4s (softmax)
    const int slot = warp < 2 * NSLOTS ? warp >> 1 : (warp - 2 * NSLOTS) >> 2;
    const uint32_t tmem = sm.tmem_base + (uint32_t)slot * SLOT_COLS;
    const int first = blockIdx.x * NSLOTS + slot, stride = gridDim.x * NSLOTS;
    if (warp < 2 * NSLOTS) {
        if (lane == 0) {
            if ((warp & 1) == 0)
                producer<MODE>(p, &tq, &tk, &tv, sm.slot[slot], sm.bars[slot], &sm.abort, first,
                               stride, ctx);
            else
                mma_issuer<MODE, LOOK>(p, sm.slot[slot], sm.bars[slot], &sm.abort, tmem, first, stride,
                                 ctx);
        }
        __syncwarp();
    } else {
        softmax_role<MODE, LOOK>(p, &to, sm.slot[slot], sm.bars[slot], &sm.abort, tmem, first, stride,
                           ctx);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(sm.tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

CUresult make_map(CUtensorMap *m, const void *base, int rows, int heads, uint32_t box_heads,
                  uint32_t box_rows) {
    const uint64_t dims[3] = {(uint64_t)HD, (uint64_t)heads, (uint64_t)rows};
    const uint64_t strides[2] = {(uint64_t)HD * 2, (uint64_t)HD * 2 * heads};
    const uint32_t box[3] = {64, box_heads, box_rows};
    return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                             strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int MODE, bool LOOK> cudaError_t launch(const TcParams &p_in, const void *q, int q_rows,
                                       const void *k, const void *v, int kv_rows,
                                       const DevInfo &dev, cudaStream_t s) {
    TcParams p = p_in;
    for (const void *ptr : {q, k, v})
        if (reinterpret_cast<uintptr_t>(ptr) & 15u) return cudaErrorMisalignedAddress;
    CUtensorMap tq, tk, tv, to;
    // Q tiles: 128 rows = BM >> gshift tokens x (1 << gshift) heads, token-major
    const int G = 1 << p.gshift;
    if (make_map(&tq, q, q_rows, p.H, G, BM / G) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (make_map(&tk, k, kv_rows, p.Hkv, 1, BN) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (make_map(&tv, v, kv_rows, p.Hkv, 1, BN) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    // window: o [T, H, d] bf16 in 32-row boxes for the epilogue's bulk stores
    // (block mode writes its fp32 partials with plain stores; the map is unused)
    if (make_map(&to, MODE == MODE_WINDOW ? (const void *)p.o : q, q_rows, p.H, G, 32 / G) !=
        CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(Smem);
    cudaError_t e = ensure_smem_attr((const void *)attn_tc_kernel<MODE, LOOK>, smem, dev);
    if (e != cudaSuccess) return e;
    const int streams = (p.num_items + NSLOTS - 1) / NSLOTS;
    const int grid = streams < dev.sm_count ? streams : dev.sm_count;
    if (!(p.work = launch_claim_counter(dev, s, &e))) return e;
    const DevCtx ctx = make_ctx(dev);
    if (verbose())
        fprintf(stderr,
                "sattn: attn_tc_kernel<%s%s> grid=%d block=%d smem=%zu slots=%d items=%d\n",
                MODE == MODE_WINDOW ? "window" : "block", LOOK ? ", lookahead" : "", grid,
                NTHREADS, smem, NSLOTS, p.num_items);
    attn_tc_kernel<MODE, LOOK><<<grid, NTHREADS, smem, s>>>(tq, tk, to, tv, p, ctx);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_window_tc(const WindowArgs &a, const DevInfo &dev, cudaStream_t s) {
    TcParams p{};
    p.H = a.H;
    p.Hkv = a.Hkv;
    p.groups = a.H / a.Hkv;
    p.scale_l2 = a.scale * LOG2E;
    p.inv_scale = 1.0f / a.scale;
    p.cu_seqlens = a.cu_seqlens;
    p.num_seqs = a.num_seqs;
    p.T = a.T;
    // Query heads that share a KV head are packed into one tile (the largest
    // power of two dividing H / Hkv, at most 8): a tile of BM / G tokens has a
    // narrower key band than one of BM tokens, and its K/V tiles serve G heads.
    int gs = 0;
    while (gs < 3 && p.groups % (2 << gs) == 0) ++gs;
    p.gshift = gs;
    p.hslots = a.H >> gs;
    p.tiles_per_seq = (a.max_seqlen + (BM >> gs) - 1) / (BM >> gs);
    p.wl = a.wl;
    p.wr = a.wr;
    p.causal = a.causal;
    p.sinks = a.sinks;
    p.sink_mode = a.sink_mode;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.lse = a.lse;
    const long long items = (long long)a.num_seqs * p.tiles_per_seq * p.hslots;
    if (items > INT_MAX) return cudaErrorInvalidValue;
    p.num_items = (int)items;
    if (reinterpret_cast<uintptr_t>(a.o) & 15u) return cudaErrorMisalignedAddress;
    // packed heads make short items (fewer key tiles per row): there, issuing
    // the next item's first S before an item's last P V measured faster; with
    // one head per tile the plain order did
    return p.gshift > 0 ? launch<MODE_WINDOW, true>(p, a.q, a.T, a.k, a.v, a.T, dev, s)
                        : launch<MODE_WINDOW, false>(p, a.q, a.T, a.k, a.v, a.T, dev, s);
}

cudaError_t launch_block_tc(const BlockArgs &a, const DevInfo &dev, cudaStream_t s) {
    if (a.kv_end <= a.kv_begin) return launch_block_simt(a, dev, s);  // nothing to gather
    TcParams p{};
    p.H = a.H;
    p.Hkv = a.Hkv;
    p.groups = a.H / a.Hkv;
    p.scale_l2 = a.scale * LOG2E;
    p.inv_scale = 1.0f / a.scale;
    p.mask = a.mask;
    p.M = a.M;
    p.Nctx = a.Nctx;
    p.q_pos0 = a.q_pos0;
    p.kv_begin = a.kv_begin;
    p.kv_end = a.kv_end;
    p.causal = a.causal;
    p.QB = (a.M + BM - 1) / BM;
    p.KB = (a.Nctx + 127) / 128;
    p.o_part = a.o_part;
    p.lse_part = a.lse_part;
    // chunk 0 (or a chunk as long as the range): one output for the range
    const int len = a.kv_end - a.kv_begin;
    p.chunk_keys = a.chunk > 0 && a.chunk < len ? a.chunk : len;
    const long long chunks = (len + p.chunk_keys - 1) / p.chunk_keys;
    const long long items = (long long)p.QB * a.H * chunks;
    if (items > INT_MAX) return cudaErrorInvalidValue;
    p.num_items = (int)items;
    if (reinterpret_cast<uintptr_t>(a.o_part) & 15u) return cudaErrorMisalignedAddress;
    return launch<MODE_BLOCK, false>(p, a.q, a.M, a.k, a.v, a.Nctx, dev, s);
}

}  // namespace sattn
