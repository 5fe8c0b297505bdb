// Tensor-core attention over contiguous key tiles (tcgen05 + TMEM + TMA).
//
// Two uses share this engine:
//  * sliding-window varlen attention with sinks ("PR #49815 report": window
//    |i-j| <= w inside each sequence, key-0 bias or null-logit sink). Only
//    the key tiles that intersect a query tile's band are visited (the report
//    notes that visiting every block and masking costs O(seq_len^2));
//  * one KV chunk of block-sparse causal attention ("XAttention Offload
//    Stream Synchronization Fix": per-chunk partial stats, merged later);
//    the key tiles are the selected 128-key blocks of the chunk.
//
// A work item is (128-query tile, query head). A persistent grid of one CTA
// per SM walks the items; each CTA has three roles:
//   warp 0        TMA producer: Q tile (double-buffered), K and V tiles
//                 (two stages each), 128B-swizzled, K-major rows of 256 B.
//   warp 1        MMA issuer (one thread): S = Q K^T into TMEM (two S
//                 buffers), then O += P V into TMEM (two O buffers).
//   warps 2..5    softmax + epilogue: thread = query row = TMEM lane. Each
//                 row keeps its running max m and sum l in the log2 domain;
//                 P (bf16) goes to shared memory as the A operand of P V.
// The running max is only moved when a tile raises it by more than 2^8, so
// the accumulator in TMEM is rarely rescaled (P <= 256 otherwise, exact in
// fp32 sums). Null-logit sinks start from m = sink, l = 1; key-0 sinks add
// the sink to key 0's logit where it is visible.
#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace sattn {
namespace {

constexpr int BM = 128;                  // queries per tile (TMEM lanes)
constexpr int BN = 128;                  // keys per tile
constexpr int HD = 128;                  // head dim
constexpr uint32_t TILE = BM * HD * 2;   // bytes of one bf16 128x128 tile
constexpr uint32_t HALF = TILE / 2;      // one 64-column (128-byte) swizzled half
constexpr int NTHREADS = 192;
constexpr float TAU = 8.0f;              // rescale threshold (log2 units)

enum : int { MODE_WINDOW = 0, MODE_BLOCK = 1 };

struct TcParams {
    int H, Hkv, groups, num_items;
    float scale_l2;  // scale * log2(e)
    // window
    const int32_t *cu_seqlens;
    int num_seqs, T, tiles_per_seq, wl, wr, causal;
    const float *sinks;
    int sink_mode;
    __nv_bfloat16 *o;
    float *lse;
    // block
    const uint8_t *mask;
    int M, Nctx, q_pos0, kv_begin, kv_end, QB, KB;
    float *o_part, *lse_part;
};

struct __align__(1024) Smem {
    uint8_t q[2][TILE];
    uint8_t k[2][TILE];
    uint8_t v[2][TILE];
    uint8_t p[TILE];
};

struct Bars {
    uint64_t q_full[2], q_empty[2], k_full[2], k_empty[2], v_full[2], v_empty[2];
    uint64_t s_full[2], s_empty[2], p_full, p_empty, o_full[2], o_empty[2], drain;
    uint32_t tmem_base;
    int abort;
};

struct Item {
    bool valid;
    bool seq_err;
    int h, g, nq, ntiles;
    int q_row0;    // first row of the tile in q / o (token index)
    int key_row0;  // global K/V row of key coordinate 0
    int qpos0;     // window: local index of query row 0; block: absolute position
    int lo, hi, L; // window: key band of the tile (local), sequence length
    const uint8_t *mrow;
    int kb_lo, kb_hi;
};

template <int MODE> __device__ __forceinline__ Item decode_item(const TcParams &p, int v) {
    Item it;
    it.valid = false;
    it.seq_err = false;
    it.ntiles = 0;
    it.h = v % p.H;
    it.g = it.h / p.groups;
    const int rest = v / p.H;
    if (MODE == MODE_WINDOW) {
        const int t = rest % p.tiles_per_seq, s = rest / p.tiles_per_seq;
        const int s0 = __ldg(p.cu_seqlens + s), s1 = __ldg(p.cu_seqlens + s + 1);
        if (s0 < 0 || s1 < s0 || s1 > p.T || __ldg(p.cu_seqlens) != 0 ||
            s1 - s0 > p.tiles_per_seq * BM) {
            it.seq_err = true;
            return it;
        }
        it.L = s1 - s0;
        const int qs = t * BM;
        if (qs >= it.L) return it;
        it.nq = min(BM, it.L - qs);
        it.q_row0 = s0 + qs;
        it.key_row0 = s0;
        it.qpos0 = qs;
        const int last = qs + it.nq - 1;
        it.lo = p.wl < 0 ? 0 : max(0, qs - p.wl);
        it.hi = p.wr < 0 ? it.L - 1 : min(it.L - 1, last + p.wr);
        if (p.causal) it.hi = min(it.hi, last);
        it.ntiles = (it.hi - it.lo + BN) / BN;
        it.valid = true;
    } else {
        const int qb = rest;
        const int qs = qb * BM;
        it.nq = min(BM, p.M - qs);
        it.q_row0 = qs;
        it.key_row0 = 0;
        it.qpos0 = p.q_pos0 + qs;
        int end = p.kv_end;
        if (p.causal) end = min(end, it.qpos0 + it.nq);
        it.kb_lo = p.kv_begin / BN;
        it.kb_hi = end > p.kv_begin ? (end - 1) / BN : it.kb_lo - 1;
        it.mrow = p.mask + ((size_t)it.h * p.QB + qb) * p.KB;
        int n = 0;
        for (int kb = it.kb_lo; kb <= it.kb_hi; ++kb) n += __ldg(it.mrow + kb) != 0;
        it.ntiles = n;
        it.valid = true;
    }
    return it;
}

// Key coordinate of the first key of each successive tile of an item.
template <int MODE> struct TileIter {
    int j, kb;
    __device__ explicit TileIter(const Item &it) : j(0), kb(it.kb_lo - 1) {}
    __device__ int next(const Item &it) {
        if (MODE == MODE_WINDOW) return it.lo + BN * (j++);
        do { ++kb; } while (kb <= it.kb_hi && __ldg(it.mrow + kb) == 0);
        ++j;
        return kb * BN;
    }
};

// K-major operand (rows of 128 B, two 64-column halves HALF bytes apart):
// descriptor for the kk-th 16-element K slice.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int kk) {
    return smem_desc_sw128(base + (uint32_t)(kk >> 2) * HALF + (uint32_t)(kk & 3) * 32u, 16u,
                           1024u);
}
// MN-major operand (V: rows = keys, 64-column halves of d HALF bytes apart):
// descriptor for the kk-th 16-key slice.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int kk) {
    return smem_desc_sw128(base + (uint32_t)kk * 2048u, HALF, 1024u);
}

constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, 0, 0);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 128, 0, 1);

// ------------------------------------------------------------------ producer

template <int MODE>
__device__ void producer(const TcParams &p, const CUtensorMap *tq, const CUtensorMap *tk,
                         const CUtensorMap *tv, Smem &sm, Bars &b, const DevCtx &ctx) {
    prefetch_tmap(tq);
    prefetch_tmap(tk);
    prefetch_tmap(tv);
    int qi = 0, kt = 0;
    bool ok = true;
    for (int v = blockIdx.x; ok && v < p.num_items; v += gridDim.x) {
        const Item it = decode_item<MODE>(p, v);
        if (!it.valid || it.ntiles == 0) continue;
        const int qb = qi & 1;
        if (qi >= 2) ok = mbar_wait(smem_u32(&b.q_empty[qb]), ((qi >> 1) - 1) & 1, ctx, &b.abort);
        if (!ok) break;
        const uint32_t qbar = smem_u32(&b.q_full[qb]);
        mbar_arrive_expect_tx(qbar, TILE);
        tma_load_3d(smem_u32(sm.q[qb]), tq, qbar, 0, it.h, it.q_row0);
        tma_load_3d(smem_u32(sm.q[qb]) + HALF, tq, qbar, 64, it.h, it.q_row0);
        ++qi;
        TileIter<MODE> ti(it);
        for (int j = 0; j < it.ntiles; ++j, ++kt) {
            const int row = it.key_row0 + ti.next(it);
            const int st = kt & 1, use = kt >> 1;
            if (use >= 1) ok = mbar_wait(smem_u32(&b.k_empty[st]), (use - 1) & 1, ctx, &b.abort);
            if (!ok) break;
            const uint32_t kbar = smem_u32(&b.k_full[st]);
            mbar_arrive_expect_tx(kbar, TILE);
            tma_load_3d(smem_u32(sm.k[st]), tk, kbar, 0, it.g, row);
            tma_load_3d(smem_u32(sm.k[st]) + HALF, tk, kbar, 64, it.g, row);
            if (use >= 1) ok = mbar_wait(smem_u32(&b.v_empty[st]), (use - 1) & 1, ctx, &b.abort);
            if (!ok) break;
            const uint32_t vbar = smem_u32(&b.v_full[st]);
            mbar_arrive_expect_tx(vbar, TILE);
            tma_load_3d(smem_u32(sm.v[st]), tv, vbar, 0, it.g, row);
            tma_load_3d(smem_u32(sm.v[st]) + HALF, tv, vbar, 64, it.g, row);
        }
    }
    if (!ok) {
        // Let copies already in flight land before the CTA leaves (bounded).
        DevCtx c2 = ctx;
        int zero = 0;
        for (int i = 0; i < 2; ++i) {
            if (qi > i) mbar_wait(smem_u32(&b.q_full[(qi - 1 - i) & 1]), ((qi - 1 - i) >> 1) & 1, c2, &zero);
            if (kt > i) {
                mbar_wait(smem_u32(&b.k_full[(kt - 1 - i) & 1]), ((kt - 1 - i) >> 1) & 1, c2, &zero);
                mbar_wait(smem_u32(&b.v_full[(kt - 1 - i) & 1]), ((kt - 1 - i) >> 1) & 1, c2, &zero);
            }
        }
    }
}

// ------------------------------------------------------------------ MMA issuer

template <int MODE>
__device__ void mma_issuer(const TcParams &p, Smem &sm, Bars &b, uint32_t tmem, const DevCtx &ctx) {
    int qi = 0, kt = 0, sc = 0, pc = 0, oc = 0;
    bool ok = true;
    const uint32_t p_base = smem_u32(sm.p);
    for (int v = blockIdx.x; ok && v < p.num_items; v += gridDim.x) {
        const Item it = decode_item<MODE>(p, v);
        if (!it.valid || it.ntiles == 0) continue;
        const int qb = qi & 1, ob = oc & 1;
        const uint32_t q_base = smem_u32(sm.q[qb]);
        const uint32_t o_tmem = tmem + 256u + (uint32_t)ob * 128u;
        ok = mbar_wait(smem_u32(&b.q_full[qb]), (qi >> 1) & 1, ctx, &b.abort);
        const int n = it.ntiles, kt0 = kt;
        auto issue_pv = [&](int jj) -> bool {
            const int st = (kt0 + jj) & 1, use = (kt0 + jj) >> 1;
            if (!mbar_wait(smem_u32(&b.p_full), pc & 1, ctx, &b.abort)) return false;
            if (!mbar_wait(smem_u32(&b.v_full[st]), use & 1, ctx, &b.abort)) return false;
            if (jj == 0 && oc >= 2 &&
                !mbar_wait(smem_u32(&b.o_empty[ob]), ((oc >> 1) - 1) & 1, ctx, &b.abort))
                return false;
            tc_fence_after();
            const uint32_t v_base = smem_u32(sm.v[st]);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
                tc_mma_f16(o_tmem, desc_kmajor(p_base, kk), desc_mnmajor(v_base, kk), IDESC_PV,
                           (jj > 0 || kk > 0) ? 1u : 0u);
            tc_commit(smem_u32(&b.v_empty[st]));
            tc_commit(smem_u32(&b.p_empty));
            ++pc;
            return true;
        };
        for (int j = 0; ok && j < n; ++j) {
            const int st = (kt0 + j) & 1, use = (kt0 + j) >> 1, sb = sc & 1;
            if (sc >= 2) ok = mbar_wait(smem_u32(&b.s_empty[sb]), ((sc >> 1) - 1) & 1, ctx, &b.abort);
            if (ok) ok = mbar_wait(smem_u32(&b.k_full[st]), use & 1, ctx, &b.abort);
            if (!ok) break;
            tc_fence_after();
            const uint32_t k_base = smem_u32(sm.k[st]);
            const uint32_t s_tmem = tmem + (uint32_t)sb * 128u;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk)
                tc_mma_f16(s_tmem, desc_kmajor(q_base, kk), desc_kmajor(k_base, kk), IDESC_S,
                           kk > 0 ? 1u : 0u);
            tc_commit(smem_u32(&b.k_empty[st]));
            tc_commit(smem_u32(&b.s_full[sb]));
            if (j == n - 1) tc_commit(smem_u32(&b.q_empty[qb]));
            ++sc;
            if (j >= 1) ok = issue_pv(j - 1);
        }
        if (ok) ok = issue_pv(n - 1);
        if (ok) tc_commit(smem_u32(&b.o_full[ob]));
        ++qi;
        ++oc;
        kt += n;
    }
    // Every tcgen05 operation issued above completes before TMEM is released.
    tc_commit(smem_u32(&b.drain));
    int zero = 0;
    mbar_wait(smem_u32(&b.drain), 0, ctx, &zero);
}

// ------------------------------------------------------------------ softmax / epilogue

template <int MODE>
__device__ void softmax_role(const TcParams &p, Smem &sm, Bars &b, uint32_t tmem,
                             const DevCtx &ctx) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t p_base = smem_u32(sm.p);
    const unsigned FULL = 0xffffffffu;
    int sc = 0, pc = 0, oc = 0;
    bool ok = true;
    for (int v = blockIdx.x; ok && v < p.num_items; v += gridDim.x) {
        const Item it = decode_item<MODE>(p, v);
        if (!it.valid) {
            if (it.seq_err && warp == 2 && lane == 0) record_error(ctx, DEVERR_SEQLENS);
            continue;
        }
        const bool row_valid = r < it.nq;
        if (it.ntiles == 0) {  // block mode: nothing visible in this chunk
            if (MODE == MODE_BLOCK && row_valid) {
                const size_t orow = (size_t)(it.q_row0 + r) * p.H + it.h;
                float4 *dst = reinterpret_cast<float4 *>(p.o_part + orow * HD);
#pragma unroll 8
                for (int i = 0; i < HD / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                p.lse_part[orow] = -INFINITY;
            }
            continue;
        }
        // visible key interval of this row (window: fixed for the item)
        const int qi_loc = it.qpos0 + r;
        int lo_r = INT_MAX, hi_r = INT_MIN;
        if (MODE == MODE_WINDOW && row_valid) {
            lo_r = p.wl < 0 ? 0 : max(0, qi_loc - p.wl);
            hi_r = p.wr < 0 ? it.L - 1 : min(it.L - 1, qi_loc + p.wr);
            if (p.causal) hi_r = min(hi_r, qi_loc);
        }
        const bool null_sink = MODE == MODE_WINDOW && p.sink_mode == 2;
        const bool key0 = MODE == MODE_WINDOW && p.sink_mode == 1;
        const float sink_l2 = (MODE == MODE_WINDOW && p.sinks) ? __ldg(p.sinks + it.h) * LOG2E : 0.f;
        float m_run = null_sink ? sink_l2 : -INFINITY;
        float l = null_sink ? 1.0f : 0.0f;
        const int ob = oc & 1;
        const uint32_t o_tmem = tmem + 256u + (uint32_t)ob * 128u + lane_off;
        TileIter<MODE> ti(it);
        for (int j = 0; j < it.ntiles; ++j) {
            const int base = ti.next(it);
            if (MODE == MODE_BLOCK) {
                if (row_valid) {
                    lo_r = max(base, p.kv_begin);
                    hi_r = min(base + BN - 1, p.kv_end - 1);
                    if (p.causal) hi_r = min(hi_r, qi_loc);
                } else {
                    lo_r = INT_MAX;
                    hi_r = INT_MIN;
                }
            }
            const int wlo = __reduce_min_sync(FULL, lo_r);
            const int whi = __reduce_max_sync(FULL, hi_r);
            const int sb = sc & 1;
            if (!mbar_wait(smem_u32(&b.s_full[sb]), (sc >> 1) & 1, ctx, &b.abort)) { ok = false; break; }
            tc_fence_after();
            uint32_t x[4][32];
            unsigned live = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int k0 = base + 32 * c;
                if (!(k0 + 31 < wlo || k0 > whi)) {
                    live |= 1u << c;
                    tmem_ld32(tmem + (uint32_t)sb * 128u + 32u * c + lane_off, x[c]);
                }
            }
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&b.s_empty[sb]));
            ++sc;
            // scale, mask, sink bias; tile maximum
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (!(live >> c & 1u)) continue;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int key = base + 32 * c + e;
                    float s = __uint_as_float(x[c][e]) * p.scale_l2;
                    if (key0 && key == 0) s += sink_l2;
                    s = (key >= lo_r && key <= hi_r) ? s : -INFINITY;
                    x[c][e] = __float_as_uint(s);
                    mt = fmaxf(mt, s);
                }
            }
            const bool upd = mt > m_run + TAU;
            float alpha = 1.0f;
            if (upd) {
                alpha = (m_run == -INFINITY) ? 0.0f : ex2(m_run - mt);
                l *= alpha;
                m_run = mt;
            }
            // P buffer free == previous P V finished (also makes O stable)
            if (pc >= 1 && !mbar_wait(smem_u32(&b.p_empty), (pc - 1) & 1, ctx, &b.abort)) {
                ok = false;
                break;
            }
            if (j >= 1 && __any_sync(FULL, upd)) {
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
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t region = p_base + (uint32_t)(c >> 1) * HALF;
                if (live >> c & 1u) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint32_t w[4];
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            const float a0 = ex2(__uint_as_float(x[c][8 * u + 2 * e2]) - mu);
                            const float a1 = ex2(__uint_as_float(x[c][8 * u + 2 * e2 + 1]) - mu);
                            l += a0 + a1;
                            w[e2] = pack_bf16x2(a0, a1);
                        }
                        const uint32_t addr = region + sw128_offset(r, (c & 1) * 4 + u);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                                     : "memory");
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t addr = region + sw128_offset(r, (c & 1) * 4 + u);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr),
                                     "r"(0u)
                                     : "memory");
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&b.p_full));
            ++pc;
        }
        if (!ok) break;
        // epilogue: O / l -> global, lse
        if (!mbar_wait(smem_u32(&b.o_full[ob]), (oc >> 1) & 1, ctx, &b.abort)) { ok = false; break; }
        tc_fence_after();
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
        const size_t orow = (size_t)(it.q_row0 + r) * p.H + it.h;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t ov[32];
            tmem_ld32(o_tmem + 32u * c, ov);
            tc_wait_ld();
            if (!row_valid) continue;
            if (MODE == MODE_WINDOW) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.o + orow * HD + 32 * c);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(ov[8 * u + 0]) * inv, __uint_as_float(ov[8 * u + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(ov[8 * u + 2]) * inv, __uint_as_float(ov[8 * u + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(ov[8 * u + 4]) * inv, __uint_as_float(ov[8 * u + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(ov[8 * u + 6]) * inv, __uint_as_float(ov[8 * u + 7]) * inv);
                    dst[u] = w;
                }
            } else {
                float4 *dst = reinterpret_cast<float4 *>(p.o_part + orow * HD + 32 * c);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    dst[u] = make_float4(__uint_as_float(ov[4 * u]) * inv, __uint_as_float(ov[4 * u + 1]) * inv,
                                         __uint_as_float(ov[4 * u + 2]) * inv, __uint_as_float(ov[4 * u + 3]) * inv);
            }
        }
        if (row_valid) {
            const float lse = l > 0.0f ? (m_run + log2f(l)) * LN2 : -INFINITY;
            if (MODE == MODE_WINDOW) {
                if (p.lse) p.lse[orow] = lse;
            } else {
                p.lse_part[orow] = lse;
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&b.o_empty[ob]));
        ++oc;
    }
}

template <int MODE>
__global__ void __launch_bounds__(NTHREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const TcParams p, const DevCtx ctx) {
    extern __shared__ uint8_t dsmem[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(dsmem) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
    __shared__ Bars b;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&b.q_full[i]), 1);
            mbar_init(smem_u32(&b.q_empty[i]), 1);
            mbar_init(smem_u32(&b.k_full[i]), 1);
            mbar_init(smem_u32(&b.k_empty[i]), 1);
            mbar_init(smem_u32(&b.v_full[i]), 1);
            mbar_init(smem_u32(&b.v_empty[i]), 1);
            mbar_init(smem_u32(&b.s_full[i]), 1);
            mbar_init(smem_u32(&b.s_empty[i]), 4);
            mbar_init(smem_u32(&b.o_full[i]), 1);
            mbar_init(smem_u32(&b.o_empty[i]), 4);
        }
        mbar_init(smem_u32(&b.p_full), 4);
        mbar_init(smem_u32(&b.p_empty), 1);
        mbar_init(smem_u32(&b.drain), 1);
        b.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&b.tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b.tmem_base;
    if (warp == 0) {
        if (lane == 0) producer<MODE>(p, &tq, &tk, &tv, sm, b, ctx);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) mma_issuer<MODE>(p, sm, b, tmem, ctx);
        __syncwarp();
    } else {
        softmax_role<MODE>(p, sm, b, tmem, ctx);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host side

CUresult make_map(CUtensorMap *m, const void *base, int rows, int heads) {
    const uint64_t dims[3] = {(uint64_t)HD, (uint64_t)heads, (uint64_t)rows};
    const uint64_t strides[2] = {(uint64_t)HD * 2, (uint64_t)HD * 2 * heads};
    const uint32_t box[3] = {64, 1, (uint32_t)BM};
    return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                             strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int MODE> cudaError_t launch(const TcParams &p, const void *q, int q_rows,
                                       const void *k, const void *v, int kv_rows,
                                       const DevInfo &dev, cudaStream_t s) {
    for (const void *ptr : {q, k, v})
        if (reinterpret_cast<uintptr_t>(ptr) & 15u) return cudaErrorMisalignedAddress;
    CUtensorMap tq, tk, tv;
    if (make_map(&tq, q, q_rows, p.H) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (make_map(&tk, k, kv_rows, p.Hkv) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (make_map(&tv, v, kv_rows, p.Hkv) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    const size_t smem = sizeof(Smem) + 1024;
    static bool attr_set[64] = {};
    if (!attr_set[dev.device & 63]) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set[dev.device & 63] = true;
    }
    const int grid = p.num_items < dev.sm_count ? p.num_items : dev.sm_count;
    DevCtx ctx{dev.err, wait_limit_ns()};
    attn_tc_kernel<MODE><<<grid, NTHREADS, smem, s>>>(tq, tk, tv, p, ctx);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_window_tc(const WindowArgs &a, const DevInfo &dev, cudaStream_t s) {
    TcParams p{};
    p.H = a.H;
    p.Hkv = a.Hkv;
    p.groups = a.H / a.Hkv;
    p.scale_l2 = a.scale * LOG2E;
    p.cu_seqlens = a.cu_seqlens;
    p.num_seqs = a.num_seqs;
    p.T = a.T;
    p.tiles_per_seq = (a.max_seqlen + BM - 1) / BM;
    p.wl = a.wl;
    p.wr = a.wr;
    p.causal = a.causal;
    p.sinks = a.sinks;
    p.sink_mode = a.sink_mode;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.lse = a.lse;
    const long long items = (long long)a.num_seqs * p.tiles_per_seq * a.H;
    if (items > INT_MAX) return cudaErrorInvalidValue;
    p.num_items = (int)items;
    if (reinterpret_cast<uintptr_t>(a.o) & 15u) return cudaErrorMisalignedAddress;
    return launch<MODE_WINDOW>(p, a.q, a.T, a.k, a.v, a.T, dev, s);
}

cudaError_t launch_block_tc(const BlockArgs &a, const DevInfo &dev, cudaStream_t s) {
    if (a.kv_end <= a.kv_begin) return launch_block_simt(a, dev, s);  // nothing to gather
    TcParams p{};
    p.H = a.H;
    p.Hkv = a.Hkv;
    p.groups = a.H / a.Hkv;
    p.scale_l2 = a.scale * LOG2E;
    p.mask = a.mask;
    p.M = a.M;
    p.Nctx = a.Nctx;
    p.q_pos0 = a.q_pos0;
    p.kv_begin = a.kv_begin;
    p.kv_end = a.kv_end;
    p.causal = a.causal;
    p.QB = (a.M + BM - 1) / BM;
    p.KB = (a.Nctx + BN - 1) / BN;
    p.o_part = a.o_part;
    p.lse_part = a.lse_part;
    const long long items = (long long)p.QB * a.H;
    if (items > INT_MAX) return cudaErrorInvalidValue;
    p.num_items = (int)items;
    if (reinterpret_cast<uintptr_t>(a.o_part) & 15u) return cudaErrorMisalignedAddress;
    return launch<MODE_BLOCK>(p, a.q, a.M, a.k, a.v, a.Nctx, dev, s);
}

}  // namespace sattn
