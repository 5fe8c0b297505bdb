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
// Both accumulators live in TMEM (H = 32 columns each). The softmax runs per
// head over the rows: S^T is transposed through shared memory so that four
// threads own one head and reduce with two shuffles.
//
// One CTA handles one (query, split) item: the item's slice of the index
// list is walked in tiles of 128 entries; gathers are 16-byte cp.async with
// zero fill for invalid entries, double-buffered against the MMAs. With more
// than one split the normalised partial output and its lse go to the
// workspace and are merged through their log-sum-exp (sinks added once).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace sattn {
namespace {

constexpr int R = 128;       // gathered rows per tile
constexpr int HD = 128;      // head dim
constexpr int NH = 32;       // query heads handled by the kernel
constexpr int NSLOT = 2;           // independent items in flight per CTA
constexpr int SLOT_THREADS = 128;
constexpr int NTHREADS = NSLOT * SLOT_THREADS;
constexpr uint32_t SLOT_COLS = 64;  // TMEM per slot: S^T (32) + O^T (32)
constexpr uint32_t TMEM_COLS = SLOT_COLS * NSLOT;
constexpr uint32_t KV_TILE = R * HD * 2;   // 32 KB
constexpr uint32_t KV_HALF = KV_TILE / 2;  // 64 columns of d
constexpr uint32_t QP_HALF = NH * 128;     // 4 KB: one 64-column half of Q or P
constexpr int SB_STRIDE = 132;             // floats per head row in the transpose buffer
constexpr float TAU = 8.0f;
constexpr int MAX_SPLITS = 64;

// Shared memory of one slot (four warps working on one item at a time).
struct SlotSmem {
    uint8_t kv[2][KV_TILE];
    uint8_t q[2 * QP_HALF];
    uint8_t p[2 * QP_HALF];
    float sbuf[NH * SB_STRIDE];
    int idx[2][R];
    float alpha[NH];
    float m[NH];
    float l[NH];
    uint8_t pad[1024 - (NH * SB_STRIDE * 4 + 2 * R * 4 + 3 * NH * 4) % 1024];
};
static_assert(sizeof(SlotSmem) % 1024 == 0, "slot tiles must stay 1024-byte aligned");

struct Smem {
    SlotSmem slot[NSLOT];
    uint64_t s_bar[NSLOT], pv_bar[NSLOT], drain_bar[NSLOT];
    uint32_t tmem_base;
    int abort;
};

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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Gather the rows listed in idx_s (128 entries, -1 = zero row) into one
// 128B-swizzled K-major tile. 16 lanes copy one 256-byte row.
__device__ __forceinline__ void gather_tile(uint32_t dst, const __nv_bfloat16 *kvb,
                                            const int *idx_s, int tid) {
    const int unit = tid & 15;  // 16-byte unit of the row (0..15)
    const uint32_t half = (uint32_t)(unit >> 3) * KV_HALF;
#pragma unroll 4
    for (int rr = tid >> 4; rr < R; rr += SLOT_THREADS / 16) {
        const int e = idx_s[rr];
        const __nv_bfloat16 *src = kvb + (size_t)(e >= 0 ? e : 0) * HD + unit * 8;
        cp_async16(dst + half + sw128_offset(rr, unit & 7), src, e >= 0 ? 16u : 0u);
    }
}

// Per-slot barrier among the slot's 128 threads (named barrier 1 + slot).
__device__ __forceinline__ void slot_sync(int slot) {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + slot), "r"(SLOT_THREADS) : "memory");
}
// Per-slot barrier that also returns whether any thread's predicate was true.
__device__ __forceinline__ int slot_sync_or(int slot, int pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.s32 p, %2, 0;\n\t"
        "bar.red.or.pred q, %1, %3, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(1 + slot), "r"(pred), "r"(SLOT_THREADS)
        : "memory");
    return r;
}

__global__ void __launch_bounds__(NTHREADS, 1)
sparse_tc_kernel(const SpParams p, const DevCtx ctx) {
    extern __shared__ __align__(1024) uint8_t dsmem[];
    Smem &all = *reinterpret_cast<Smem *>(dsmem);
    const int slot = threadIdx.x / SLOT_THREADS;
    const int tid = threadIdx.x % SLOT_THREADS, warp = tid >> 5;
    SlotSmem &sm = all.slot[slot];
    if (smem_u32(dsmem) & 1023u) {  // the 128B swizzle needs an aligned base
        if (threadIdx.x == 0) record_error(ctx, DEVERR_LAYOUT);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(smem_u32(&all.s_bar[s]), 1);
            mbar_init(smem_u32(&all.pv_bar[s]), 1);
            mbar_init(smem_u32(&all.drain_bar[s]), 1);
        }
        all.abort = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(smem_u32(&all.tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t t_s = all.tmem_base + (uint32_t)slot * SLOT_COLS, t_o = t_s + 32u;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t s_bar = smem_u32(&all.s_bar[slot]), pv_bar = smem_u32(&all.pv_bar[slot]);
    volatile int *abort = &all.abort;
    // per-head state is owned by the 4 threads of head h = tid / 4
    const int h = tid >> 2, part = tid & 3;
    const bool key0 = p.sink_mode == 1;
    const float sink_h = p.sinks ? __ldg(p.sinks + h) * LOG2E : 0.0f;
    const int nitems = p.B * p.M * p.splits;
    int s_phase = 0, pv_phase = 0;
    bool ok = true, bad_index = false;

    for (int item = blockIdx.x * NSLOT + slot; ok && item < nitems; item += gridDim.x * NSLOT) {
        const int bm = item / p.splits, split = item % p.splits;
        const int b = bm / p.M;
        const int e_begin = split * p.split_len;
        const int e_end = min(p.K, e_begin + p.split_len);
        const int ntiles = e_end > e_begin ? (e_end - e_begin + R - 1) / R : 0;
        const __nv_bfloat16 *kvb = p.kv + (size_t)b * p.N * HD;
        const int32_t *list = p.idx + (size_t)bm * p.K;
        // Q rows (32 heads x 256 B) -> K-major swizzled B operand
        {
            const __nv_bfloat16 *qb = p.q + (size_t)bm * NH * HD;
            const uint32_t qs = smem_u32(sm.q);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int u = tid + i * SLOT_THREADS;  // 512 units of 16 B
                const int hh = u >> 4, unit = u & 15;
                cp_async16(qs + (uint32_t)(unit >> 3) * QP_HALF + sw128_offset(hh, unit & 7),
                           qb + hh * HD + unit * 8, 16u);
            }
        }
        auto load_idx = [&](int t) -> int {
            const int e = e_begin + t * R + tid;
            int v = e < e_end ? __ldg(list + e) : -1;
            if (v < -1 || v >= p.N) {
                bad_index = true;
                v = -1;
            }
            return v;
        };
        const bool null_sink = p.sink_mode == 2 && p.splits == 1;
        float m_run = null_sink ? sink_h : -INFINITY;
        float l_run = null_sink ? 1.0f : 0.0f;
        int stage = 0;
        bool o_written = false;
        // prologue: tile 0 gather (the previous item left both stages free)
        int cur_any = 0;
        if (ntiles > 0) {
            const int v0 = load_idx(0);
            sm.idx[0][tid] = v0;
            cur_any = slot_sync_or(slot, v0 >= 0);
            if (cur_any) gather_tile(smem_u32(sm.kv[0]), kvb, sm.idx[0], tid);
        }
        cp_async_commit();
        for (int t = 0; t < ntiles && ok; ++t) {
            // stage the next tile's gather while this one is consumed
            int nxt_any = 0;
            if (t + 1 < ntiles) {
                const int nv = load_idx(t + 1);
                sm.idx[stage ^ 1][tid] = nv;
                nxt_any = slot_sync_or(slot, nv >= 0);
                if (nxt_any) gather_tile(smem_u32(sm.kv[stage ^ 1]), kvb, sm.idx[stage ^ 1], tid);
            }
            cp_async_commit();
            if (!cur_any) {  // all entries of this tile are -1: nothing to do
                stage ^= 1;
                cur_any = nxt_any;
                continue;
            }
            cp_async_wait<1>();
            fence_proxy_async_smem();
            slot_sync(slot);
            const uint32_t kv_s = smem_u32(sm.kv[stage]);
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    tc_mma_f16(t_s, desc_k(kv_s, kk, KV_HALF), desc_k(smem_u32(sm.q), kk, QP_HALF),
                               IDESC_S, kk > 0 ? 1u : 0u);
                tc_commit(s_bar);
            }
            __syncwarp();
            if (!mbar_wait(s_bar, s_phase, ctx, abort)) { ok = false; break; }
            s_phase ^= 1;
            tc_fence_after();
            // S^T row (this thread's gathered row) for all 32 heads -> transpose buffer
            {
                uint32_t sv[32];
                tmem_ld32(t_s + lane_off, sv);
                tc_wait_ld();
                const int row = tid, prt = row >> 5, i = row & 31;
#pragma unroll
                for (int hh = 0; hh < NH; ++hh)
                    sm.sbuf[hh * SB_STRIDE + prt * 33 + i] = __uint_as_float(sv[hh]);
            }
            tc_fence_before();
            slot_sync(slot);
            // softmax for head h over rows part*32 .. part*32+31
            float x[32];
            float mt = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int row = part * 32 + i;
                const int e = sm.idx[stage][row];
                float sc = sm.sbuf[h * SB_STRIDE + part * 33 + i] * p.scale_l2;
                if (key0 && e == 0) sc += sink_h;
                sc = e >= 0 ? sc : -INFINITY;
                x[i] = sc;
                mt = fmaxf(mt, sc);
            }
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
            const bool upd = mt > m_run + TAU;
            float alpha = 1.0f;
            if (upd) {
                alpha = (m_run == -INFINITY) ? 0.0f : ex2(m_run - mt);
                l_run *= alpha;
                m_run = mt;
            }
            const float mu = m_run == -INFINITY ? 0.0f : m_run;
            float ls = 0.0f;
            const uint32_t pbase = smem_u32(sm.p) + (uint32_t)(part >> 1) * QP_HALF;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint32_t w[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const float a0 = ex2(x[8 * u + 2 * e2] - mu);
                    const float a1 = ex2(x[8 * u + 2 * e2 + 1] - mu);
                    ls += a0 + a1;
                    w[e2] = pack_bf16x2(a0, a1);
                }
                const uint32_t addr = pbase + sw128_offset(h, (part & 1) * 4 + u);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]),
                             "r"(w[1]), "r"(w[2]), "r"(w[3])
                             : "memory");
            }
            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
            l_run += ls;
            if (part == 0) sm.alpha[h] = alpha;
            const int any_upd = slot_sync_or(slot, upd && o_written);
            if (any_upd) {  // rescale O^T columns (heads) whose max moved
                tc_fence_after();
                uint32_t ov[32];
                tmem_ld32(t_o + lane_off, ov);
                tc_wait_ld();
#pragma unroll
                for (int hh = 0; hh < NH; ++hh)
                    ov[hh] = __float_as_uint(__uint_as_float(ov[hh]) * sm.alpha[hh]);
                tmem_st32(t_o + lane_off, ov);
                tc_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            slot_sync(slot);
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < R / 16; ++kk)
                    tc_mma_f16(t_o, desc_mn(kv_s, kk), desc_k(smem_u32(sm.p), kk, QP_HALF),
                               IDESC_O, (o_written || kk > 0) ? 1u : 0u);
                tc_commit(pv_bar);
            }
            __syncwarp();
            o_written = true;
            // the tile's buffers (KV stage, P) are reused only after this MMA finishes
            if (!mbar_wait(pv_bar, pv_phase, ctx, abort)) { ok = false; break; }
            pv_phase ^= 1;
            tc_fence_after();
            stage ^= 1;
            cur_any = nxt_any;
        }
        cp_async_wait<0>();
        if (!ok) break;
        // epilogue
        if (part == 0) {
            sm.m[h] = m_run;
            sm.l[h] = l_run;
        }
        slot_sync(slot);
        uint32_t ov[32];
        if (o_written) {
            tmem_ld32(t_o + lane_off, ov);
            tc_wait_ld();
        } else {
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) ov[hh] = 0u;
        }
        const int d = tid;  // TMEM lane of O^T == head-dim index
        if (p.splits == 1) {
            __nv_bfloat16 *ob = p.o + (size_t)bm * NH * HD;
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const float l = sm.l[hh];
                ob[hh * HD + d] = __float2bfloat16_rn(l > 0.f ? __uint_as_float(ov[hh]) / l : 0.f);
            }
            if (p.lse && tid < NH) {
                const float l = sm.l[tid];
                p.lse[(size_t)bm * NH + tid] = l > 0.f ? (sm.m[tid] + log2f(l)) * LN2 : -INFINITY;
            }
        } else {
            const size_t rows = (size_t)p.B * p.M * NH;
            float *op = p.o_part + ((size_t)split * rows + (size_t)bm * NH) * HD;
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const float l = sm.l[hh];
                op[hh * HD + d] = l > 0.f ? __uint_as_float(ov[hh]) / l : 0.f;
            }
            if (tid < NH) {
                const float l = sm.l[tid];
                p.lse_part[(size_t)split * rows + (size_t)bm * NH + tid] =
                    l > 0.f ? (sm.m[tid] + log2f(l)) * LN2 : -INFINITY;
            }
        }
        tc_fence_before();
        slot_sync(slot);  // m/l and O^T of this item are consumed before the next reuses them
    }
    cp_async_wait<0>();
    if (bad_index) record_error(ctx, DEVERR_INDEX);
    if (!ok && tid == 0) {  // let any MMA still in flight finish before TMEM is released
        tc_commit(smem_u32(&all.drain_bar[slot]));
        int zero = 0;
        mbar_wait(smem_u32(&all.drain_bar[slot]), 0, ctx, &zero);
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
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
    const long long want = (nitems + NSLOT - 1) / NSLOT;
    const int grid = (int)(want < dev.sm_count ? want : dev.sm_count);
    const size_t smem = sizeof(Smem);
    static bool attr_set[64] = {};
    if (!attr_set[dev.device & 63]) {
        cudaError_t e = cudaFuncSetAttribute(sparse_tc_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        // Ask for the largest shared-memory carveout so that co-resident CTAs fit.
        e = cudaFuncSetAttribute(sparse_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        attr_set[dev.device & 63] = true;
    }
    DevCtx ctx{dev.err, wait_limit_ns()};
    sparse_tc_kernel<<<grid, NTHREADS, smem, s>>>(p, ctx);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || splits == 1) return e;
    MergeArgs m{p.o_part, p.lse_part, splits, (int64_t)rows, a.d, a.H,
                a.sink_mode == 2 ? a.sinks : nullptr, a.o, a.lse, a.dtype};
    return launch_merge(m, dev, s);
}

}  // namespace sattn
