/*
 * sattn: index-gathered attention forward with sinks, for GB300 (sm_103a).
 *
 * C ABI of libsattn.so. Every tensor argument is a DEVICE pointer to a
 * contiguous, row-major buffer unless stated otherwise; scalars are passed by
 * value. The caller owns every buffer; the library allocates no device or
 * host memory. Its state: on the host, a per-device cache of attributes and
 * device addresses, the tensor-map encoder entry point, the debug flag and
 * wait limit, and a launch counter; on each device, module-scope arrays built
 * into the library: the error word, a ring of 256 item-claim counters and the
 * scratch array of sattn_sparse_fwd_static_scratch.
 *
 * Claim counters: each call of sattn_window_fwd, sattn_block_sparse_fwd and
 * sattn_block_sparse_chunks_fwd takes the next counter of the ring (zeroed
 * on its stream by an asynchronous memset) and its CTAs claim work items
 * from it. LIMIT: two such calls 256 calls apart in issue order use the same
 * counter and must not run at the same time on the GPU (different streams,
 * or CUDA graphs that captured them replayed concurrently); keep fewer than
 * 256 of these calls in flight at once. Calls on one stream never overlap.
 *
 * Execution: every compute call is asynchronous on `cuda_stream` (a
 * cudaStream_t; NULL selects the per-thread default stream, never the legacy
 * NULL stream). Calls do not synchronise unless debug mode is on.
 *
 * Errors: arguments are validated on the host before anything is launched and
 * rejected with SATTN_ERR_INVALID_ARG; nothing is written in that case. A
 * failed launch returns SATTN_ERR_CUDA. A device without sm_103 (or a
 * combination that has no kernel) returns SATTN_ERR_UNSUPPORTED. Kernels
 * never trap: an out-of-range index or a malformed cu_seqlens is skipped and
 * recorded in a device error word, and every wait inside a kernel gives up
 * after a bounded time and records a timeout. sattn_check_device() (or debug
 * mode) reports and clears that word. No C++ exception crosses this ABI.
 *
 * Empty work (zero tokens, zero queries or zero rows) returns SATTN_OK and
 * launches nothing.
 */
#ifndef SATTN_H_
#define SATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SATTN_OK = 0,
    SATTN_ERR_INVALID_ARG = 1,
    SATTN_ERR_UNSUPPORTED = 2,
    SATTN_ERR_CUDA = 3,
    SATTN_ERR_DEVICE_CHECK = 4, /* a kernel skipped an out-of-range index or sequence */
    SATTN_ERR_TIMEOUT = 5       /* a kernel-side wait gave up */
} sattn_status;

/* Sink semantics.
 *  KEY0_BIAS  sinks[h] is added to the logit of each sequence's first key
 *             (local position 0) wherever that key is visible; the softmax
 *             starts empty. ("PR #49815 report", Implementation item 2 and the
 *             `_fwd_kernel` listing: SINKS_BIAS_KEY0.) In the gathered path the
 *             bias goes to list entries equal to 0.
 *  NULL_LOGIT exp(sinks[h]) joins the softmax denominator only, never the
 *             numerator (same report, the USE_SINKS default; "DeepSeek-V4
 *             CSA/HCA walkthrough", section 4.4).
 * `sinks` is float32[H] on the device and must be non-NULL unless NONE. */
typedef enum {
    SATTN_SINK_NONE = 0,
    SATTN_SINK_KEY0_BIAS = 1,
    SATTN_SINK_NULL_LOGIT = 2
} sattn_sink_mode;

/* Element type of q/k/v/kv/o. Accumulation is always fp32. */
typedef enum { SATTN_F32 = 0, SATTN_BF16 = 1 } sattn_dtype;

/* Key-block size of the block-sparse mask. */
#define SATTN_BLOCK 128

/*
 * Sliding-window attention over packed varlen sequences
 * ("PR #49815 report", `_forward_window_attn` and `context_attention_fwd`
 * call: cu_seqlens, sliding_window_q/k = w, is_causal = False, per-head sinks).
 *
 *   q [T, H, d], k/v [T, Hkv, d], o [T, H, d]   (dtype), T = total_tokens
 *   lse [T, H] float32 natural-log denominator of each row, or NULL
 *   cu_seqlens int32 [num_seqs + 1] on the device, cu_seqlens[0] = 0,
 *     non-decreasing, cu_seqlens[num_seqs] = T
 *   max_seqlen >= every sequence length (used to size the grid)
 *
 * Query i sees key j iff both are in the same sequence and, with local
 * positions, -window_left <= j - i <= window_right (a negative bound means
 * unbounded on that side) and, if causal, j <= i. Query head h reads KV head
 * h / (H / Hkv). Logits are scale * <q, k> with scale > 0. o has q's dtype (round to
 * nearest even for bf16). With dtype BF16 and d = 128 the tcgen05 kernel
 * runs (the query heads of a KV group share its 128-row tiles: the largest
 * power of two dividing H / Hkv, at most 8, of them); other combinations run
 * the SIMT kernel.
 * Requirements: H % Hkv == 0, d in {64, 128}, num_seqs >= 0; with BF16 and
 * d = 128, q, k, v and o 16-byte aligned (SATTN_ERR_INVALID_ARG otherwise).
 */
sattn_status sattn_window_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                              const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                              int32_t max_seqlen, int32_t H, int32_t Hkv, int32_t d,
                              int32_t window_left, int32_t window_right, int32_t causal,
                              const float *sinks, sattn_sink_mode sink_mode, float scale,
                              sattn_dtype dtype, void *cuda_stream);

/*
 * Gathered attention over a [window ring | compressed] cache with one KV head
 * shared by all query heads ("DeepSeek-V4 CSA/HCA walkthrough", section 2.3
 * step 7 `sparse_attn(q, kv_cache, topk_idxs, attn_sink, scale)`, sections
 * 3.3 and 4.1-4.4).
 *
 *   q [B, M, H, d], kv_cache [B, N, d] (each row is both key and value),
 *   topk_idxs int32 [B, M, K] with entries in [-1, N); -1 is an invalid entry
 *     and contributes nothing; other entries count with multiplicity.
 *   o [B, M, H, d] (dtype), lse [B, M, H] float32 or NULL.
 *   workspace: NULL or a caller-owned device buffer of at least
 *     sattn_sparse_workspace_bytes(B, M, H, d, K) bytes, 256-byte aligned.
 * Execution (bf16, H == 32, d == 128): with at most as many queries (B M) as
 *   the device has SMs, and lists short enough for eight CTAs of 384 entries,
 *   each query's list is cut into segments handled by the CTAs of one
 *   thread-block cluster, whose partials merge through their LSE in shared
 *   memory, in one launch; the workspace is not used. Otherwise a persistent
 *   kernel runs: with a workspace it may split each list across CTAs and
 *   merge the partial results in a second launch; without one each query's
 *   list is processed by a single CTA. Every path gives the same result up to
 *   floating-point summation order. F32 (and bf16 with other H) runs one warp
 *   per query row and uses no workspace.
 * Requirements: d == 128 for BF16 (d in {64, 128} for F32), N >= 1, K >= 0;
 * with BF16, q, kv_cache and o 16-byte aligned (SATTN_ERR_INVALID_ARG
 * otherwise).
 */
sattn_status sattn_sparse_fwd(const void *q, const void *kv_cache, const int32_t *topk_idxs,
                              const float *sinks, sattn_sink_mode sink_mode, float scale, void *o,
                              float *lse, int32_t B, int32_t M, int32_t H, int32_t d, int32_t N,
                              int32_t K, void *workspace, size_t workspace_bytes,
                              sattn_dtype dtype, void *cuda_stream);

/* Workspace size (bytes) that lets sattn_sparse_fwd's persistent kernel split
 * each index list (an upper bound for any GPU of at most 256 SMs); calls that
 * take the cluster path ignore the workspace. 0 when no split is possible. */
size_t sattn_sparse_workspace_bytes(int32_t B, int32_t M, int32_t H, int32_t d, int32_t K);

/* Size in bytes of the scratch array built into the library for
 * sattn_sparse_fwd_static_scratch. */
#define SATTN_SPARSE_STATIC_SCRATCH_BYTES (8u << 20)

/*
 * sattn_sparse_fwd for callers that cannot allocate device memory. (The pages
 * have no counterpart to this call; it exists for such callers: a plug-in
 * whose host application owns all device memory, a loop whose policy forbids
 * cudaMalloc/cudaFree after start-up, or C code given only tensor pointers
 * and a stream.)
 *
 * Same arguments and results as sattn_sparse_fwd without the workspace: the
 * partial results of a split index list go to a fixed array of
 * SATTN_SPARSE_STATIC_SCRATCH_BYTES compiled into the library, which every GPU
 * that loads the library holds until the process exits. Nothing is allocated.
 * Only bf16 calls with H = 32 and d = 128 can split lists and use the array;
 * such a call whose sattn_sparse_workspace_bytes(B, M, H, d, K) exceeds its
 * size is rejected with SATTN_ERR_INVALID_ARG before anything runs. Other
 * shapes never need it and are not limited by it.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture. All calls share the array and it keeps the last call's contents
 * (nothing in it needs to start at zero); calls whose work overlaps on the GPU
 * race on it, so issue them on one stream.
 */
sattn_status sattn_sparse_fwd_static_scratch(const void *q, const void *kv_cache,
                                             const int32_t *topk_idxs, const float *sinks,
                                             sattn_sink_mode sink_mode, float scale, void *o,
                                             float *lse, int32_t B, int32_t M, int32_t H,
                                             int32_t d, int32_t N, int32_t K, sattn_dtype dtype,
                                             void *cuda_stream);

/*
 * Merge of chunk partials through their log-sum-exp ("XAttention Offload
 * Stream Synchronization Fix", technical details: partial (m_i, l_i) stats per
 * KV chunk, merged into (m_global, l_global), outputs normalised with them).
 *
 *   o_parts float32 [C, R, d] (each normalised within its chunk),
 *   lse_parts float32 [C, R] (-inf for a chunk in which the row saw nothing)
 *   sinks float32 [H] or NULL: a null-logit term exp(sinks[r % H]) is added
 *     to the merged denominator exactly once.
 *   o [R, d] (dtype), lse [R] float32 or NULL.
 *   lse = ln(sum_c exp(lse_c) [+ exp(sink)]),  o = sum_c exp(lse_c - lse) o_c.
 * A row with every lse_c = -inf and no sink gives o = 0, lse = -inf.
 */
sattn_status sattn_merge_lse(const float *o_parts, const float *lse_parts, int32_t C, int64_t R,
                             int32_t d, int32_t H, const float *sinks, void *o, float *lse,
                             sattn_dtype dtype, void *cuda_stream);

/*
 * One KV chunk of block-sparse causal attention (same nano-vllm page: chunked
 * KV with per-chunk partial stats; test results give ~10% block density).
 *
 *   q [M, H, d] at absolute positions q_pos0 .. q_pos0 + M - 1,
 *   k/v [Nctx, Hkv, d],
 *   block_mask uint8 [H, ceil(M/128), ceil(Nctx/128)]: entry [h][i/128][j/128]
 *     != 0 lets query i of head h see key j (query blocks local, key blocks
 *     absolute);
 *   only keys in [kv_begin, kv_end) are used; with causal, key j needs
 *     j <= q_pos0 + i.
 *   o_part float32 [M, H, d] normalised within the chunk, lse_part float32
 *   [M, H] (-inf where the row sees nothing in the chunk; o_part is then 0).
 * Merge the chunks with sattn_merge_lse (C = number of chunks, R = M * H).
 * Requirements: H % Hkv == 0, dtype BF16 with d == 128 or F32 with d in {64, 128},
 *   0 <= kv_begin <= kv_end <= Nctx.
 */
sattn_status sattn_block_sparse_fwd(const void *q, const void *k, const void *v,
                                    const uint8_t *block_mask, int32_t M, int32_t Nctx, int32_t H,
                                    int32_t Hkv, int32_t d, int32_t q_pos0, int32_t kv_begin,
                                    int32_t kv_end, int32_t causal, float scale, float *o_part,
                                    float *lse_part, sattn_dtype dtype, void *cuda_stream);

/*
 * All chunks of a block-sparse call at once: [kv_begin, kv_end) is cut into
 * C = ceil((kv_end - kv_begin) / chunk) chunks [kv_begin + c chunk,
 * min(kv_end, kv_begin + (c + 1) chunk)), and chunk c writes o_parts[c]
 * (float32 [C, M, H, d]) and lse_parts[c] ([C, M, H]) exactly as
 * sattn_block_sparse_fwd called on that chunk would, bit for bit. With BF16
 * this is one launch over every (chunk, query block, head); F32 runs one
 * launch per chunk. Merge with sattn_merge_lse (C, R = M * H).
 * Requirements: those of sattn_block_sparse_fwd, and chunk > 0
 * (SATTN_ERR_INVALID_ARG otherwise). M == 0 or kv_begin == kv_end: nothing
 * to do.
 */
sattn_status sattn_block_sparse_chunks_fwd(const void *q, const void *k, const void *v,
                                           const uint8_t *block_mask, int32_t M, int32_t Nctx,
                                           int32_t H, int32_t Hkv, int32_t d, int32_t q_pos0,
                                           int32_t kv_begin, int32_t kv_end, int32_t chunk,
                                           int32_t causal, float scale, float *o_parts,
                                           float *lse_parts, sattn_dtype dtype,
                                           void *cuda_stream);

/*
 * Index lists over a [window ring | compressed] cache ("DeepSeek-V4 CSA/HCA
 * walkthrough", section 2.3 steps 5-6: the window indices concatenated with
 * the compressed-region indices form topk_idxs; section 3.3: cache layout
 * [window_size + max_seq_len / ratio rows], ring row = position mod window).
 *
 *   topk_idxs int32 [B, M, K] (device, written), start_pos int32 [B] (device):
 *   query m of request b sits at absolute position p = start_pos[b] + m and
 *   lists, in order:
 *     - win window entries: slot k holds token t = p - win + 1 + k at its
 *       ring row t mod win, or -1 when t < 0;
 *     - the compressed rows visible at p, c = 0 .. floor(p / ratio), as cache
 *       rows win + c in ascending order; when more are visible than the
 *       K - win entries left, the most recent ones (the pages select these
 *       with a learned indexer, which is not part of this library);
 *     - -1 in the entries left over. ratio = 0: no compressed part.
 * Requirements: B, M, K >= 0, win >= 1, ratio >= 0; positions
 * start_pos[b] + m in [0, 2^31 - 2] (a query outside that range keeps a list
 * of -1 and is reported by sattn_check_device as a device check failure).
 */
sattn_status sattn_build_topk_idxs(int32_t *topk_idxs, const int32_t *start_pos, int32_t B,
                                   int32_t M, int32_t K, int32_t win, int32_t ratio,
                                   void *cuda_stream);

/*
 * Ring write of new KV rows into the window part of the cache (section 3.3:
 * the last window_size new rows are stored from row start_pos mod window on,
 * wrapping to row 0; older rows are overwritten).
 *
 *   kv_cache [B, N, d] (dtype, device, updated), kv_new [B, S, d] (dtype,
 *   device), start_pos int32 [B] (device): the S new rows of request b have
 *   positions start_pos[b] .. start_pos[b] + S - 1; the last min(S, win) of
 *   them are stored at rows (position mod win). Rows win .. N-1 (the
 *   compressed region) are not touched.
 * Requirements: N >= win >= 1, S >= 0, d * element size a multiple of 16 and
 * kv_cache, kv_new 16-byte aligned; start_pos[b] >= 0 (a negative entry
 * writes nothing for that request and is reported by sattn_check_device).
 */
sattn_status sattn_kv_ring_write(void *kv_cache, const void *kv_new, const int32_t *start_pos,
                                 int32_t B, int32_t S, int32_t N, int32_t d, int32_t win,
                                 sattn_dtype dtype, void *cuda_stream);

/*
 * FP8 KV cache (DeepSeek-V4 CSA/HCA walkthrough, section 2.3 step 4 and section
 * 5.3: the non-RoPE part of each KV row is quantised to FP8, the RoPE part keeps
 * a wider type; the pages leave the format open). Layout used here, per row of
 * d columns whose last rd are the RoPE part:
 *   kv_nope uint8 [rows, d - rd]: OCP e4m3 codes of x / scale, round to nearest
 *     even, saturating at +-448;
 *   kv_scale float32 [rows]: amax of the row's first d - rd values / 448 (1 when
 *     they are all zero); value = e4m3(code) * scale;
 *   kv_rope bf16 [rows, rd]: the last rd values, round to nearest even.
 *
 * sattn_quantize_kv_fp8 writes that layout from rows kv [rows, d] (dtype,
 * device); scale and codes are computed in fp32 with IEEE division.
 * Requirements: d and rd multiples of 4 with 0 <= rd <= d; all pointers 16-byte
 * aligned (SATTN_ERR_INVALID_ARG otherwise). Caller-owned buffers.
 */
sattn_status sattn_quantize_kv_fp8(const void *kv, uint8_t *kv_nope, void *kv_rope,
                                   float *kv_scale, int64_t rows, int32_t d, int32_t rd,
                                   sattn_dtype dtype, void *cuda_stream);

/*
 * sattn_sparse_fwd over an FP8 cache: the same operation, arguments and
 * results (q, o bf16), the KV rows of request b being the dequantised rows
 * b * N .. b * N + N - 1 of the layout above (kv_nope [B, N, d - rd],
 * kv_scale [B, N], kv_rope [B, N, rd]). The gathered rows are dequantised to
 * bf16 in shared memory (e4m3 value * scale, rounded to nearest even), so a
 * gathered row costs d - rd + 2 rd + 4 bytes instead of 2 d.
 * Supported: H = 32, d = 128, rd = 64 (SATTN_ERR_UNSUPPORTED otherwise);
 * q, kv_nope, kv_rope and o 16-byte aligned. Execution and workspace as for
 * sattn_sparse_fwd with bf16 (few queries: the cluster path, no workspace;
 * otherwise the persistent kernel, split through the workspace if given).
 */
sattn_status sattn_sparse_fp8_fwd(const void *q, const uint8_t *kv_nope, const void *kv_rope,
                                  const float *kv_scale, const int32_t *topk_idxs,
                                  const float *sinks, sattn_sink_mode sink_mode, float scale,
                                  void *o, float *lse, int32_t B, int32_t M, int32_t H, int32_t d,
                                  int32_t rd, int32_t N, int32_t K, void *workspace,
                                  size_t workspace_bytes, void *cuda_stream);

/*
 * XAttention block selection (XAttention Offload Stream Synchronization Fix,
 * technical details: three-stage KV chunking, then the block selection step).
 * It produces the block mask that sattn_block_sparse_fwd consumes. The
 * estimate is the exact softmax at full resolution (the pages describe no
 * cheaper one). Query rows i = 0 .. M-1 sit at positions q_pos0 + i; key j is
 * visible to row i iff kv_begin <= j < kv_end and (causal == 0 or
 * j <= q_pos0 + i). Scores s_ij = scale <q[i, h], k[j, h / (H / Hkv)]>.
 * Blocks are 128 x 128: query block qb = i / 128 (local), key block
 * kb = j / 128 (absolute); QB = ceil(M / 128), KB = ceil(Nctx / 128).
 *   q bf16 [M, H, d], k bf16 [Nctx, Hkv, d] (device, 16-byte aligned).
 * A chunk [kv_begin, kv_end) must start on a block boundary and end on one or
 * at Nctx (SATTN_ERR_INVALID_ARG otherwise); H <= 65535. Supported: d = 128
 * (SATTN_ERR_UNSUPPORTED otherwise); scale > 0.
 *
 * Stage 1, sattn_xattn_partial_stats: m[i, h] = max of the visible scores of
 *   the chunk and l[i, h] = sum of exp(s_ij - m) (m = -inf, l = 0 when the row
 *   sees no key of the chunk); m, l float32 [M, H].
 * Stage 2, sattn_xattn_merge_stats: m_parts, l_parts float32 [C, R] (R rows,
 *   e.g. M * H) -> m = max_c m_c, l = sum_c l_c exp(m_c - m).
 * Stage 3, sattn_xattn_block_sum: with the merged (m, l), block_sum[h, qb, kb]
 *   = sum over rows i of qb and visible keys j of kb of exp(s_ij - m_i) / l_i,
 *   written for the chunk's key blocks kb = kv_begin/128 .. ceil(kv_end/128)-1
 *   (zero for those no row of qb sees); other entries are not touched.
 *   block_sum float32 [H, QB, KB].
 * Step 4, sattn_xattn_find_blocks: for each (h, qb) the key blocks ordered by
 *   block_sum (largest first, the lower kb first among equal values; negative
 *   and NaN values count as 0) and the shortest leading run whose cumulative sum
 *   (float64, in that order) reaches threshold x their total is selected:
 *   mask[h, qb, kb] = 1 (uint8 [H, QB, KB]), others 0; nothing where the total
 *   is 0. Requirements: 0 <= threshold <= 1, KB <= 4096.
 * All buffers are caller-owned; every call is asynchronous on cuda_stream.
 */
sattn_status sattn_xattn_partial_stats(const void *q, const void *k, int32_t M, int32_t Nctx,
                                       int32_t H, int32_t Hkv, int32_t d, int32_t q_pos0,
                                       int32_t kv_begin, int32_t kv_end, int32_t causal,
                                       float scale, float *m, float *l, void *cuda_stream);
sattn_status sattn_xattn_merge_stats(const float *m_parts, const float *l_parts, int32_t C,
                                     int64_t R, float *m, float *l, void *cuda_stream);
sattn_status sattn_xattn_block_sum(const void *q, const void *k, const float *m, const float *l,
                                   int32_t M, int32_t Nctx, int32_t H, int32_t Hkv, int32_t d,
                                   int32_t q_pos0, int32_t kv_begin, int32_t kv_end,
                                   int32_t causal, float scale, float *block_sum,
                                   void *cuda_stream);
sattn_status sattn_xattn_find_blocks(const float *block_sum, int32_t H, int32_t QB, int32_t KB,
                                     float threshold, uint8_t *mask, void *cuda_stream);

/*
 * The four steps in one call over the whole key range [0, Nctx): stage 1 for
 * the C = ceil(Nctx / chunk) chunks [c chunk, min(Nctx, (c + 1) chunk)) in
 * one launch, stage 2 over those C partial stats, stage 3 over [0, Nctx),
 * step 4. The results are those of the four calls above made chunk by chunk,
 * bit for bit. Four kernel launches in all.
 *   chunk: a positive multiple of 128 with C <= 65535 (SATTN_ERR_INVALID_ARG
 *     otherwise); KB <= 4096.
 *   workspace: a caller-owned device buffer of at least
 *     sattn_xattn_select_workspace_bytes(M, H, Nctx, chunk) bytes, 16-byte
 *     aligned; it receives the per-chunk stats and the merged stats (float32
 *     [2 C + 2, M, H]) and is free again when the call's work has run.
 *   block_sum float32 [H, QB, KB] and mask uint8 [H, QB, KB]: every entry is
 *     written.
 * M == 0 or Nctx == 0: nothing to do (SATTN_OK).
 */
size_t sattn_xattn_select_workspace_bytes(int32_t M, int32_t H, int32_t Nctx, int32_t chunk);
sattn_status sattn_xattn_select_blocks(const void *q, const void *k, int32_t M, int32_t Nctx,
                                       int32_t H, int32_t Hkv, int32_t d, int32_t q_pos0,
                                       int32_t causal, float scale, int32_t chunk,
                                       float threshold, void *workspace, size_t workspace_bytes,
                                       float *block_sum, uint8_t *mask, void *cuda_stream);

/*
 * Compressor gated pooling (DeepSeek-V4 CSA/HCA walkthrough, sections 5.1 and
 * 5.2): every `ratio` consecutive tokens of a sequence become one compressed
 * KV row, the softmax-weighted sum of their kv projections.
 *
 *   kv, score [B, S, coff * d] (in_dtype, device, row-major): the tokens' kv
 *   and gate projections, coff = 2 when `overlap` is 1, else 1.
 *   ape float32 [ratio, coff * d] (device): the absolute position term.
 *   out (out_dtype, device, written): row w of sequence b, w = 0 .. S/ratio - 1,
 *   at out + b * out_batch_stride + w * d elements; e.g. the compressed region
 *   of a [window | compressed] cache with out_batch_stride = N * d.
 * For window w and column j (0 <= j < d) the entries are the window's tokens
 *   t = w * ratio + i, i < ratio, with value kv[t, c] and score score[t, c] +
 *   ape[i, c] where c = (coff - 1) * d + j; with overlap also the previous
 *   window's tokens t' = (w - 1) * ratio + i with kv[t', j] and score[t', j] +
 *   ape[i, j] (window 0 has no previous window). out[w, j] = sum over the
 *   entries of value * softmax(scores). The S % ratio tail tokens produce no
 *   row: a decode step passes the tokens of the current and previous window.
 * Computed in fp32; out rounded to nearest even for BF16.
 * Requirements: B, S >= 0; ratio >= 1; overlap 0 or 1; d a multiple of 4;
 *   out_batch_stride >= (S / ratio) * d and a multiple of 4; kv, score, ape and
 *   out 16-byte aligned; otherwise SATTN_ERR_INVALID_ARG before anything runs.
 *   The caller owns every buffer; nothing is allocated.
 */
sattn_status sattn_compress_kv(const void *kv, const void *score, const float *ape, void *out,
                               int64_t out_batch_stride, int32_t B, int32_t S, int32_t d,
                               int32_t ratio, int32_t overlap, sattn_dtype in_dtype,
                               sattn_dtype out_dtype, void *cuda_stream);

/* Human-readable name of a status code (static storage). */
const char *sattn_status_str(sattn_status s);

/* Debug mode: every compute call synchronises its stream and reports the
 * device error word (SATTN_ERR_DEVICE_CHECK / SATTN_ERR_TIMEOUT). */
void sattn_set_debug(int on);

/* Synchronise `cuda_stream`, then read and clear the device error word of the
 * current device. Returns SATTN_OK, SATTN_ERR_DEVICE_CHECK, SATTN_ERR_TIMEOUT
 * or SATTN_ERR_CUDA. */
sattn_status sattn_check_device(void *cuda_stream);

/* Upper bound, in nanoseconds, on any single wait inside a kernel (default
 * one second). A value of 0 restores the default. */
void sattn_set_wait_limit_ns(uint64_t ns);

/* Test hook for the failure path of the tensor-core kernels (window,
 * block-sparse, gathered, gathered FP8, block-selection stats and sums). With
 * `on` nonzero, launches made afterwards start with their MMA-issuing thread
 * waiting for a barrier phase that nothing completes: that wait runs out
 * after the wait limit, the kernel records SATTN_ERR_TIMEOUT in the device
 * error word, stops every role of the CTA, lets its own copies and MMAs in
 * flight finish (bounded) and frees its tensor memory. The outputs of such a
 * launch are undefined; nothing faults, traps or hangs. 0 (the default) turns
 * the hook off. Keep the wait limit short while it is on (a few
 * milliseconds: every launch then takes about that long). */
void sattn_set_test_wait_stall(int on);

/* Library ABI version (major * 100 + minor). */
int32_t sattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SATTN_H_ */
