"""fp64 CPU oracle for index-gathered attention with sinks.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers. The library path never
imports this package. The C source (`sattn_oracle.c`) shares nothing with the
CUDA implementation.

`topk_idxs` and `kv_ring_write` (cache bookkeeping around the path) are
plain Python; `compress_kv` (the compressor's gated pooling), the FP8 row
layout (`e4m3_encode` .. `dequantize_kv_fp8`) and the block-selection stages
(`xattn_partial_stats` .. `xattn_find_blocks`) are numpy fp64. The attention functions take float32 numpy arrays (the exact input
values, bf16 inputs widened) and return float64 outputs; each accepts an
optional `rows` array of row ids so that large workloads can be checked on
sampled rows:
  window:  row = token * H + head
  sparse:  row = (b * M + m) * H + head
  block:   row = i * H + head
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sattn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fno-fast-math", "-fPIC", "-shared",
                               "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_window.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, i32, P, i32,
                                          f64, P, i64, P, P]
            lib.oracle_sparse.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, P, i32, f64, P,
                                          i64, P, P]
            lib.oracle_block_sparse.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                                i32, i32, i32, f64, P, i64, P, P]
            lib.oracle_merge.argtypes = [P, P, i32, i64, i32, i32, P, P, P]
            lib.oracle_set_threads.argtypes = [i32]
            lib.oracle_get_threads.restype = i32
            _lib = lib
    return _lib


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def _f32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _rows(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, int(r.size)


def window(q, k, v, cu_seqlens, H, Hkv, d, window_left, window_right, causal, sinks,
           sink_mode, scale, rows=None):
    """Window attention; returns (o[nrows, d], lse[nrows]) in float64."""
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    s = None if sinks is None else _f32(sinks)
    r, nr = _rows(rows)
    n = nr if r is not None else int(cu[-1]) * H
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    rc = lib.oracle_window(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, H, Hkv, d,
                           window_left, window_right, causal, _ptr(s), sink_mode, float(scale),
                           _ptr(r), nr, _ptr(o), _ptr(lse))
    if rc:
        raise ValueError("oracle_window rejected its arguments (%d)" % rc)
    return o, lse


def sparse(q, kv, idx, sinks, sink_mode, scale, rows=None):
    """Gathered attention with one shared KV head; returns (o[nrows,d], lse[nrows])."""
    lib = _load()
    q, kv = _f32(q), _f32(kv)
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    B, M, H, d = q.shape
    N, K = kv.shape[1], ix.shape[2]
    s = None if sinks is None else _f32(sinks)
    r, nr = _rows(rows)
    n = nr if r is not None else B * M * H
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    rc = lib.oracle_sparse(_ptr(q), _ptr(kv), _ptr(ix), B, M, H, d, N, K, _ptr(s), sink_mode,
                           float(scale), _ptr(r), nr, _ptr(o), _ptr(lse))
    if rc:
        raise ValueError("oracle_sparse rejected its arguments (%d)" % rc)
    return o, lse


def block_sparse(q, k, v, mask, q_pos0, kv_begin, kv_end, causal, scale, blk=128, rows=None):
    """One KV chunk of block-sparse attention; returns (o_part[nrows,d], lse_part[nrows])."""
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    M, H, d = q.shape
    Nctx, Hkv = k.shape[0], k.shape[1]
    r, nr = _rows(rows)
    n = nr if r is not None else M * H
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    rc = lib.oracle_block_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(m), M, Nctx, H, Hkv, d,
                                 q_pos0, kv_begin, kv_end, causal, blk, float(scale), _ptr(r),
                                 nr, _ptr(o), _ptr(lse))
    if rc:
        raise ValueError("oracle_block_sparse rejected its arguments (%d)" % rc)
    return o, lse


def merge(o_parts, lse_parts, H, sinks=None):
    """LSE merge of C chunk partials o_parts[C,R,d], lse_parts[C,R]."""
    lib = _load()
    op = np.ascontiguousarray(o_parts, dtype=np.float64)
    lp = np.ascontiguousarray(lse_parts, dtype=np.float64)
    C, R, d = op.shape
    s = None if sinks is None else _f32(sinks)
    o = np.zeros((R, d), dtype=np.float64)
    lse = np.zeros(R, dtype=np.float64)
    lib.oracle_merge(_ptr(op), _ptr(lp), C, R, d, H, _ptr(s), _ptr(o), _ptr(lse))
    return o, lse


# ---------------------------------------------------------------------------
# Cache bookkeeping around the gathered path ("DeepSeek-V4 CSA/HCA
# walkthrough", section 2.3 steps 5-6 and section 3.3). Plain Python: these
# produce integers and copies, so parity with the GPU is exact.

def topk_idxs(start_pos, M, K, win, ratio):
    """Index lists of M consecutive queries of each request over a
    [window ring | compressed] cache; returns int32 [B, M, K].

    The query at absolute position p = start_pos[b] + m lists, in order:
      * the window: the win most recent tokens t = p-win+1 .. p, each at its
        ring row t mod win (the ring keeps token t in row t mod win), or -1
        for t < 0;
      * the compressed rows it may see, c = 0 .. floor(p / ratio) (cache row
        win + c) in ascending order; when more are visible than the K - win
        entries left, the most recent ones (no learned indexer here);
      * -1 for the entries left over. ratio = 0 means no compressed part.
    """
    start_pos = np.asarray(start_pos, dtype=np.int64)
    B = len(start_pos)
    out = np.full((B, M, K), -1, dtype=np.int32)
    for b in range(B):
        for m in range(M):
            p = int(start_pos[b]) + m
            entries = []
            for k in range(win):
                t = p - win + 1 + k
                entries.append(t % win if t >= 0 else -1)
            if ratio > 0:
                visible = list(range(p // ratio + 1))
                room = K - win
                chosen = visible if len(visible) <= room else visible[len(visible) - room:]
                entries.extend(win + c for c in chosen)
            n = min(len(entries), K)
            out[b, m, :n] = entries[:n]
    return out


def kv_ring_write(kv_cache, kv_new, start_pos, win):
    """Ring write of new KV rows: returns a copy of kv_cache [B, N, d] in which
    the last min(S, win) of the S new rows of request b (positions
    start_pos[b] .. start_pos[b] + S - 1) are stored.

    Written as the pages split it: with `cutoff` = the ring row of the first
    row written, the block goes to rows [cutoff, win) and then wraps to
    [0, cutoff) (rows before the block's last win are overwritten anyway).
    """
    out = np.array(kv_cache, copy=True)
    kv_new = np.asarray(kv_new)
    S = kv_new.shape[1]
    n = min(S, win)
    for b in range(out.shape[0]):
        block = kv_new[b, S - n:]
        cutoff = (int(start_pos[b]) + S - n) % win
        first = min(win - cutoff, n)
        out[b, cutoff:cutoff + first] = block[:first]
        out[b, :n - first] = block[first:]
    return out


# ---------------------------------------------------------------------------
# Compressor gated pooling ("DeepSeek-V4 CSA/HCA walkthrough", sections 5.1
# and 5.2). numpy fp64, steps in the pages' order.

def compress_kv(kv, score, ape, ratio, overlap):
    """Gated pooling of every `ratio` consecutive tokens into one compressed
    row; returns float64 [B, S // ratio, d].

    kv, score: [B, S, coff * d] with coff = 2 when `overlap` else 1 (the
    token projections the pages call wkv(x) and wgate(x)); ape: [ratio,
    coff * d], the learned absolute position term. The S % ratio tail tokens
    produce no row (the pages keep them in kv_state / score_state until their
    window is complete).

      1. the first S - S % ratio tokens form windows of `ratio` tokens;
      2. ape is added to each window's scores (entry i gets ape[i]);
      3. with overlap each window [ratio, 2d] becomes [2 ratio, d]: entries
         ratio .. 2 ratio - 1 are its own tokens' last d columns, entries
         0 .. ratio - 1 the previous window's tokens' first d columns; window 0
         has no previous window, so those entries hold kv = 0 and score = -inf
         (weight 0 after the softmax);
      4. softmax of the scores over the window entries, for each column;
      5. the row is the sum over the entries of kv times those weights.
    """
    kv = np.asarray(kv, dtype=np.float64)
    score = np.asarray(score, dtype=np.float64)
    ape = np.asarray(ape, dtype=np.float64)
    B, S, W = kv.shape
    coff = 2 if overlap else 1
    d = W // coff
    n = S // ratio
    kv_w = kv[:, :n * ratio].reshape(B, n, ratio, W)
    sc_w = score[:, :n * ratio].reshape(B, n, ratio, W) + ape
    if overlap:
        kv_o = np.zeros((B, n, 2 * ratio, d))
        sc_o = np.full((B, n, 2 * ratio, d), -np.inf)
        kv_o[:, :, ratio:] = kv_w[..., d:]
        sc_o[:, :, ratio:] = sc_w[..., d:]
        kv_o[:, 1:, :ratio] = kv_w[:, :-1, :, :d]
        sc_o[:, 1:, :ratio] = sc_w[:, :-1, :, :d]
        kv_w, sc_w = kv_o, sc_o
    if n == 0:
        return np.zeros((B, 0, d))
    m = sc_w.max(axis=2, keepdims=True)
    e = np.exp(sc_w - m)
    weights = e / e.sum(axis=2, keepdims=True)
    return (kv_w * weights).sum(axis=2)


# ---------------------------------------------------------------------------
# FP8 KV cache ("DeepSeek-V4 CSA/HCA walkthrough", section 2.3 step 4 and
# section 5.3: the non-RoPE part of each KV row is quantised to FP8, the RoPE
# part keeps a wider type). The pages leave the format open; the one used
# here: e4m3 (OCP FP8: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
# no infinities, S.1111.111 is NaN, largest finite 448) for the first d - rd
# columns with one float32 scale per row, scale = amax / 448 (1 when the row
# part is all zero), code = e4m3(x / scale) rounded to nearest even and
# saturated to +-448; the last rd columns stored as bf16.

def e4m3_decode(codes):
    """Values of e4m3 codes (uint8 array) as float64."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    val = np.where((e == 0xF) & (m == 0x7), np.nan, val)
    return sign * val


def _e4m3_table():
    codes = np.arange(0x7F, dtype=np.uint8)  # non-negative finite codes, ascending values
    return codes, e4m3_decode(codes)


def e4m3_encode(x):
    """Nearest e4m3 code of each value (float64 comparison, ties to the even
    code), saturating at +-448, the sign kept (also for results of zero);
    NaN -> 0x7F. A search over the 127 non-negative finite codes, so it does
    not depend on any bit manipulation."""
    x = np.asarray(x, dtype=np.float64)
    codes, vals = _e4m3_table()
    a = np.abs(x)
    hi = np.searchsorted(vals, np.minimum(a, 448.0), side="left")  # first value >= a
    hi = np.clip(hi, 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    dlo = np.abs(a - vals[lo])
    dhi = np.abs(vals[hi] - a)
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(codes[lo] % 2 == 0, lo, hi)))
    out = codes[pick].astype(np.uint8)
    out = np.where(a > 448.0, np.uint8(0x7E), out)
    out = np.where(np.signbit(x), out | 0x80, out)  # the sign is kept, zeros included
    out = np.where(np.isnan(x), np.uint8(0x7F), out)
    return out.astype(np.uint8)


def bf16_round(x):
    """float32 values rounded to bf16 (nearest even), widened back to float32."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def quantize_kv_fp8(kv, rd):
    """Split rows kv [..., d] (float32) into (codes uint8 [..., d - rd],
    rope float32 [..., rd] holding bf16 values, scale float32 [...]).
    All arithmetic in float32 as stated above."""
    kv = np.asarray(kv, dtype=np.float32)
    d = kv.shape[-1]
    nope, rope = kv[..., :d - rd], kv[..., d - rd:]
    amax = np.max(np.abs(nope), axis=-1) if d > rd else np.zeros(kv.shape[:-1], np.float32)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    codes = e4m3_encode((nope / scale[..., None]).astype(np.float32))
    return codes, bf16_round(rope), scale


def dequantize_kv_fp8(codes, rope, scale):
    """Rows [..., d] (float64) from the FP8 layout: e4m3 value x scale for the
    first d - rd columns, the rope part as stored."""
    nope = e4m3_decode(codes) * np.asarray(scale, dtype=np.float64)[..., None]
    return np.concatenate([nope, np.asarray(rope, dtype=np.float64)], axis=-1)


# ---------------------------------------------------------------------------
# XAttention block selection ("XAttention Offload Stream Synchronization Fix",
# technical details: three-stage KV chunking and the block selection step).
# The estimate here is the exact softmax at full resolution (the pages do not
# describe a cheaper estimator). numpy fp64.

def _visible(M, q_pos0, j0, j1, causal):
    """[M, j1 - j0] mask of keys j0 .. j1-1 each query row may see."""
    i = np.arange(M)[:, None]
    j = np.arange(j0, j1)[None, :]
    return (j <= q_pos0 + i) if causal else np.ones((M, j1 - j0), dtype=bool)


def xattn_partial_stats(q, k, q_pos0, kv_begin, kv_end, causal, scale):
    """Stage 1: over the keys j in [kv_begin, kv_end) that query row i may see
    (j <= q_pos0 + i when causal), per head h: m = max_j s_ij and
    l = sum_j exp(s_ij - m), with s_ij = scale <q[i, h], k[j, g]> and
    g = h // (H / Hkv); m = -inf, l = 0 when the row sees none of them.
    q [M, H, d], k [Nctx, Hkv, d]; returns float64 (m, l), each [M, H]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    M, H, _ = q.shape
    group = H // k.shape[1]
    vis = _visible(M, q_pos0, kv_begin, kv_end, causal)
    m = np.full((M, H), -np.inf)
    l = np.zeros((M, H))
    for h in range(H):
        s = scale * (q[:, h, :] @ k[kv_begin:kv_end, h // group, :].T)
        s = np.where(vis, s, -np.inf)
        if s.shape[1] == 0:
            continue
        mh = s.max(axis=1)
        ok = np.isfinite(mh)
        e = np.exp(s[ok] - mh[ok, None])
        m[ok, h] = mh[ok]
        l[ok, h] = e.sum(axis=1)
    return m, l


def xattn_merge_stats(m_parts, l_parts):
    """Stage 2: stats of the union of the chunks: m = max_c m_c,
    l = sum_c l_c exp(m_c - m) (chunks a row sees nothing of add nothing)."""
    m_parts = np.asarray(m_parts, dtype=np.float64)
    l_parts = np.asarray(l_parts, dtype=np.float64)
    m = m_parts.max(axis=0)
    fin = np.isfinite(m)
    w = np.where(np.isfinite(m_parts) & fin, np.exp(m_parts - np.where(fin, m, 0.0)), 0.0)
    l = np.where(fin, (l_parts * w).sum(axis=0), 0.0)
    return m, l


def xattn_block_sum(q, k, m, l, q_pos0, kv_begin, kv_end, causal, scale, blk=128):
    """Stage 3: softmax probabilities normalised with the global stats (m, l),
    p_ij = exp(s_ij - m_i) / l_i, summed over blk x blk blocks: entry
    [h, qb, kb] adds p_ij over rows i in query block qb (i // blk, local) and
    visible keys j in key block kb (j // blk, absolute) within [kv_begin,
    kv_end). Returns float64 [H, ceil(M/blk), ceil(Nctx/blk)], zero for key
    blocks outside the range."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    M, H, _ = q.shape
    Nctx = k.shape[0]
    group = H // k.shape[1]
    QB, KB = -(-M // blk), -(-Nctx // blk)
    out = np.zeros((H, QB, KB))
    vis = _visible(M, q_pos0, kv_begin, kv_end, causal)
    for h in range(H):
        s = scale * (q[:, h, :] @ k[kv_begin:kv_end, h // group, :].T)
        ok = np.isfinite(m[:, h]) & (l[:, h] > 0)
        p = np.zeros_like(s)
        p[ok] = np.exp(s[ok] - m[ok, h, None]) / l[ok, h, None]
        p = np.where(vis, p, 0.0)
        kb_of = np.arange(kv_begin, kv_end) // blk
        qb_of = np.arange(M) // blk
        for kb in np.unique(kb_of):
            cols = p[:, kb_of == kb].sum(axis=1)
            for qb in range(QB):
                out[h, qb, kb] = cols[qb_of == qb].sum()
    return out


def xattn_find_blocks(block_sum, threshold):
    """Step 4: for each (head, query block) the key blocks ordered by mass
    (largest first, the lower block first among equal masses) and the
    shortest leading run of them whose cumulative mass reaches threshold x
    the total is selected. Sums in float64, in that order, from the given
    values (a kernel's fp32 sums reproduce the decisions exactly). A block
    mass is a sum of probabilities, so it cannot be negative; a given value
    that is negative or NaN counts as a mass of 0 (the library's contract for
    caller-supplied sums). Returns uint8 [H, QB, KB]; nothing is selected
    where the total is not positive."""
    bs = np.asarray(block_sum)
    H, QB, KB = bs.shape
    out = np.zeros((H, QB, KB), dtype=np.uint8)
    for h in range(H):
        for qb in range(QB):
            v = [float(x) if float(x) > 0.0 else 0.0 for x in bs[h, qb]]
            order = sorted(range(KB), key=lambda kb: (-v[kb], kb))
            total = 0.0
            for kb in order:
                total += v[kb]
            if not total > 0.0:
                continue
            target = float(threshold) * total
            cum = 0.0
            for kb in order:
                cum += v[kb]
                out[h, qb, kb] = 1
                if cum >= target:
                    break
    return out
