"""sattn for GB300: index-gathered attention forward with sinks.

A thin binding over libsattn.so (C ABI, include/sattn.h). The functions here
only marshal torch tensors into device pointers, sizes and the current CUDA
stream; every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback: if the library is missing or cannot load, every
call raises.
"""
from __future__ import annotations

import ctypes
import os

from . import workloads  # noqa: F401  (seeded input generators)

SINK_NONE, SINK_KEY0_BIAS, SINK_NULL_LOGIT = 0, 1, 2
F32, BF16 = 0, 1
BLOCK = 128

_PKG = os.path.dirname(os.path.abspath(__file__))
# SATTN_LIBRARY may name another build of libsattn.so to load instead.
LIB_PATH = os.environ.get("SATTN_LIBRARY") or os.path.join(_PKG, "libsattn.so")

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error",
          4: "device check failed", 5: "device wait timed out"}

_lib = None


class SattnError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__("%s failed: %s (%d)" % (fn, STATUS.get(code, "?"), code))
        self.code = code


def lib() -> ctypes.CDLL:
    """Load libsattn.so (built by build.build()) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libsattn.so is not built; run windowed_attention_sinks_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    L.sattn_window_fwd.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                   P, ctypes.c_int, f32, ctypes.c_int, P]
    L.sattn_window_fwd.restype = ctypes.c_int
    L.sattn_sparse_fwd.argtypes = [P, P, P, P, ctypes.c_int, f32, P, P, i32, i32, i32, i32, i32,
                                   i32, P, sz, ctypes.c_int, P]
    L.sattn_sparse_fwd.restype = ctypes.c_int
    L.sattn_sparse_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    L.sattn_sparse_workspace_bytes.restype = sz
    L.sattn_merge_lse.argtypes = [P, P, i32, i64, i32, i32, P, P, P, ctypes.c_int, P]
    L.sattn_merge_lse.restype = ctypes.c_int
    L.sattn_block_sparse_fwd.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                         f32, P, P, ctypes.c_int, P]
    L.sattn_block_sparse_fwd.restype = ctypes.c_int
    L.sattn_block_sparse_chunks_fwd.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                                i32, i32, i32, f32, P, P, ctypes.c_int, P]
    L.sattn_block_sparse_chunks_fwd.restype = ctypes.c_int
    L.sattn_build_topk_idxs.argtypes = [P, P, i32, i32, i32, i32, i32, P]
    L.sattn_build_topk_idxs.restype = ctypes.c_int
    L.sattn_kv_ring_write.argtypes = [P, P, P, i32, i32, i32, i32, i32, ctypes.c_int, P]
    L.sattn_kv_ring_write.restype = ctypes.c_int
    L.sattn_quantize_kv_fp8.argtypes = [P, P, P, P, i64, i32, i32, ctypes.c_int, P]
    L.sattn_quantize_kv_fp8.restype = ctypes.c_int
    L.sattn_sparse_fp8_fwd.argtypes = [P, P, P, P, P, P, ctypes.c_int, f32, P, P, i32, i32, i32,
                                       i32, i32, i32, i32, P, sz, P]
    L.sattn_sparse_fp8_fwd.restype = ctypes.c_int
    L.sattn_xattn_partial_stats.argtypes = [P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                            f32, P, P, P]
    L.sattn_xattn_partial_stats.restype = ctypes.c_int
    L.sattn_xattn_merge_stats.argtypes = [P, P, i32, i64, P, P, P]
    L.sattn_xattn_merge_stats.restype = ctypes.c_int
    L.sattn_xattn_block_sum.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                        f32, P, P]
    L.sattn_xattn_block_sum.restype = ctypes.c_int
    L.sattn_xattn_find_blocks.argtypes = [P, i32, i32, i32, f32, P, P]
    L.sattn_xattn_find_blocks.restype = ctypes.c_int
    L.sattn_xattn_select_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.sattn_xattn_select_workspace_bytes.restype = sz
    L.sattn_xattn_select_blocks.argtypes = [P, P, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                                            f32, P, sz, P, P, P]
    L.sattn_xattn_select_blocks.restype = ctypes.c_int
    L.sattn_compress_kv.argtypes = [P, P, P, P, i64, i32, i32, i32, i32, i32, ctypes.c_int,
                                    ctypes.c_int, P]
    L.sattn_compress_kv.restype = ctypes.c_int
    L.sattn_status_str.argtypes = [ctypes.c_int]
    L.sattn_status_str.restype = ctypes.c_char_p
    L.sattn_set_debug.argtypes = [ctypes.c_int]
    L.sattn_set_debug.restype = None
    L.sattn_check_device.argtypes = [P]
    L.sattn_check_device.restype = ctypes.c_int
    L.sattn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.sattn_set_wait_limit_ns.restype = None
    L.sattn_set_test_wait_stall.argtypes = [ctypes.c_int]
    L.sattn_set_test_wait_stall.restype = None
    L.sattn_version.restype = i32
    _lib = L
    return L


def _check(fn, code):
    if code != 0:
        raise SattnError(fn, code)


def _dtype_code(t):
    import torch

    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("unsupported dtype %s" % t.dtype)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _need(t, name, dtype=None, device=None):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s" % (name, dtype))
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))


def window_fwd(q, k, v, cu_seqlens, max_seqlen, window_left, window_right, causal=False,
               sinks=None, sink_mode=SINK_NONE, scale=None, o=None, lse=None, stream=None):
    """Sliding-window varlen attention (sattn_window_fwd). Returns (o, lse)."""
    import torch

    T, H, d = q.shape
    Hkv = k.shape[1]
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, q.device)
    _need(cu_seqlens, "cu_seqlens", torch.int32, q.device)
    if sinks is not None:
        _need(sinks, "sinks", torch.float32, q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    scale = float(d ** -0.5 if scale is None else scale)
    code = lib().sattn_window_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens),
                                  cu_seqlens.numel() - 1, T, int(max_seqlen), H, Hkv, d,
                                  int(window_left), int(window_right), int(bool(causal)),
                                  _ptr(sinks), int(sink_mode), scale, _dtype_code(q),
                                  _stream(stream))
    _check("sattn_window_fwd", code)
    return o, lse


def sparse_workspace_bytes(B, M, H, d, K):
    return int(lib().sattn_sparse_workspace_bytes(B, M, H, d, K))


def sparse_fwd(q, kv_cache, topk_idxs, sinks=None, sink_mode=SINK_NONE, scale=None, o=None,
               lse=None, workspace=None, stream=None):
    """Gathered attention over one shared KV head (sattn_sparse_fwd). Returns (o, lse)."""
    import torch

    B, M, H, d = q.shape
    N = kv_cache.shape[1]
    K = topk_idxs.shape[2]
    _need(q, "q", None, q.device)
    _need(kv_cache, "kv_cache", q.dtype, q.device)
    _need(topk_idxs, "topk_idxs", torch.int32, q.device)
    if sinks is not None:
        _need(sinks, "sinks", torch.float32, q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, M, H), dtype=torch.float32, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = float(d ** -0.5 if scale is None else scale)
    code = lib().sattn_sparse_fwd(_ptr(q), _ptr(kv_cache), _ptr(topk_idxs), _ptr(sinks),
                                  int(sink_mode), scale, _ptr(o), _ptr(lse), B, M, H, d, N, K,
                                  _ptr(workspace), ws_bytes, _dtype_code(q), _stream(stream))
    _check("sattn_sparse_fwd", code)
    return o, lse


def quantize_kv_fp8(kv, rd, stream=None):
    """FP8 layout of KV rows (sattn_quantize_kv_fp8): kv [..., d] (bf16 or fp32)
    -> (codes uint8 [..., d - rd], rope bf16 [..., rd], scale fp32 [...])."""
    import torch

    _need(kv, "kv", None, kv.device)
    d = kv.shape[-1]
    lead = tuple(kv.shape[:-1])
    rows = kv.numel() // d if d else 0
    nope = torch.empty(lead + (d - rd,), dtype=torch.uint8, device=kv.device)
    rope = torch.empty(lead + (rd,), dtype=torch.bfloat16, device=kv.device)
    scale = torch.empty(lead, dtype=torch.float32, device=kv.device)
    _check("sattn_quantize_kv_fp8",
           lib().sattn_quantize_kv_fp8(_ptr(kv), _ptr(nope), _ptr(rope), _ptr(scale), rows, d,
                                       int(rd), _dtype_code(kv), _stream(stream)))
    return nope, rope, scale


def sparse_fp8_fwd(q, kv_nope, kv_rope, kv_scale, topk_idxs, sinks=None, sink_mode=SINK_NONE,
                   scale=None, o=None, lse=None, workspace=None, stream=None):
    """Gathered attention over an FP8 cache (sattn_sparse_fp8_fwd): kv_nope
    uint8 [B, N, d - rd], kv_rope bf16 [B, N, rd], kv_scale fp32 [B, N].
    Returns (o, lse)."""
    import torch

    B, M, H, d = q.shape
    N, rd = kv_rope.shape[1], kv_rope.shape[2]
    K = topk_idxs.shape[2]
    _need(q, "q", torch.bfloat16, q.device)
    _need(kv_nope, "kv_nope", torch.uint8, q.device)
    _need(kv_rope, "kv_rope", torch.bfloat16, q.device)
    _need(kv_scale, "kv_scale", torch.float32, q.device)
    _need(topk_idxs, "topk_idxs", torch.int32, q.device)
    if tuple(kv_nope.shape) != (B, N, d - rd) or tuple(kv_scale.shape) != (B, N):
        raise ValueError("kv_nope must be [B, N, d - rd] and kv_scale [B, N]")
    if sinks is not None:
        _need(sinks, "sinks", torch.float32, q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, M, H), dtype=torch.float32, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = float(d ** -0.5 if scale is None else scale)
    code = lib().sattn_sparse_fp8_fwd(_ptr(q), _ptr(kv_nope), _ptr(kv_rope), _ptr(kv_scale),
                                      _ptr(topk_idxs), _ptr(sinks), int(sink_mode), scale, _ptr(o),
                                      _ptr(lse), B, M, H, d, rd, N, K, _ptr(workspace), ws_bytes,
                                      _stream(stream))
    _check("sattn_sparse_fp8_fwd", code)
    return o, lse


def merge_lse(o_parts, lse_parts, H, sinks=None, out_dtype=None, o=None, lse=None, stream=None):
    """LSE merge of chunk partials (sattn_merge_lse). o_parts[C,R,d], lse_parts[C,R] fp32."""
    import torch

    C, R, d = o_parts.shape
    _need(o_parts, "o_parts", torch.float32)
    _need(lse_parts, "lse_parts", torch.float32, o_parts.device)
    if o is None:
        o = torch.empty((R, d), dtype=out_dtype or torch.float32, device=o_parts.device)
    if lse is None:
        lse = torch.empty((R,), dtype=torch.float32, device=o_parts.device)
    code = lib().sattn_merge_lse(_ptr(o_parts), _ptr(lse_parts), C, R, d, H, _ptr(sinks), _ptr(o),
                                 _ptr(lse), _dtype_code(o), _stream(stream))
    _check("sattn_merge_lse", code)
    return o, lse


def block_sparse_fwd(q, k, v, block_mask, q_pos0, kv_begin, kv_end, causal=True, scale=None,
                     o_part=None, lse_part=None, stream=None):
    """One KV chunk of block-sparse attention (sattn_block_sparse_fwd). Returns fp32 partials."""
    import torch

    M, H, d = q.shape
    Nctx, Hkv = k.shape[0], k.shape[1]
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, q.device)
    _need(block_mask, "block_mask", torch.uint8, q.device)
    if o_part is None:
        o_part = torch.empty((M, H, d), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((M, H), dtype=torch.float32, device=q.device)
    scale = float(d ** -0.5 if scale is None else scale)
    code = lib().sattn_block_sparse_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(block_mask), M, Nctx, H,
                                        Hkv, d, int(q_pos0), int(kv_begin), int(kv_end),
                                        int(bool(causal)), scale, _ptr(o_part), _ptr(lse_part),
                                        _dtype_code(q), _stream(stream))
    _check("sattn_block_sparse_fwd", code)
    return o_part, lse_part


def block_sparse_chunks_fwd(q, k, v, block_mask, q_pos0, kv_begin, kv_end, chunk, causal=True,
                            scale=None, o_parts=None, lse_parts=None, stream=None):
    """Every chunk of `chunk` keys of [kv_begin, kv_end) at once
    (sattn_block_sparse_chunks_fwd): fp32 partials [C, M, H, d] and [C, M, H],
    the same as block_sparse_fwd chunk by chunk."""
    import torch

    M, H, d = q.shape
    Nctx, Hkv = k.shape[0], k.shape[1]
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, q.device)
    _need(block_mask, "block_mask", torch.uint8, q.device)
    C = -(-(int(kv_end) - int(kv_begin)) // int(chunk)) if chunk > 0 else 0
    if o_parts is None:
        o_parts = torch.empty((C, M, H, d), dtype=torch.float32, device=q.device)
    if lse_parts is None:
        lse_parts = torch.empty((C, M, H), dtype=torch.float32, device=q.device)
    scale = float(d ** -0.5 if scale is None else scale)
    code = lib().sattn_block_sparse_chunks_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(block_mask), M,
                                               Nctx, H, Hkv, d, int(q_pos0), int(kv_begin),
                                               int(kv_end), int(chunk), int(bool(causal)), scale,
                                               _ptr(o_parts), _ptr(lse_parts), _dtype_code(q),
                                               _stream(stream))
    _check("sattn_block_sparse_chunks_fwd", code)
    return o_parts, lse_parts


def build_topk_idxs(start_pos, M, K, win, ratio, out=None, stream=None):
    """Index lists over a [window ring | compressed] cache (sattn_build_topk_idxs).
    start_pos: int32 [B] CUDA tensor. Returns int32 [B, M, K]."""
    import torch

    _need(start_pos, "start_pos", torch.int32)
    B = start_pos.numel()
    if out is None:
        out = torch.empty((B, M, K), dtype=torch.int32, device=start_pos.device)
    _need(out, "out", torch.int32, start_pos.device)
    _check("sattn_build_topk_idxs",
           lib().sattn_build_topk_idxs(_ptr(out), _ptr(start_pos), B, int(M), int(K), int(win),
                                       int(ratio), _stream(stream)))
    return out


def kv_ring_write(kv_cache, kv_new, start_pos, win, stream=None):
    """Store the last min(S, win) new rows of each request at their ring rows
    (sattn_kv_ring_write). kv_cache [B, N, d] is updated in place."""
    import torch

    B, N, d = kv_cache.shape
    S = kv_new.shape[1]
    _need(kv_cache, "kv_cache", None, kv_cache.device)
    _need(kv_new, "kv_new", kv_cache.dtype, kv_cache.device)
    _need(start_pos, "start_pos", torch.int32, kv_cache.device)
    _check("sattn_kv_ring_write",
           lib().sattn_kv_ring_write(_ptr(kv_cache), _ptr(kv_new), _ptr(start_pos), B, S, N, d,
                                     int(win), _dtype_code(kv_cache), _stream(stream)))
    return kv_cache


def compress_kv(kv, score, ape, ratio, overlap, out=None, out_dtype=None, stream=None):
    """Compressor gated pooling (sattn_compress_kv): every `ratio` tokens of
    kv / score [B, S, coff*d] (coff = 2 with overlap) become one row of out
    [B, S // ratio, d]. `out` may be a view with a batch stride (e.g. the
    compressed rows of a cache: kv_cache[:, win:win + S // ratio]) whose rows
    are contiguous; by default a new tensor of `out_dtype` (kv's dtype)."""
    import torch

    B, S, W = kv.shape
    coff = 2 if overlap else 1
    if W % coff:
        raise ValueError("kv width %d is not a multiple of %d" % (W, coff))
    d = W // coff
    _need(kv, "kv", None, kv.device)
    _need(score, "score", kv.dtype, kv.device)
    _need(ape, "ape", torch.float32, kv.device)
    if tuple(score.shape) != tuple(kv.shape) or tuple(ape.shape) != (int(ratio), W):
        raise ValueError("score must match kv and ape must be [ratio, coff*d]")
    nwin = S // int(ratio)
    if out is None:
        out = torch.empty((B, nwin, d), dtype=out_dtype or kv.dtype, device=kv.device)
    if out.dim() != 3 or tuple(out.shape) != (B, nwin, d) or out.stride(2) != 1 or \
            (nwin > 1 and out.stride(1) != d) or out.device != kv.device:
        raise ValueError("out must be [B, S // ratio, d] with contiguous rows")
    _check("sattn_compress_kv",
           lib().sattn_compress_kv(_ptr(kv), _ptr(score), _ptr(ape), _ptr(out),
                                   int(out.stride(0)) if B > 1 else nwin * d, B, S, d,
                                   int(ratio), 1 if overlap else 0, _dtype_code(kv),
                                   _dtype_code(out), _stream(stream)))
    return out


def xattn_partial_stats(q, k, q_pos0, kv_begin, kv_end, causal, scale=None, m=None, l=None,
                        stream=None):
    """Stage 1 of the block selection over keys [kv_begin, kv_end)
    (sattn_xattn_partial_stats): q bf16 [M, H, 128], k bf16 [Nctx, Hkv, 128].
    Returns (m, l), float32 [M, H]."""
    import torch

    M, H, d = q.shape
    Nctx, Hkv = k.shape[0], k.shape[1]
    _need(q, "q", torch.bfloat16, q.device)
    _need(k, "k", torch.bfloat16, q.device)
    if m is None:
        m = torch.empty((M, H), dtype=torch.float32, device=q.device)
    if l is None:
        l = torch.empty((M, H), dtype=torch.float32, device=q.device)
    scale = float(d ** -0.5 if scale is None else scale)
    _check("sattn_xattn_partial_stats",
           lib().sattn_xattn_partial_stats(_ptr(q), _ptr(k), M, Nctx, H, Hkv, d, int(q_pos0),
                                           int(kv_begin), int(kv_end), int(bool(causal)), scale,
                                           _ptr(m), _ptr(l), _stream(stream)))
    return m, l


def xattn_merge_stats(m_parts, l_parts, m=None, l=None, stream=None):
    """Stage 2 (sattn_xattn_merge_stats): [C, ...] partial stats -> merged (m, l)."""
    import torch

    _need(m_parts, "m_parts", torch.float32)
    _need(l_parts, "l_parts", torch.float32, m_parts.device)
    C = m_parts.shape[0]
    R = m_parts[0].numel() if C else 0
    if m is None:
        m = torch.empty(m_parts.shape[1:], dtype=torch.float32, device=m_parts.device)
    if l is None:
        l = torch.empty(m_parts.shape[1:], dtype=torch.float32, device=m_parts.device)
    _check("sattn_xattn_merge_stats",
           lib().sattn_xattn_merge_stats(_ptr(m_parts), _ptr(l_parts), C, R, _ptr(m), _ptr(l),
                                         _stream(stream)))
    return m, l


def xattn_block_sum(q, k, m, l, q_pos0, kv_begin, kv_end, causal, scale=None, block_sum=None,
                    stream=None):
    """Stage 3 (sattn_xattn_block_sum): adds the chunk's key blocks to
    block_sum float32 [H, ceil(M/128), ceil(Nctx/128)] (zeros if not given)."""
    import torch

    M, H, d = q.shape
    Nctx, Hkv = k.shape[0], k.shape[1]
    _need(q, "q", torch.bfloat16, q.device)
    _need(k, "k", torch.bfloat16, q.device)
    _need(m, "m", torch.float32, q.device)
    _need(l, "l", torch.float32, q.device)
    if block_sum is None:
        block_sum = torch.zeros((H, -(-M // BLOCK), -(-Nctx // BLOCK)), dtype=torch.float32,
                                device=q.device)
    _need(block_sum, "block_sum", torch.float32, q.device)
    scale = float(d ** -0.5 if scale is None else scale)
    _check("sattn_xattn_block_sum",
           lib().sattn_xattn_block_sum(_ptr(q), _ptr(k), _ptr(m), _ptr(l), M, Nctx, H, Hkv, d,
                                       int(q_pos0), int(kv_begin), int(kv_end),
                                       int(bool(causal)), scale, _ptr(block_sum),
                                       _stream(stream)))
    return block_sum


def xattn_find_blocks(block_sum, threshold, mask=None, stream=None):
    """Step 4 (sattn_xattn_find_blocks): uint8 mask [H, QB, KB]."""
    import torch

    _need(block_sum, "block_sum", torch.float32)
    H, QB, KB = block_sum.shape
    if mask is None:
        mask = torch.empty((H, QB, KB), dtype=torch.uint8, device=block_sum.device)
    _check("sattn_xattn_find_blocks",
           lib().sattn_xattn_find_blocks(_ptr(block_sum), H, QB, KB, float(threshold), _ptr(mask),
                                         _stream(stream)))
    return mask


def xattn_select_workspace_bytes(M, H, Nctx, chunk=4096):
    """Workspace bytes of xattn_select_blocks (sattn_xattn_select_workspace_bytes)."""
    return int(lib().sattn_xattn_select_workspace_bytes(int(M), int(H), int(Nctx), int(chunk)))


def xattn_select_blocks(q, k, q_pos0, causal, threshold, scale=None, chunk=4096, workspace=None,
                        block_sum=None, mask=None, stream=None):
    """The whole selection in one call (sattn_xattn_select_blocks): partial
    stats per KV chunk of `chunk` keys, their merge, block sums with the
    merged stats, the threshold selection. Returns (mask uint8 [H, QB, KB],
    block_sum float32 [H, QB, KB])."""
    import torch

    M, H, d = q.shape
    Nctx, Hkv = k.shape[0], k.shape[1]
    _need(q, "q", torch.bfloat16, q.device)
    _need(k, "k", torch.bfloat16, q.device)
    shape = (H, -(-M // BLOCK), -(-Nctx // BLOCK))
    if block_sum is None:
        block_sum = torch.empty(shape, dtype=torch.float32, device=q.device)
    if mask is None:
        mask = torch.empty(shape, dtype=torch.uint8, device=q.device)
    _need(block_sum, "block_sum", torch.float32, q.device)
    _need(mask, "mask", torch.uint8, q.device)
    if tuple(block_sum.shape) != shape or tuple(mask.shape) != shape:
        raise ValueError("block_sum and mask must have shape %s" % (shape,))
    nb = xattn_select_workspace_bytes(M, H, Nctx, chunk)
    if workspace is None:
        workspace = torch.empty(max(nb, 16), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", None, q.device)
    scale = float(d ** -0.5 if scale is None else scale)
    _check("sattn_xattn_select_blocks",
           lib().sattn_xattn_select_blocks(_ptr(q), _ptr(k), M, Nctx, H, Hkv, d, int(q_pos0),
                                           int(bool(causal)), scale, int(chunk), float(threshold),
                                           _ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _ptr(block_sum), _ptr(mask), _stream(stream)))
    return mask, block_sum


def check_device(stream=None):
    """Synchronise and read/clear the device error word; raises on a recorded error."""
    _check("sattn_check_device", lib().sattn_check_device(_stream(stream)))


def set_debug(on: bool):
    lib().sattn_set_debug(1 if on else 0)


def set_wait_limit_ns(ns: int):
    """Bound on any single wait inside a kernel (sattn_set_wait_limit_ns); 0 = default."""
    lib().sattn_set_wait_limit_ns(int(ns))


def set_test_wait_stall(on: bool):
    """Test hook (sattn_set_test_wait_stall): later tensor-core launches take
    their timeout path; outputs undefined, SATTN_ERR_TIMEOUT recorded."""
    lib().sattn_set_test_wait_stall(1 if on else 0)
