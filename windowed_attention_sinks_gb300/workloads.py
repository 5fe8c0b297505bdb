"""Seeded synthetic inputs for the attention workloads and the compressor.

This module only draws random numbers and builds index structures. It holds
none of the attention arithmetic, so both the CUDA path and the CPU oracle
consume its output without sharing any computation.

Every tensor comes from its own numpy PCG64 stream keyed by
(workload id, tensor id, seed). Floating-point tensors are returned as float32
numpy arrays; for bf16 workloads they are already rounded to bf16
(round-to-nearest-even, via torch) and widened back, so the float32 array
holds exactly the values the GPU receives.

Workload shapes follow the pages:
  * window, fp32, tiny: vLLM PR #49815 report, "Implementation" item 4 and the
    `_reference` test listing (sequences of 5 and 37 tokens, window 8).
  * window, bf16, vision encoder: same report, `_forward_window_attn`
    (non-causal, window on both sides, per-head sinks on key 0).
  * sparse decode / prefill: DeepSeek-V4 CSA/HCA walkthrough, sections 2.2,
    2.3 (steps 5-7) and 3.3 (`kv_cache` = window ring then compressed rows,
    `topk_idxs` = window indices concatenated with compressed indices, -1 for
    invalid entries, section 4.2).
  * chunked block-sparse: nano-vllm "XAttention Offload Stream
    Synchronization Fix", technical details (4096-key chunks, partial
    (m, l) stats merged afterwards) and test results (~10% density at 32K).
  * compressor gated pooling: DeepSeek-V4 CSA/HCA walkthrough, sections 2.2
    (compress_ratio 4) and 5.1-5.2 (kv / gate projections of every token,
    ape, overlap windows); the projections are drawn directly (no weights).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

SINK_NONE = 0
SINK_KEY0_BIAS = 1
SINK_NULL_LOGIT = 2
SINK_MODES = {"none": SINK_NONE, "key0_bias": SINK_KEY0_BIAS, "null_logit": SINK_NULL_LOGIT}

_TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "kv": 4, "sinks": 5, "lens": 6, "idx": 7, "drop": 8, "mask": 9,
               "score": 10, "ape": 11}


def _rng(workload: int, tensor: str, seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([workload, _TENSOR_IDS[tensor], seed]))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even) and widen back to float32."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def _normal(workload: int, tensor: str, seed: int, shape, std: float = 1.0) -> np.ndarray:
    x = _rng(workload, tensor, seed).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


@dataclass
class WindowCase:
    """Packed varlen window attention: q[T,H,d], k/v[T,Hkv,d], cu_seqlens[S+1]."""

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    sinks: np.ndarray
    cu_seqlens: np.ndarray
    H: int
    Hkv: int
    d: int
    window_left: int
    window_right: int
    causal: int
    scale: float
    dtype: str  # "f32" or "bf16"
    sink_mode: int = SINK_KEY0_BIAS

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def num_seqs(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def max_seqlen(self) -> int:
        return int(np.max(np.diff(self.cu_seqlens))) if self.num_seqs else 0


def window_tiny_f32(seed: int, hkv: int, sink_mode: int = SINK_KEY0_BIAS) -> WindowCase:
    """Two sequences (5 and 37 tokens), 8 query heads, d=64, window 8, fp32."""
    W = 1
    cu = np.array([0, 5, 42], dtype=np.int32)
    T, H, d = 42, 8, 64
    return WindowCase(
        q=_normal(W, "q", seed, (T, H, d)),
        k=_normal(W, "k", seed, (T, hkv, d)),
        v=_normal(W, "v", seed, (T, hkv, d)),
        sinks=_normal(W, "sinks", seed, (H,)),
        cu_seqlens=cu, H=H, Hkv=hkv, d=d, window_left=8, window_right=8, causal=0,
        scale=1.0 / math.sqrt(d), dtype="f32", sink_mode=sink_mode)


def window_vision_bf16(seed: int, hkv: int, sink_mode: int = SINK_KEY0_BIAS,
                       num_seqs: int = 256, min_len: int = 64, max_len: int = 1024,
                       H: int = 16, d: int = 128, window: int = 128) -> WindowCase:
    """Vision-encoder windowed attention: lengths ~ U{min_len..max_len}, q,k,v ~ 0.5 N(0,1)."""
    W = 2
    lens = _rng(W, "lens", seed).integers(min_len, max_len + 1, size=num_seqs)
    cu = np.zeros(num_seqs + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    T = int(cu[-1])
    return WindowCase(
        q=round_bf16(_normal(W, "q", seed, (T, H, d), 0.5)),
        k=round_bf16(_normal(W, "k", seed, (T, hkv, d), 0.5)),
        v=round_bf16(_normal(W, "v", seed, (T, hkv, d), 0.5)),
        sinks=_normal(W, "sinks", seed, (H,)),
        cu_seqlens=cu, H=H, Hkv=hkv, d=d, window_left=window, window_right=window, causal=0,
        scale=1.0 / math.sqrt(d), dtype="bf16", sink_mode=sink_mode)


@dataclass
class SparseCase:
    """Index-gathered attention over one shared KV head.

    q[B,M,H,d], kv_cache[B,N,d] (the row is both key and value),
    topk_idxs[B,M,K] int32 in [-1, N).
    """

    q: np.ndarray
    kv: np.ndarray
    idx: np.ndarray
    sinks: np.ndarray
    scale: float
    sink_mode: int = SINK_NULL_LOGIT
    dtype: str = "bf16"

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def M(self):
        return self.q.shape[1]

    @property
    def H(self):
        return self.q.shape[2]

    @property
    def d(self):
        return self.q.shape[3]

    @property
    def N(self):
        return self.kv.shape[1]

    @property
    def K(self):
        return self.idx.shape[2]


def sparse_decode_bf16(seed: int, B: int = 64, H: int = 32, d: int = 128, win: int = 128,
                       n_compressed: int = 8192, n_window_idx: int = 128,
                       n_compress_idx: int = 512, n_invalid: int = 64,
                       sink_mode: int = SINK_NULL_LOGIT) -> SparseCase:
    """Decode: one query per request over a [ring window | compressed] cache.

    The index list is the full ring (0..win-1) followed by distinct draws from
    the compressed region (stored at win + c); exactly `n_invalid` of the
    entries are then replaced by -1 at seeded positions.
    """
    W = 3
    N = win + n_compressed
    K = n_window_idx + n_compress_idx
    q = round_bf16(_normal(W, "q", seed, (B, 1, H, d)))
    kv = round_bf16(_normal(W, "kv", seed, (B, N, d)))
    rng = _rng(W, "idx", seed)
    drop = _rng(W, "drop", seed)
    idx = np.empty((B, 1, K), dtype=np.int32)
    for b in range(B):
        window = np.arange(n_window_idx, dtype=np.int64) % win
        comp = win + rng.choice(n_compressed, size=n_compress_idx, replace=False)
        row = np.concatenate([window, comp]).astype(np.int32)
        row[drop.permutation(K)[:n_invalid]] = -1
        idx[b, 0] = row
    return SparseCase(q=q, kv=kv, idx=idx, sinks=_normal(W, "sinks", seed, (H,)),
                      scale=1.0 / math.sqrt(d), sink_mode=sink_mode)


def prefill_topk_idxs(seed: int, M: int, win: int = 128, ratio: int = 4,
                      K: int = 2048, pos0: int = 0) -> np.ndarray:
    """Per-query index lists for causal sparse prefill.

    For the query at position p (= pos0 + i):
      * window part, `win` entries: slot k maps to token t = p - (win-1) + k,
        stored at ring position t mod win, or -1 when t < 0;
      * compressed part: compressed rows c <= p // ratio, stored at win + c.
        If all fit in K - win they are taken in ascending order, otherwise
        K - win distinct ones are drawn with the seed (kept ascending);
      * -1 padding up to K entries.
    """
    W = 4
    rng = _rng(W, "idx", seed)
    cap = K - win
    out = np.full((1, M, K), -1, dtype=np.int32)
    ks = np.arange(win, dtype=np.int64)
    for i in range(M):
        p = pos0 + i
        t = p - (win - 1) + ks
        out[0, i, :win] = np.where(t >= 0, t % win, -1)
        avail = p // ratio + 1
        if avail <= cap:
            comp = np.arange(avail, dtype=np.int64)
        else:
            comp = np.sort(rng.choice(avail, size=cap, replace=False))
        out[0, i, win:win + len(comp)] = win + comp
    return out


def sparse_prefill_bf16(seed: int, M: int = 8192, H: int = 32, d: int = 128, win: int = 128,
                        n_compressed: int = 8192, K: int = 2048, ratio: int = 4,
                        sink_mode: int = SINK_NULL_LOGIT) -> SparseCase:
    """Prefill: M query tokens of one sequence, K index entries per query."""
    W = 4
    N = win + n_compressed
    q = round_bf16(_normal(W, "q", seed, (1, M, H, d)))
    kv = round_bf16(_normal(W, "kv", seed, (1, N, d)))
    idx = prefill_topk_idxs(seed, M, win=win, ratio=ratio, K=K)
    return SparseCase(q=q, kv=kv, idx=idx, sinks=_normal(W, "sinks", seed, (H,)),
                      scale=1.0 / math.sqrt(d), sink_mode=sink_mode)


@dataclass
class BlockSparseCase:
    """Chunked block-sparse causal attention.

    q[M,H,d] at positions q_pos0 .. q_pos0+M-1; k/v[Nctx,Hkv,d];
    block_mask uint8[H, ceil(M/blk), ceil(Nctx/blk)]: query blocks are local
    (i // blk), key blocks are global (j // blk).
    """

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    mask: np.ndarray
    q_pos0: int
    chunk: int
    scale: float
    blk: int = 128
    causal: int = 1
    dtype: str = "bf16"

    @property
    def M(self):
        return self.q.shape[0]

    @property
    def H(self):
        return self.q.shape[1]

    @property
    def d(self):
        return self.q.shape[2]

    @property
    def Nctx(self):
        return self.k.shape[0]

    @property
    def Hkv(self):
        return self.k.shape[1]

    @property
    def chunks(self):
        return [(c, min(c + self.chunk, self.Nctx)) for c in range(0, self.Nctx, self.chunk)]


def block_sparse_bf16(seed: int, Nctx: int = 32768, M: int = 4096, H: int = 32, Hkv: int = 8,
                      d: int = 128, chunk: int = 4096, blk: int = 128,
                      density: float = 0.1) -> BlockSparseCase:
    """Last M positions of an Nctx context attend causally over 128-token blocks.

    Each (head, query block, earlier key block) is kept with probability
    `density`; the diagonal block is always kept and later blocks never are.
    """
    W = 5
    q_pos0 = Nctx - M
    QB = -(-M // blk)
    KB = -(-Nctx // blk)
    u = _rng(W, "mask", seed).random((H, QB, KB))
    mask = (u < density).astype(np.uint8)
    for qb in range(QB):
        gq = (q_pos0 // blk) + qb
        mask[:, qb, gq] = 1
        mask[:, qb, gq + 1:] = 0
    return BlockSparseCase(
        q=round_bf16(_normal(W, "q", seed, (M, H, d))),
        k=round_bf16(_normal(W, "k", seed, (Nctx, Hkv, d))),
        v=round_bf16(_normal(W, "v", seed, (Nctx, Hkv, d))),
        mask=mask, q_pos0=q_pos0, chunk=chunk, scale=1.0 / math.sqrt(d), blk=blk)


@dataclass
class CompressCase:
    """Compressor inputs: kv / score [B, S, coff*d], ape [ratio, coff*d]."""

    kv: np.ndarray
    score: np.ndarray
    ape: np.ndarray
    ratio: int
    overlap: bool

    @property
    def d(self):
        return self.kv.shape[2] // (2 if self.overlap else 1)


def compress_case(seed: int, B: int = 8, S: int = 32768, d: int = 128, ratio: int = 4,
                  overlap: bool = True, bf16: bool = False) -> CompressCase:
    """Token projections of B sequences of S tokens for the compressor; the
    default is the prefill of eight 32K sequences at ratio 4 with overlapping
    windows (8192 compressed rows each, as in the gathered prefill cache).
    kv ~ N(0,1), score ~ 2 N(0,1) and ape ~ 0.5 N(0,1), fp32 (or bf16-rounded)."""
    W = 6
    coff = 2 if overlap else 1
    rnd = round_bf16 if bf16 else (lambda x: x)
    return CompressCase(kv=rnd(_normal(W, "kv", seed, (B, S, coff * d))),
                        score=rnd(_normal(W, "score", seed, (B, S, coff * d), std=2.0)),
                        ape=_normal(W, "ape", seed, (ratio, coff * d), std=0.5),
                        ratio=ratio, overlap=overlap)
