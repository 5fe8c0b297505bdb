"""GPU parity: sliding-window varlen attention with sinks vs the fp64 oracle.

Workloads follow the vLLM PR #49815 report (5/37-token sequences, window 8,
key-0 sinks; vision-encoder window attention) and its named risk cases
(window smaller than a key tile, tiles spanning sequence boundaries)."""
import math

import numpy as np
import pytest
import torch

import oracle
import windowed_attention_sinks_gb300 as sa
from windowed_attention_sinks_gb300 import workloads as W

from gpu_helpers import TOL_BF16_O, TOL_F32_O, compare, dev, tdtype

pytestmark = pytest.mark.gpu


def run_window(case, mode, sinks=None):
    dt = tdtype(case.dtype)
    q, k, v = dev(case.q, dt), dev(case.k, dt), dev(case.v, dt)
    cu = dev(case.cu_seqlens, torch.int32)
    s = dev(case.sinks if sinks is None else sinks, torch.float32)
    o, lse = sa.window_fwd(q, k, v, cu, case.max_seqlen, case.window_left, case.window_right,
                           case.causal, s if mode else None, mode, case.scale)
    sa.check_device()
    return o, lse


def oracle_window(case, mode, rows=None, sinks=None):
    return oracle.window(case.q, case.k, case.v, case.cu_seqlens, case.H, case.Hkv, case.d,
                         case.window_left, case.window_right, case.causal,
                         case.sinks if sinks is None else sinks, mode, case.scale, rows=rows)


@pytest.mark.parametrize("hkv", [4, 2])
@pytest.mark.parametrize("mode", [1, 2, 0])
def test_tiny_fp32(hkv, mode):
    case = W.window_tiny_f32(0, hkv)
    o, lse = run_window(case, mode)
    ro, rl = oracle_window(case, mode)
    compare(o, lse, ro, rl, TOL_F32_O, what="tiny fp32 hkv=%d mode=%d" % (hkv, mode))


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("hkv", [16, 8])
@pytest.mark.parametrize("mode", [1, 2])
def test_vision_bf16_small(seed, hkv, mode):
    """A handful of sequences: several 128-row tiles per sequence and ragged tails."""
    case = W.window_vision_bf16(seed, hkv, num_seqs=6)
    o, lse = run_window(case, mode)
    ro, rl = oracle_window(case, mode)
    compare(o, lse, ro, rl, TOL_BF16_O, what="vision bf16 hkv=%d mode=%d" % (hkv, mode))


def _custom_case(lens, H, Hkv, d, wl, wr, causal, dtype, seed=0, std=1.0):
    rng = np.random.default_rng(seed)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    T = int(cu[-1])
    q = (rng.standard_normal((T, H, d)) * std).astype(np.float32)
    k = (rng.standard_normal((T, Hkv, d)) * std).astype(np.float32)
    v = rng.standard_normal((T, Hkv, d)).astype(np.float32)
    if dtype == "bf16":
        q, k, v = W.round_bf16(q), W.round_bf16(k), W.round_bf16(v)
    return W.WindowCase(q=q, k=k, v=v, sinks=rng.standard_normal(H).astype(np.float32),
                        cu_seqlens=cu, H=H, Hkv=Hkv, d=d, window_left=wl, window_right=wr,
                        causal=causal, scale=1.0 / math.sqrt(d), dtype=dtype)


EDGE_LENS = [1, 127, 128, 129, 5, 300, 2, 255, 256, 257]


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64), ("bf16", 64), ("f32", 128)])
@pytest.mark.parametrize("w", [0, 1, 7, 8, 127, 128, 129, 1000])
def test_window_edges(dtype, d, w):
    case = _custom_case(EDGE_LENS, 4, 2, d, w, w, 0, dtype, seed=w)
    tol = TOL_BF16_O if dtype == "bf16" else TOL_F32_O
    for mode in (0, 1, 2):
        o, lse = run_window(case, mode)
        ro, rl = oracle_window(case, mode)
        compare(o, lse, ro, rl, tol, what="edge w=%d mode=%d %s d=%d" % (w, mode, dtype, d))


@pytest.mark.parametrize("wl,wr,causal", [(-1, -1, 1), (64, 0, 1), (5, 200, 0), (-1, 3, 0),
                                          (130, -1, 0), (300, 300, 1)])
def test_window_asymmetric_and_causal(wl, wr, causal):
    case = _custom_case(EDGE_LENS, 8, 8, 128, wl, wr, causal, "bf16", seed=3)
    for mode in (1, 2):
        o, lse = run_window(case, mode)
        ro, rl = oracle_window(case, mode)
        compare(o, lse, ro, rl, TOL_BF16_O, what="wl=%d wr=%d causal=%d" % (wl, wr, causal))


@pytest.mark.parametrize("H,Hkv", [(8, 2), (16, 2), (16, 1), (12, 2), (12, 4), (6, 2), (1, 1),
                                   (32, 4)])
def test_query_head_packing(H, Hkv):
    """The query heads of a KV group share a tile (two, four or eight of them:
    the largest power of two dividing H / Hkv); groups of 3 run one head per
    tile, groups of 6 two. Ragged sequences put every packed layout across
    sequence ends and partial warp tiles."""
    for wl, wr, causal in [(128, 128, 0), (37, 5, 1), (-1, -1, 1), (0, 300, 0)]:
        case = _custom_case(EDGE_LENS, H, Hkv, 128, wl, wr, causal, "bf16", seed=H * 10 + Hkv)
        for mode in (1, 2):
            o, lse = run_window(case, mode)
            ro, rl = oracle_window(case, mode)
            compare(o, lse, ro, rl, TOL_BF16_O,
                    what="H=%d Hkv=%d wl=%d wr=%d causal=%d mode=%d" % (H, Hkv, wl, wr, causal, mode))


@pytest.mark.parametrize("H,Hkv", [(4, 2), (8, 2), (8, 1)])
def test_long_sequence_full_causal(H, Hkv):
    """One long sequence with unbounded causal attention: items of about 70 key
    tiles, the running max moving many times per row, and a second short
    sequence after it in the same batch."""
    case = _custom_case([4500, 77], H, Hkv, 128, -1, -1, 1, "bf16", seed=H + 7 * Hkv, std=1.5)
    for mode in (1, 2):
        o, lse = run_window(case, mode)
        ro, rl = oracle_window(case, mode)
        compare(o, lse, ro, rl, TOL_BF16_O, tol_lse=2e-3,
                what="long causal H=%d Hkv=%d mode=%d" % (H, Hkv, mode))


def test_large_logits_rescale():
    """Scores spread over a wide range force the running max to move by large
    steps inside a row (exercises the rescaling of the accumulator)."""
    case = _custom_case([700, 129, 1000], 4, 4, 128, 128, 128, 0, "bf16", seed=5, std=3.0)
    ramp = np.linspace(0.2, 4.0, case.q.shape[0]).astype(np.float32)[:, None, None]
    case.q = W.round_bf16(case.q * ramp)
    for mode in (0, 1, 2):
        o, lse = run_window(case, mode)
        ro, rl = oracle_window(case, mode)
        compare(o, lse, ro, rl, TOL_BF16_O, tol_lse=2e-3, what="large logits mode=%d" % mode)


@pytest.mark.parametrize("dtype,d,H,Hkv", [("bf16", 128, 4, 2), ("f32", 64, 4, 2),
                                           ("bf16", 128, 8, 1), ("bf16", 128, 8, 2)])
def test_mask_decisions_bit_exact(dtype, d, H, Hkv):
    """q = 0 and one-hot values: the support of each output row is exactly the
    set of visible keys, so the zero pattern must equal the oracle's bit for bit
    (bf16 d = 128 runs the tensor-core kernel with 2, 8 and 4 query heads per tile)."""
    lens = [1, 5, 37, 128, 129, 200]
    case = _custom_case(lens, H, Hkv, d, 8, 8, 0, dtype)
    case.q[:] = 0
    case.v[:] = 0
    for s in range(len(lens)):
        for j in range(lens[s]):
            case.v[case.cu_seqlens[s] + j, :, j % d] = 1.0
    for wl, wr, causal in [(8, 8, 0), (0, 0, 0), (3, 20, 1), (130, 130, 0)]:
        case.window_left, case.window_right, case.causal = wl, wr, causal
        for mode in (0, 1, 2):
            o, lse = run_window(case, mode)
            ro, rl = oracle_window(case, mode)
            got = o.float().cpu().numpy().reshape(ro.shape) != 0
            assert np.array_equal(got, ro != 0), "support differs wl=%d wr=%d" % (wl, wr)
            compare(o, lse, ro, rl, TOL_BF16_O if dtype == "bf16" else TOL_F32_O)


def test_misaligned_tensors_are_refused():
    """The tensor-core path reads q, k, v and writes o through TMA, which needs
    16-byte aligned bases: a misaligned one is an invalid argument, reported
    before any launch."""
    case = _custom_case([40, 7], 4, 2, 128, 8, 8, 0, "bf16")
    q, k, v = dev(case.q, torch.bfloat16), dev(case.k, torch.bfloat16), dev(case.v, torch.bfloat16)
    cu = dev(case.cu_seqlens, torch.int32)
    buf = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device="cuda")
    o_bad = buf[1:1 + q.numel()].view(q.shape)  # 2 bytes past a 16-byte boundary
    q_bad = buf[1:1 + q.numel()].view(q.shape).copy_(q)
    for kw, args in (({"o": o_bad}, (q, k, v)), ({}, (q_bad, k, v))):
        with pytest.raises(sa.SattnError) as e:
            sa.window_fwd(*args, cu, case.max_seqlen, 8, 8, False, None, 0, case.scale, **kw)
        assert e.value.code == 1
    o, lse = sa.window_fwd(q, k, v, cu, case.max_seqlen, 8, 8, False, None, 0, case.scale)
    sa.check_device()
    ro, rl = oracle_window(case, 0)
    compare(o, lse, ro, rl, TOL_BF16_O, what="after refused calls")


def test_sink_reductions_on_gpu():
    """key-0 sink 0 and null sink -inf reproduce the no-sink output on the GPU."""
    case = W.window_vision_bf16(2, 8, num_seqs=3)
    o0, l0 = run_window(case, 0)
    ok, lk = run_window(case, 1, sinks=np.zeros(case.H, np.float32))
    on, ln_ = run_window(case, 2, sinks=np.full(case.H, -np.inf, np.float32))
    assert torch.equal(o0, ok) and torch.equal(l0, lk)
    assert torch.equal(o0, on) and torch.equal(l0, ln_)


def test_vision_bf16_full_size_sampled():
    """The full 256-sequence vision workload, checked on sampled rows."""
    for hkv, mode in ((16, 1), (8, 2)):
        case = W.window_vision_bf16(0, hkv, sink_mode=mode)
        o, lse = run_window(case, mode)
        rng = np.random.default_rng(1)
        T, H = case.T, case.H
        rows = np.concatenate([rng.integers(0, T * H, 3000),
                               np.arange(H), np.arange(T * H - H, T * H)])
        # rows at every sequence start and end
        starts = case.cu_seqlens[:-1].astype(np.int64) * H
        rows = np.unique(np.concatenate([rows, starts, starts + H * 127 + 1]))
        rows = rows[rows < T * H]
        ro, rl = oracle_window(case, mode, rows=rows)
        og = o.reshape(T * H, -1)[torch.from_numpy(rows).cuda()]
        lg = lse.reshape(-1)[torch.from_numpy(rows).cuda()]
        compare(og, lg, ro, rl, TOL_BF16_O, what="full-size hkv=%d" % hkv)


def test_invalid_cu_seqlens_is_reported_not_faulted():
    case = _custom_case([10, 20], 2, 2, 128, 4, 4, 0, "bf16")
    dt = torch.bfloat16
    q, k, v = dev(case.q, dt), dev(case.k, dt), dev(case.v, dt)
    bad = torch.tensor([0, 25, 20], dtype=torch.int32, device="cuda")  # decreasing
    sa.window_fwd(q, k, v, bad, 25, 4, 4)
    with pytest.raises(sa.SattnError) as e:
        sa.check_device()
    assert e.value.code == 4
