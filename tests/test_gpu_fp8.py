"""GPU parity of the FP8 KV layout: the quantiser bit-exact against the
oracle's, and gathered attention over an FP8 cache against the oracle run on
the dequantised rows ("DeepSeek-V4 CSA/HCA walkthrough", section 2.3 step 4
and section 5.3; the layout is e4m3 codes with one fp32 scale per row for the
first d - rd columns, the last rd columns in bf16)."""
import numpy as np
import pytest
import torch

import oracle
import windowed_attention_sinks_gb300 as sa
from windowed_attention_sinks_gb300 import workloads as W

from gpu_helpers import TOL_BF16_O, compare, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,rd", [(128, 64), (64, 32), (512, 64), (16, 8), (128, 4)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantiser_bit_exact(d, rd, dtype):
    rng = np.random.default_rng(d + rd)
    x = (rng.standard_normal((333, d)) * rng.uniform(1e-3, 50, (333, 1))).astype(np.float32)
    x[5] = 0.0          # an all-zero row: scale 1, codes 0
    x[6, : d - rd] = 0.0  # an all-zero non-RoPE part
    x[7, 3] = -0.0
    if dtype == torch.bfloat16:
        x = oracle.bf16_round(x)
    codes, rope, scale = sa.quantize_kv_fp8(dev(x, dtype), rd)
    sa.check_device()
    want_c, want_r, want_s = oracle.quantize_kv_fp8(x, rd)
    assert np.array_equal(scale.cpu().numpy(), want_s)
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert np.array_equal(rope.float().cpu().numpy(), want_r)


def _fp8_cache(case):
    # the kernel multiplies the rows as gathered: e4m3 value x scale rounded to bf16
    codes, rope, scale = oracle.quantize_kv_fp8(case.kv, 64)
    deq = oracle.bf16_round(oracle.dequantize_kv_fp8(codes, rope, scale).astype(np.float32))
    return codes, rope, scale, deq


def run_fp8(case, codes, rope, scale, mode=None, workspace=True):
    mode = case.sink_mode if mode is None else mode
    q = dev(case.q, torch.bfloat16)
    idx = dev(case.idx, torch.int32)
    s = dev(case.sinks, torch.float32)
    ws = None
    if workspace:
        nb = sa.sparse_workspace_bytes(case.B, case.M, case.H, case.d, case.K)
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    o, lse = sa.sparse_fp8_fwd(q, dev(codes, torch.uint8), dev(rope, torch.bfloat16),
                               dev(scale, torch.float32), idx, s if mode else None, mode,
                               case.scale, workspace=ws)
    sa.check_device()
    return o, lse


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("workspace", [True, False])
def test_decode_full_size(seed, workspace):
    case = W.sparse_decode_bf16(seed)
    codes, rope, scale, deq = _fp8_cache(case)
    o, lse = run_fp8(case, codes, rope, scale, workspace=workspace)
    ro, rl = oracle.sparse(case.q, deq, case.idx, case.sinks, case.sink_mode, case.scale)
    compare(o, lse, ro, rl, TOL_BF16_O, what="fp8 decode seed=%d ws=%s" % (seed, workspace))


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_decode_sink_modes(mode):
    case = W.sparse_decode_bf16(3, B=8)
    case.idx[:, 0, 5] = 0  # row 0 listed: the key-0 bias has something to act on
    codes, rope, scale, deq = _fp8_cache(case)
    o, lse = run_fp8(case, codes, rope, scale, mode)
    ro, rl = oracle.sparse(case.q, deq, case.idx, case.sinks, mode, case.scale)
    compare(o, lse, ro, rl, TOL_BF16_O, what="fp8 decode mode=%d" % mode)


def test_wide_scales_and_invalid_entries():
    # row magnitudes spread over three decades (each row's scale differs) and
    # lists with runs of -1; values stay of order one so that the absolute
    # tolerance keeps its meaning
    case = W.sparse_decode_bf16(4, B=4)
    rng = np.random.default_rng(4)
    mag = 10.0 ** rng.uniform(-3, 0, case.kv.shape[:2] + (1,))
    case.kv[...] = oracle.bf16_round((case.kv * mag).astype(np.float32))
    case.idx[:, :, 100:300] = -1
    codes, rope, scale, deq = _fp8_cache(case)
    o, lse = run_fp8(case, codes, rope, scale)
    ro, rl = oracle.sparse(case.q, deq, case.idx, case.sinks, case.sink_mode, case.scale)
    compare(o, lse, ro, rl, TOL_BF16_O, what="fp8 wide scales")


def test_prefill_sampled():
    case = W.sparse_prefill_bf16(0, M=2048)
    codes, rope, scale, deq = _fp8_cache(case)
    o, lse = run_fp8(case, codes, rope, scale)
    rng = np.random.default_rng(5)
    R = case.B * case.M * case.H
    rows = np.unique(np.concatenate([rng.integers(0, R, 1500), np.arange(64),
                                     np.arange(R - 64, R)]))
    ro, rl = oracle.sparse(case.q, deq, case.idx, case.sinks, case.sink_mode, case.scale,
                           rows=rows)
    sel = torch.from_numpy(rows).cuda()
    compare(o.reshape(R, -1)[sel], lse.reshape(-1)[sel], ro, rl, TOL_BF16_O, what="fp8 prefill")


def test_matches_bf16_path_on_exact_rows():
    # rows whose non-RoPE part is e4m3 values / 64 with a maximum of exactly
    # 448 / 64 (so the scale is 2^-6) dequantise to themselves: the FP8 path
    # must then reproduce the bf16 path's result bit for bit. 100 queries of
    # 640 entries: the bf16 call then takes the same persistent kernel (and
    # the same list splits) as the FP8 call, not the cluster kernel that
    # serves fewer queries, so the two sum in the same order
    case = W.sparse_decode_bf16(6, B=100)
    rng = np.random.default_rng(6)
    vals = oracle.e4m3_decode(rng.integers(0, 0x7F, case.kv.shape[:2] + (64,)).astype(np.uint8))
    sign = np.where(rng.random(vals.shape) < 0.5, -1.0, 1.0)
    case.kv[..., :64] = (vals * sign / 64.0).astype(np.float32)
    case.kv[..., 0] = 7.0
    codes, rope, scale, deq = _fp8_cache(case)
    assert np.array_equal(deq, case.kv)
    o8, l8 = run_fp8(case, codes, rope, scale)
    q, kv, idx = dev(case.q, torch.bfloat16), dev(case.kv, torch.bfloat16), dev(case.idx, torch.int32)
    nb = sa.sparse_workspace_bytes(case.B, case.M, case.H, case.d, case.K)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    o16, l16 = sa.sparse_fwd(q, kv, idx, dev(case.sinks, torch.float32), case.sink_mode,
                             case.scale, workspace=ws)
    sa.check_device()
    assert torch.equal(o8, o16) and torch.equal(l8, l16)


def test_cluster_path_matches_bf16_on_exact_rows():
    # 16 queries take the cluster kernel with either cache; on rows that
    # dequantise to themselves the two calls sum the same values in the same
    # order, so the results agree bit for bit
    case = W.sparse_decode_bf16(8, B=16)
    rng = np.random.default_rng(8)
    vals = oracle.e4m3_decode(rng.integers(0, 0x7F, case.kv.shape[:2] + (64,)).astype(np.uint8))
    sign = np.where(rng.random(vals.shape) < 0.5, -1.0, 1.0)
    case.kv[..., :64] = (vals * sign / 64.0).astype(np.float32)
    case.kv[..., 0] = 7.0
    codes, rope, scale, deq = _fp8_cache(case)
    assert np.array_equal(deq, case.kv)
    for mode in (0, 1, 2):
        o8, l8 = run_fp8(case, codes, rope, scale, mode=mode, workspace=False)
        q, kv = dev(case.q, torch.bfloat16), dev(case.kv, torch.bfloat16)
        idx = dev(case.idx, torch.int32)
        s16 = dev(case.sinks, torch.float32) if mode else None
        o16, l16 = sa.sparse_fwd(q, kv, idx, s16, mode, case.scale)
        sa.check_device()
        assert torch.equal(o8, o16) and torch.equal(l8, l16), mode
        ro, rl = oracle.sparse(case.q, deq, case.idx, case.sinks, mode, case.scale)
        compare(o8, l8, ro, rl, TOL_BF16_O, what="fp8 cluster mode=%d" % mode)


def test_lists_of_only_invalid_entries():
    # every entry -1: o = 0 and lse = the sink (null logit) for every head
    case = W.sparse_decode_bf16(7, B=3)
    case.idx[...] = -1
    codes, rope, scale, deq = _fp8_cache(case)
    o, lse = run_fp8(case, codes, rope, scale)
    assert torch.all(o == 0)
    np.testing.assert_allclose(lse.cpu().numpy(),
                               np.broadcast_to(case.sinks, lse.shape), rtol=0, atol=1e-5)
