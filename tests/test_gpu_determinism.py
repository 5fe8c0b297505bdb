"""Repeated calls on the same inputs give bit-identical outputs.

Persistent CTAs claim work items dynamically and pass them through
multi-stage pipelines, and a decode query's list is split over the CTAs of a
cluster. Which CTA takes which item changes from call to call, but every
output element is computed by one item (or one fixed merge) in a fixed order.
A race, such as a buffer reused too early or an item claimed twice, would show
as a difference between calls, even one inside the oracle tolerance."""
import pytest
import torch

import windowed_attention_sinks_gb300 as sa
from windowed_attention_sinks_gb300 import workloads as W

from gpu_helpers import dev

pytestmark = pytest.mark.gpu

REPEATS = 12


def _all_equal(runs):
    o0, l0 = runs[0]
    for i, (o, l) in enumerate(runs[1:], 1):
        assert torch.equal(o, o0), "o differs on call %d" % i
        assert torch.equal(l, l0), "lse differs on call %d" % i


@pytest.mark.parametrize("hkv,mode", [(16, 1), (8, 2)])
def test_window_calls_repeat_bit_for_bit(hkv, mode):
    case = W.window_vision_bf16(4, hkv, num_seqs=64)
    q, k, v = (dev(x, torch.bfloat16) for x in (case.q, case.k, case.v))
    cu = dev(case.cu_seqlens, torch.int32)
    s = dev(case.sinks, torch.float32)
    runs = []
    for _ in range(REPEATS):
        o, lse = sa.window_fwd(q, k, v, cu, case.max_seqlen, case.window_left,
                               case.window_right, False, s, mode, case.scale)
        runs.append((o.clone(), lse.clone()))
    sa.check_device()
    _all_equal(runs)


@pytest.mark.parametrize("kind", ["decode_cluster", "decode_split", "prefill"])
def test_gathered_calls_repeat_bit_for_bit(kind):
    # 64 queries: one launch of the cluster kernel; 100 queries: the
    # persistent kernel with split lists and the merge; 1024 queries: the
    # persistent kernel, one CTA slot per list
    if kind == "prefill":
        case = W.sparse_prefill_bf16(6, M=1024)
    else:
        case = W.sparse_decode_bf16(6, B=64 if kind == "decode_cluster" else 100)
    q, kv = dev(case.q, torch.bfloat16), dev(case.kv, torch.bfloat16)
    idx = dev(case.idx, torch.int32)
    s = dev(case.sinks, torch.float32)
    nb = sa.sparse_workspace_bytes(case.B, case.M, case.H, case.d, case.K)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    runs = []
    for _ in range(REPEATS):
        o, lse = sa.sparse_fwd(q, kv, idx, s, case.sink_mode, case.scale, workspace=ws)
        runs.append((o.clone(), lse.clone()))
    sa.check_device()
    _all_equal(runs)


def test_block_chunks_and_merge_repeat_bit_for_bit():
    case = W.block_sparse_bf16(3, Nctx=8192, M=1024, chunk=1024, density=0.3)
    q, k, v = (dev(x, torch.bfloat16) for x in (case.q, case.k, case.v))
    mask = dev(case.mask, torch.uint8)
    C = len(case.chunks)
    chunk = case.chunks[0][1] - case.chunks[0][0]
    op = torch.empty((C, case.M, case.H, case.d), dtype=torch.float32, device="cuda")
    lp = torch.empty((C, case.M, case.H), dtype=torch.float32, device="cuda")
    runs = []
    for _ in range(REPEATS):
        sa.block_sparse_chunks_fwd(q, k, v, mask, case.q_pos0, 0, case.k.shape[0], chunk,
                                   bool(case.causal), case.scale, o_parts=op, lse_parts=lp)
        o, lse = sa.merge_lse(op.view(C, case.M * case.H, case.d), lp.view(C, case.M * case.H),
                              case.H, out_dtype=torch.bfloat16)
        runs.append((o.clone(), lse.clone()))
    sa.check_device()
    _all_equal(runs)
