"""CUDA-graph replay of the persistent kernels: the window/block engine and the
block-selection kernel claim work items through per-launch counters, so a
captured call must give the eager call's result, bit for bit, on every
replay."""
import numpy as np
import pytest
import torch

import windowed_attention_sinks_gb300 as sa
from windowed_attention_sinks_gb300 import workloads as W

from gpu_helpers import dev

pytestmark = pytest.mark.gpu


def _replays_match(call, outs, n=3):
    """Eager result of call() into outs, then n replays of a captured call()."""
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        call(st)
    st.synchronize()
    sa.check_device()
    want = [t.clone() for t in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        call(st)
    for it in range(n):
        for t in outs:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        sa.check_device()
        for a, b in zip(outs, want):
            assert torch.equal(a, b), it


@pytest.mark.parametrize("mode", [sa.SINK_KEY0_BIAS, sa.SINK_NULL_LOGIT])
def test_window_under_graph_replay(mode):
    case = W.window_vision_bf16(3, 8, num_seqs=40)
    q, k, v = (dev(x, torch.bfloat16) for x in (case.q, case.k, case.v))
    cu = dev(case.cu_seqlens, torch.int32)
    s = dev(case.sinks, torch.float32)
    T = case.q.shape[0]
    o = torch.empty((T, case.H, case.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, case.H), dtype=torch.float32, device="cuda")

    def call(st):
        sa.window_fwd(q, k, v, cu, case.max_seqlen, case.window_left, case.window_right,
                      case.causal, s, mode, case.scale, o=o, lse=lse, stream=st)
    _replays_match(call, [o, lse])


def test_block_chunks_under_graph_replay():
    case = W.block_sparse_bf16(4, Nctx=4096, M=512, chunk=1024, density=0.3)
    q, k, v = (dev(x, torch.bfloat16) for x in (case.q, case.k, case.v))
    mask = dev(case.mask, torch.uint8)
    C = len(case.chunks)
    op = torch.empty((C, case.M, case.H, case.d), dtype=torch.float32, device="cuda")
    lp = torch.empty((C, case.M, case.H), dtype=torch.float32, device="cuda")

    def call(st):
        sa.block_sparse_chunks_fwd(q, k, v, mask, case.q_pos0, 0, case.Nctx, case.chunk, True,
                                   case.scale, o_parts=op, lse_parts=lp, stream=st)
    _replays_match(call, [op, lp])


def test_selection_under_graph_replay():
    rng = np.random.default_rng(9)
    M, Nctx, H, Hkv = 384, 3000, 8, 2
    q = dev(W.round_bf16(rng.standard_normal((M, H, 128)).astype(np.float32)), torch.bfloat16)
    k = dev(W.round_bf16(rng.standard_normal((Nctx, Hkv, 128)).astype(np.float32)),
            torch.bfloat16)
    shape = (H, -(-M // 128), -(-Nctx // 128))
    ws = torch.empty(sa.xattn_select_workspace_bytes(M, H, Nctx, 1024), dtype=torch.uint8,
                     device="cuda")
    bs = torch.empty(shape, dtype=torch.float32, device="cuda")
    mask = torch.empty(shape, dtype=torch.uint8, device="cuda")

    def call(st):
        sa.xattn_select_blocks(q, k, Nctx - M, True, 0.9, None, chunk=1024, workspace=ws,
                               block_sum=bs, mask=mask, stream=st)
    _replays_match(call, [bs, mask])


def test_window_calls_on_two_streams_at_once():
    # two different problems in flight together, each launch with its own
    # work counter: the results equal those of the calls made one at a time
    cases = [W.window_vision_bf16(5, 16, num_seqs=48), W.window_vision_bf16(6, 8, num_seqs=40)]
    ins, outs = [], []
    for case in cases:
        q, k, v = (dev(x, torch.bfloat16) for x in (case.q, case.k, case.v))
        cu = dev(case.cu_seqlens, torch.int32)
        s = dev(case.sinks, torch.float32)
        ins.append((case, q, k, v, cu, s))
        T = case.q.shape[0]
        outs.append((torch.empty((T, case.H, case.d), dtype=torch.bfloat16, device="cuda"),
                     torch.empty((T, case.H), dtype=torch.float32, device="cuda")))

    def run(i, st):
        case, q, k, v, cu, s = ins[i]
        o, lse = outs[i]
        sa.window_fwd(q, k, v, cu, case.max_seqlen, case.window_left, case.window_right,
                      case.causal, s, sa.SINK_KEY0_BIAS, case.scale, o=o, lse=lse, stream=st)
    st = [torch.cuda.Stream(), torch.cuda.Stream()]
    for i in range(2):
        run(i, st[i])
        st[i].synchronize()
    sa.check_device()
    want = [(o.clone(), lse.clone()) for o, lse in outs]
    for rep in range(3):
        for o, lse in outs:
            o.zero_()
            lse.zero_()
        torch.cuda.synchronize()
        for i in range(2):
            run(i, st[i])
        torch.cuda.synchronize()
        sa.check_device()
        for (o, lse), (wo, wl) in zip(outs, want):
            assert torch.equal(o, wo) and torch.equal(lse, wl), rep
