"""GPU parity: gathered attention over one shared KV head vs the fp64 oracle.

Workloads follow the DeepSeek-V4 CSA/HCA walkthrough: a [window ring |
compressed] cache, topk_idxs = window indices then compressed indices, -1 for
invalid entries, null-logit sinks (sections 2.3, 3.3, 4.1-4.4)."""
import numpy as np
import pytest
import torch

import oracle
import windowed_attention_sinks_gb300 as sa
from windowed_attention_sinks_gb300 import workloads as W

from gpu_helpers import TOL_BF16_O, TOL_F32_O, compare, dev, tdtype

pytestmark = pytest.mark.gpu


def run_sparse(case, mode=None, workspace=True, sinks=None):
    mode = case.sink_mode if mode is None else mode
    dt = tdtype(case.dtype)
    q, kv = dev(case.q, dt), dev(case.kv, dt)
    idx = dev(case.idx, torch.int32)
    s = dev(case.sinks if sinks is None else sinks, torch.float32)
    ws = None
    if workspace:
        nb = sa.sparse_workspace_bytes(case.B, case.M, case.H, case.d, case.K)
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    o, lse = sa.sparse_fwd(q, kv, idx, s if mode else None, mode, case.scale, workspace=ws)
    sa.check_device()
    return o, lse


def oracle_sparse(case, mode=None, rows=None, sinks=None):
    mode = case.sink_mode if mode is None else mode
    return oracle.sparse(case.q, case.kv, case.idx, case.sinks if sinks is None else sinks, mode,
                         case.scale, rows=rows)


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("workspace", [True, False])
def test_decode_full_size(seed, workspace):
    """Sparse decode at full size: 64 requests, 640 entries each (64 of them -1)."""
    case = W.sparse_decode_bf16(seed)
    o, lse = run_sparse(case, workspace=workspace)
    ro, rl = oracle_sparse(case)
    compare(o, lse, ro, rl, TOL_BF16_O, what="decode seed=%d ws=%s" % (seed, workspace))


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_decode_sink_modes(mode):
    case = W.sparse_decode_bf16(3, B=8)
    # make idx 0 appear so the key-0 bias has something to act on
    case.idx[:, 0, 5] = 0
    o, lse = run_sparse(case, mode)
    ro, rl = oracle_sparse(case, mode)
    compare(o, lse, ro, rl, TOL_BF16_O, what="decode mode=%d" % mode)


def test_prefill_small():
    """Causal prefill index lists (window ring + compressed <= pos/4 + padding)."""
    case = W.sparse_prefill_bf16(0, M=384)
    o, lse = run_sparse(case)
    ro, rl = oracle_sparse(case)
    compare(o, lse, ro, rl, TOL_BF16_O, what="prefill small")


def test_prefill_full_size_sampled():
    case = W.sparse_prefill_bf16(0)
    o, lse = run_sparse(case)
    rng = np.random.default_rng(2)
    R = case.B * case.M * case.H
    rows = np.unique(np.concatenate([rng.integers(0, R, 2000), np.arange(64),
                                     np.arange(R - 64, R), 7680 * 32 + np.arange(64)]))
    ro, rl = oracle_sparse(case, rows=rows)
    sel = torch.from_numpy(rows).cuda()
    compare(o.reshape(R, -1)[sel], lse.reshape(-1)[sel], ro, rl, TOL_BF16_O,
            what="prefill full sampled")


@pytest.mark.parametrize("K", [0, 1, 17, 128, 129, 640, 2048])
def test_ragged_lists_and_all_invalid(K):
    rng = np.random.default_rng(K)
    B, M, H, d, N = 3, 5, 32, 128, 1000
    q = W.round_bf16(rng.standard_normal((B, M, H, d)).astype(np.float32))
    kv = W.round_bf16(rng.standard_normal((B, N, d)).astype(np.float32))
    idx = rng.integers(0, N, size=(B, M, K)).astype(np.int32)
    if K:
        idx[rng.random((B, M, K)) < 0.4] = -1
        idx[1, 2, :] = -1  # a row that sees nothing
    case = W.SparseCase(q=q, kv=kv, idx=idx, sinks=rng.standard_normal(H).astype(np.float32),
                        scale=d ** -0.5)
    for mode in (0, 2):
        for ws in (True, False):
            o, lse = run_sparse(case, mode, workspace=ws)
            ro, rl = oracle_sparse(case, mode)
            compare(o, lse, ro, rl, TOL_BF16_O, what="K=%d mode=%d ws=%s" % (K, mode, ws))


def test_duplicates_count_twice():
    rng = np.random.default_rng(7)
    B, M, H, d, N, K = 1, 2, 32, 128, 50, 300
    q = W.round_bf16(rng.standard_normal((B, M, H, d)).astype(np.float32))
    kv = W.round_bf16(rng.standard_normal((B, N, d)).astype(np.float32))
    idx = rng.integers(0, 5, size=(B, M, K)).astype(np.int32)
    case = W.SparseCase(q=q, kv=kv, idx=idx, sinks=np.zeros(H, np.float32), scale=d ** -0.5,
                        sink_mode=0)
    o, lse = run_sparse(case)
    ro, rl = oracle_sparse(case)
    compare(o, lse, ro, rl, TOL_BF16_O)


def test_fp32_sparse_d64():
    rng = np.random.default_rng(8)
    B, M, H, d, N, K = 2, 3, 8, 64, 200, 150
    q = rng.standard_normal((B, M, H, d)).astype(np.float32)
    kv = rng.standard_normal((B, N, d)).astype(np.float32)
    idx = rng.integers(-1, N, size=(B, M, K)).astype(np.int32)
    case = W.SparseCase(q=q, kv=kv, idx=idx, sinks=rng.standard_normal(H).astype(np.float32),
                        scale=d ** -0.5, dtype="f32")
    o, lse = run_sparse(case)
    ro, rl = oracle_sparse(case)
    compare(o, lse, ro, rl, TOL_F32_O)


def test_gather_decisions_bit_exact():
    """q = 0, one-hot rows: the support of o is exactly the set of valid entries."""
    B, M, H, d, N, K = 2, 3, 32, 128, 128, 200
    rng = np.random.default_rng(9)
    q = np.zeros((B, M, H, d), np.float32)
    kv = np.zeros((B, N, d), np.float32)
    for n in range(N):
        kv[:, n, n % d] = 1.0
    idx = rng.integers(-1, N, size=(B, M, K)).astype(np.int32)
    case = W.SparseCase(q=q, kv=kv, idx=idx, sinks=rng.standard_normal(H).astype(np.float32),
                        scale=d ** -0.5)
    for mode in (0, 1, 2):
        o, lse = run_sparse(case, mode)
        ro, rl = oracle_sparse(case, mode)
        got = o.float().cpu().numpy().reshape(ro.shape) != 0
        assert np.array_equal(got, ro != 0)
        compare(o, lse, ro, rl, TOL_BF16_O)


def test_out_of_range_index_is_reported_not_faulted():
    B, M, H, d, N, K = 1, 1, 32, 128, 10, 16
    q = torch.zeros((B, M, H, d), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((B, N, d), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((B, M, K), dtype=torch.int32, device="cuda")
    idx[0, 0, 3] = N + 5
    idx[0, 0, 4] = -7
    sa.sparse_fwd(q, kv, idx)
    with pytest.raises(sa.SattnError) as e:
        sa.check_device()
    assert e.value.code == 4


def _decode_inputs(case):
    q, kv = dev(case.q, torch.bfloat16), dev(case.kv, torch.bfloat16)
    idx = dev(case.idx, torch.int32)
    s = dev(case.sinks, torch.float32)
    nb = sa.sparse_workspace_bytes(case.B, case.M, case.H, case.d, case.K)
    return q, kv, idx, s, nb


def test_split_merge_reuses_a_workspace_and_ignores_its_contents():
    # split lists: a workspace full of random bytes, then the same workspace
    # again and again, all give the oracle's result and the same bits. 100
    # queries of 640 entries are too many for one cluster per query on 152
    # SMs (a CTA holds at most 384 entries), so the persistent kernel splits
    # the lists through the workspace
    case = W.sparse_decode_bf16(11, B=100)
    q, kv, idx, s, nb = _decode_inputs(case)
    ws = torch.randint(0, 256, (nb,), dtype=torch.uint8, device="cuda")
    ro, rl = oracle_sparse(case)
    first = None
    for it in range(4):
        o, lse = sa.sparse_fwd(q, kv, idx, s, case.sink_mode, case.scale, workspace=ws)
        sa.check_device()
        compare(o, lse, ro, rl, TOL_BF16_O, what="reuse %d" % it)
        if first is None:
            first = (o.clone(), lse.clone())
        else:
            assert torch.equal(o, first[0]) and torch.equal(lse, first[1])


def test_split_merge_under_graph_replay():
    # a captured split call (the gathered kernel and the merge) gives the
    # oracle's result on every replay (100 queries: the split path, as above)
    case = W.sparse_decode_bf16(12, B=100)
    q, kv, idx, s, nb = _decode_inputs(case)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    o = torch.empty((case.B, case.M, case.H, case.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((case.B, case.M, case.H), dtype=torch.float32, device="cuda")
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        sa.sparse_fwd(q, kv, idx, s, case.sink_mode, case.scale, o=o, lse=lse, workspace=ws,
                      stream=st)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        sa.sparse_fwd(q, kv, idx, s, case.sink_mode, case.scale, o=o, lse=lse, workspace=ws,
                      stream=st)
    ro, rl = oracle_sparse(case)
    for it in range(3):
        o.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        sa.check_device()
        compare(o, lse, ro, rl, TOL_BF16_O, what="replay %d" % it)


@pytest.mark.parametrize("B,K", [(1, 3072), (2, 1), (3, 100), (5, 383), (8, 0), (19, 700),
                                 (38, 384), (64, 640), (76, 768), (77, 384)])
def test_decode_clusters(B, K):
    """Few queries: each list is cut into C = 1..8 segments, one CTA of a
    cluster each, merged through distributed shared memory. Lists of every
    length the kernel takes (up to 3 tiles per CTA), -1 entries, empty
    segments (K < C), a list with nothing valid, all three sink modes."""
    rng = np.random.default_rng(B * 1000 + K)
    M, H, d, N = 1, 32, 128, 5000
    q = W.round_bf16(rng.standard_normal((B, M, H, d)).astype(np.float32))
    kv = W.round_bf16(rng.standard_normal((B, N, d)).astype(np.float32))
    idx = rng.integers(0, N, size=(B, M, K)).astype(np.int32)
    if K:
        idx[rng.random((B, M, K)) < 0.15] = -1
        idx[0, 0, : min(K, 7)] = 0  # key 0 for the key-0 bias (seven times)
        if B > 1:
            idx[B - 1, 0, :] = -1  # a query that sees nothing
    case = W.SparseCase(q=q, kv=kv, idx=idx, sinks=rng.standard_normal(H).astype(np.float32),
                        scale=d ** -0.5)
    for mode in (0, 1, 2):
        o, lse = run_sparse(case, mode, workspace=False)
        ro, rl = oracle_sparse(case, mode)
        compare(o, lse, ro, rl, TOL_BF16_O, what="B=%d K=%d mode=%d" % (B, K, mode))


def test_decode_gather_decisions_bit_exact():
    """The cluster path's visible sets: q = 0, row n = e_(n mod 128); with
    |S| <= 128 per query the support of o recovers every valid entry."""
    B, M, H, d, N, K = 4, 1, 32, 128, 128, 700
    rng = np.random.default_rng(19)
    q = np.zeros((B, M, H, d), np.float32)
    kv = np.zeros((B, N, d), np.float32)
    for n in range(N):
        kv[:, n, n % d] = 1.0
    idx = np.full((B, M, K), -1, np.int32)
    for b in range(B):  # a handful of valid entries scattered over the segments
        pos = rng.choice(K, size=40, replace=False)
        idx[b, 0, pos] = rng.integers(0, N, size=40)
    case = W.SparseCase(q=q, kv=kv, idx=idx, sinks=rng.standard_normal(H).astype(np.float32),
                        scale=d ** -0.5)
    for mode in (0, 1, 2):
        o, lse = run_sparse(case, mode, workspace=False)
        ro, rl = oracle_sparse(case, mode)
        got = o.float().cpu().numpy().reshape(ro.shape) != 0
        assert np.array_equal(got, ro != 0), mode
        compare(o, lse, ro, rl, TOL_BF16_O)
