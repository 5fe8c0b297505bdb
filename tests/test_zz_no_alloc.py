"""GPU check of sattn_sparse_fwd_static_scratch.

This entry point is for callers that cannot allocate device memory (a plug-in
whose host application owns all device memory, a loop that forbids
cudaMalloc/cudaFree after start-up, or C code handed only pointers and a
stream). It keeps the partial results of split index lists in a scratch array
built into the library instead of a caller workspace. Its output must match
sattn_sparse_fwd with a caller-allocated workspace, on two calls in a row
(the second call sees the first call's leftovers in the shared array), and
requests larger than the built-in array must be refused.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import windowed_attention_sinks_gb300 as sa
from windowed_attention_sinks_gb300 import workloads as W

from gpu_helpers import TOL_BF16_O, TOL_F32_O, compare, dev

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 8 << 20  # SATTN_SPARSE_STATIC_SCRATCH_BYTES in include/sattn.h


def _entry():
    f = sa.lib().sattn_sparse_fwd_static_scratch
    P = ctypes.c_void_p
    i32 = ctypes.c_int32
    f.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_float, P, P, i32, i32, i32, i32, i32, i32,
                  ctypes.c_int, P]
    f.restype = ctypes.c_int
    return f


def _tensors(case):
    q, kv = dev(case.q, torch.bfloat16), dev(case.kv, torch.bfloat16)
    idx = dev(case.idx, torch.int32)
    sinks = dev(case.sinks, torch.float32)
    return q, kv, idx, sinks


def _static_call(case, q, kv, idx, sinks):
    o = torch.empty_like(q)
    lse = torch.empty((case.B, case.M, case.H), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = _entry()(q.data_ptr(), kv.data_ptr(), idx.data_ptr(), sinks.data_ptr(), case.sink_mode,
                  case.scale, o.data_ptr(), lse.data_ptr(), case.B, case.M, case.H, case.d, case.N,
                  case.K, sa.BF16, stream)
    return rc, o, lse


def test_static_scratch_matches_workspace_entry_point():
    for seed in (0, 1):  # two calls in a row, with different inputs
        # 100 requests of 512 entries: more queries than one cluster per query
        # can hold on 152 SMs, so the call splits each list across the CTAs of
        # the persistent kernel, with the partials in the scratch array
        case = W.sparse_decode_bf16(seed, B=100, n_compress_idx=384)
        need = sa.sparse_workspace_bytes(case.B, case.M, case.H, case.d, case.K)
        assert 0 < need <= STATIC_SCRATCH_BYTES
        q, kv, idx, sinks = _tensors(case)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        o_ref, lse_ref = sa.sparse_fwd(q, kv, idx, sinks, case.sink_mode, case.scale, workspace=ws)
        rc, o, lse = _static_call(case, q, kv, idx, sinks)
        assert rc == 0, "sattn_sparse_fwd_static_scratch returned %d" % rc
        sa.check_device()
        ref_o = o_ref.float().cpu().numpy().reshape(-1, case.d).astype(np.float64)
        ref_l = lse_ref.float().cpu().numpy().reshape(-1).astype(np.float64)
        compare(o.reshape(-1, case.d), lse.reshape(-1), ref_o, ref_l, TOL_BF16_O,
                what="static scratch, call %d" % seed)
        # and against the oracle itself
        ro, rl = oracle.sparse(case.q, case.kv, case.idx, case.sinks, case.sink_mode, case.scale)
        compare(o, lse, ro, rl, TOL_BF16_O, what="static scratch vs oracle, call %d" % seed)


def test_static_scratch_takes_shapes_that_need_no_scratch():
    # fp32 runs on the SIMT path, which never splits lists: a shape whose
    # tensor-core split would need more than the built-in array is accepted
    B, M, H, d, N, K = 64, 1, 64, 128, 300, 4096
    assert sa.sparse_workspace_bytes(B, M, H, d, K) > STATIC_SCRATCH_BYTES
    rng = np.random.default_rng(5)
    case = W.SparseCase(q=rng.standard_normal((B, M, H, d)).astype(np.float32),
                        kv=rng.standard_normal((B, N, d)).astype(np.float32),
                        idx=rng.integers(-1, N, size=(B, M, K)).astype(np.int32),
                        sinks=rng.standard_normal(H).astype(np.float32), scale=d ** -0.5,
                        sink_mode=2, dtype="f32")
    q, kv = dev(case.q, torch.float32), dev(case.kv, torch.float32)
    idx, sinks = dev(case.idx, torch.int32), dev(case.sinks, torch.float32)
    o = torch.empty_like(q)
    lse = torch.empty((B, M, H), dtype=torch.float32, device="cuda")
    rc = _entry()(q.data_ptr(), kv.data_ptr(), idx.data_ptr(), sinks.data_ptr(), 2, case.scale,
                  o.data_ptr(), lse.data_ptr(), B, M, H, d, N, K, sa.F32,
                  torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    sa.check_device()
    rows = np.arange(0, B * M * H, 37)
    ro, rl = oracle.sparse(case.q, case.kv, case.idx, case.sinks, 2, case.scale, rows=rows)
    sel = torch.from_numpy(rows).cuda()
    compare(o.reshape(-1, d)[sel], lse.reshape(-1)[sel], ro, rl, TOL_F32_O, what="fp32 static")


def test_static_scratch_refuses_oversized_requests():
    # 64 single-token requests (32 heads, d = 128) with 4096-entry lists, split
    # eight ways on the tensor-core path, need about 8.5 MB of partials
    B, M, H, d, N, K = 64, 1, 32, 128, 16, 4096
    assert sa.sparse_workspace_bytes(B, M, H, d, K) > STATIC_SCRATCH_BYTES
    rng = np.random.default_rng(0)
    case = W.SparseCase(q=W.round_bf16(rng.standard_normal((B, M, H, d)).astype(np.float32)),
                        kv=W.round_bf16(rng.standard_normal((B, N, d)).astype(np.float32)),
                        idx=rng.integers(-1, N, size=(B, M, K)).astype(np.int32),
                        sinks=np.zeros(H, np.float32), scale=d ** -0.5)
    q, kv, idx, sinks = _tensors(case)
    rc, _, _ = _static_call(case, q, kv, idx, sinks)
    assert rc == 1  # SATTN_ERR_INVALID_ARG: nothing was launched
    sa.check_device()
