"""GPU parity: chunked block-sparse attention and the LSE merge vs the oracle.

Workload follows the nano-vllm XAttention page: a 32K context split into
4096-key chunks, per-chunk partial stats, merged afterwards; ~10% block
density with diagonal blocks kept, causal."""
import numpy as np
import pytest
import torch

import oracle
import windowed_attention_sinks_gb300 as sa
from windowed_attention_sinks_gb300 import workloads as W

from gpu_helpers import TOL_BF16_O, TOL_F32_O, compare, dev

pytestmark = pytest.mark.gpu


def run_chunks(case, dt=torch.bfloat16):
    q, k, v = dev(case.q, dt), dev(case.k, dt), dev(case.v, dt)
    mask = dev(case.mask, torch.uint8)
    C = len(case.chunks)
    o_parts = torch.empty((C, case.M * case.H, case.d), dtype=torch.float32, device="cuda")
    lse_parts = torch.empty((C, case.M * case.H), dtype=torch.float32, device="cuda")
    for c, (a, b) in enumerate(case.chunks):
        sa.block_sparse_fwd(q, k, v, mask, case.q_pos0, a, b, bool(case.causal), case.scale,
                            o_part=o_parts[c].view(case.M, case.H, case.d),
                            lse_part=lse_parts[c].view(case.M, case.H))
    sa.check_device()
    return o_parts, lse_parts


def test_chunks_and_merge_small():
    case = W.block_sparse_bf16(0, Nctx=2048, M=512, chunk=512, density=0.3)
    o_parts, lse_parts = run_chunks(case)
    refs = [oracle.block_sparse(case.q, case.k, case.v, case.mask, case.q_pos0, a, b, 1,
                                case.scale) for a, b in case.chunks]
    for c, (ro, rl) in enumerate(refs):
        compare(o_parts[c], lse_parts[c], ro, rl, TOL_BF16_O, what="chunk %d" % c)
    o, lse = sa.merge_lse(o_parts, lse_parts, case.H, out_dtype=torch.bfloat16)
    ro, rl = oracle.block_sparse(case.q, case.k, case.v, case.mask, case.q_pos0, 0, case.Nctx, 1,
                                 case.scale)
    compare(o, lse, ro, rl, TOL_BF16_O, what="merged")


def test_full_size_sampled():
    """32K context, 4096-query chunk at the end, 8 chunks + merge; sampled rows.
    The chunks run as the bench times them: all eight in one launch."""
    case = W.block_sparse_bf16(0)
    q, k, v = (dev(x, torch.bfloat16) for x in (case.q, case.k, case.v))
    chunk = case.chunks[0][1] - case.chunks[0][0]
    o4, l4 = sa.block_sparse_chunks_fwd(q, k, v, dev(case.mask, torch.uint8), case.q_pos0, 0,
                                        case.Nctx, chunk, True, case.scale)
    sa.check_device()
    C = len(case.chunks)
    o_parts = o4.reshape(C, case.M * case.H, case.d)
    lse_parts = l4.reshape(C, case.M * case.H)
    o, lse = sa.merge_lse(o_parts, lse_parts, case.H, out_dtype=torch.bfloat16)
    rng = np.random.default_rng(3)
    R = case.M * case.H
    rows = np.unique(np.concatenate([rng.integers(0, R, 600), np.arange(32),
                                     np.arange(R - 32, R)]))
    ro, rl = oracle.block_sparse(case.q, case.k, case.v, case.mask, case.q_pos0, 0, case.Nctx, 1,
                                 case.scale, rows=rows)
    sel = torch.from_numpy(rows).cuda()
    compare(o.reshape(R, -1)[sel], lse.reshape(-1)[sel], ro, rl, TOL_BF16_O,
            what="full-size merged")
    # one chunk's partials too
    c = 6
    a, b = case.chunks[c]
    ro, rl = oracle.block_sparse(case.q, case.k, case.v, case.mask, case.q_pos0, a, b, 1,
                                 case.scale, rows=rows)
    compare(o_parts[c][sel], lse_parts[c][sel], ro, rl, TOL_BF16_O, what="full-size chunk")


@pytest.mark.parametrize("M,q_pos0,Nctx", [(1, 0, 1), (130, 126, 300), (257, 1000, 1300),
                                           (128, 0, 128)])
def test_ragged_shapes(M, q_pos0, Nctx):
    rng = np.random.default_rng(M)
    H, Hkv, d = 4, 2, 128
    q = W.round_bf16(rng.standard_normal((M, H, d)).astype(np.float32))
    k = W.round_bf16(rng.standard_normal((Nctx, Hkv, d)).astype(np.float32))
    v = W.round_bf16(rng.standard_normal((Nctx, Hkv, d)).astype(np.float32))
    QB, KB = -(-M // 128), -(-Nctx // 128)
    mask = (rng.random((H, QB, KB)) < 0.6).astype(np.uint8)
    case = W.BlockSparseCase(q=q, k=k, v=v, mask=mask, q_pos0=q_pos0, chunk=100,
                             scale=d ** -0.5)
    o_parts, lse_parts = run_chunks(case)
    for c, (a, b) in enumerate(case.chunks):
        ro, rl = oracle.block_sparse(q, k, v, mask, q_pos0, a, b, 1, case.scale)
        compare(o_parts[c], lse_parts[c], ro, rl, TOL_BF16_O, what="ragged chunk %d" % c)


def test_fp32_block_sparse_d64():
    rng = np.random.default_rng(4)
    M, Nctx, H, Hkv, d = 200, 600, 4, 4, 64
    q = rng.standard_normal((M, H, d)).astype(np.float32)
    k = rng.standard_normal((Nctx, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((Nctx, Hkv, d)).astype(np.float32)
    mask = (rng.random((H, 2, 5)) < 0.5).astype(np.uint8)
    case = W.BlockSparseCase(q=q, k=k, v=v, mask=mask, q_pos0=400, chunk=256, scale=0.125,
                             dtype="f32")
    o_parts, lse_parts = run_chunks(case, torch.float32)
    for c, (a, b) in enumerate(case.chunks):
        ro, rl = oracle.block_sparse(q, k, v, mask, 400, a, b, 1, 0.125)
        compare(o_parts[c], lse_parts[c], ro, rl, TOL_F32_O, what="fp32 chunk %d" % c)


@pytest.mark.parametrize("C", [0, 1, 3, 40])
@pytest.mark.parametrize("with_sinks", [False, True])
def test_merge_kernel(C, with_sinks):
    rng = np.random.default_rng(C)
    R, d, H = 333, 128, 8
    op = rng.standard_normal((C, R, d))
    lp = rng.standard_normal((C, R)) * 3
    if C:
        lp[rng.random((C, R)) < 0.3] = -np.inf
        lp[:, 5] = -np.inf  # a row empty in every chunk
    sinks = rng.standard_normal(H).astype(np.float32) if with_sinks else None
    opt = torch.from_numpy(op.astype(np.float32)).cuda()
    lpt = torch.from_numpy(lp.astype(np.float32)).cuda()
    st = torch.from_numpy(sinks).cuda() if with_sinks else None
    o, lse = sa.merge_lse(opt, lpt, H, sinks=st)
    ro, rl = oracle.merge(op.astype(np.float32).astype(np.float64),
                          lp.astype(np.float32).astype(np.float64), H, sinks)
    compare(o, lse, ro, rl, 1e-5, what="merge C=%d" % C)


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("Nctx,M,chunk,kv_begin,kv_end", [(2048, 512, 512, 0, 2048),
                                                          (2300, 300, 1000, 0, 2300),
                                                          (4096, 256, 768, 640, 3900),
                                                          (1024, 128, 4096, 0, 1024)])
def test_all_chunks_in_one_call_match_the_chunk_calls(dt, Nctx, M, chunk, kv_begin, kv_end):
    # every chunk at once (one launch over (chunk, query block, head) with
    # bf16) gives each chunk's partials bit for bit; chunks need not be
    # aligned to key blocks, and the last one may be short
    case = W.block_sparse_bf16(5, Nctx=Nctx, M=M, chunk=chunk, density=0.3)
    q, k, v = dev(case.q, dt), dev(case.k, dt), dev(case.v, dt)
    mask = dev(case.mask, torch.uint8)
    o_all, l_all = sa.block_sparse_chunks_fwd(q, k, v, mask, case.q_pos0, kv_begin, kv_end, chunk,
                                              True, case.scale)
    sa.check_device()
    bounds = [(a, min(a + chunk, kv_end)) for a in range(kv_begin, kv_end, chunk)]
    assert o_all.shape[0] == len(bounds)
    for c, (a, b) in enumerate(bounds):
        o1, l1 = sa.block_sparse_fwd(q, k, v, mask, case.q_pos0, a, b, True, case.scale)
        sa.check_device()
        assert torch.equal(o_all[c], o1) and torch.equal(l_all[c], l1), c
    # and the merge of the chunk partials against the oracle over the range
    o, lse = sa.merge_lse(o_all.reshape(len(bounds), M * case.H, case.d),
                          l_all.reshape(len(bounds), M * case.H), case.H, out_dtype=dt)
    ro, rl = oracle.block_sparse(case.q, case.k, case.v, case.mask, case.q_pos0, kv_begin, kv_end,
                                 1, case.scale)
    compare(o.reshape(M, case.H, case.d), lse.reshape(M, case.H), ro, rl,
            TOL_BF16_O if dt == torch.bfloat16 else TOL_F32_O, what="merged chunks")
