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


def _support_counts(o, lse):
    """With q = 0 every visible key has the same weight: lse = ln|S| and
    o = (counts of the one-hot codes of the visible keys) / |S|. Rounding
    recovers |S| and the integer counts exactly (fp32 partials)."""
    lse = np.asarray(lse, dtype=np.float64)
    n = np.rint(np.exp(lse))  # -inf (nothing visible) -> 0
    counts = np.rint(np.asarray(o, dtype=np.float64) * n[..., None])
    return n.astype(np.int64), counts.astype(np.int64)


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_block_mask_decisions_bit_exact(dt):
    """Visible sets of the block-sparse path, bit for bit: q = 0 and one-hot
    values, first v_j = e_(j mod 128) (the key's offset in its block), then
    v_j = e_(j // 128) (its block). Per row and chunk, |S| and both code
    histograms must equal the oracle's exactly. Chunk bounds and q_pos0 are
    not multiples of 128, so the chunk edges cut blocks, the causal limit
    cuts the diagonal blocks, and the mask is random elsewhere."""
    rng = np.random.default_rng(21)
    M, Nctx, H, Hkv, d = 300, 2600, 4, 2, 128
    q_pos0, kv_begin, kv_end, chunk = 2250, 77, 2555, 700
    QB, KB = -(-M // 128), -(-Nctx // 128)
    mask = (rng.random((H, QB, KB)) < 0.45).astype(np.uint8)
    for qb in range(QB):  # blocks on the causal diagonal of each query block
        lo, hi = (q_pos0 + 128 * qb) // 128, (q_pos0 + min(M, 128 * qb + 128) - 1) // 128
        mask[:, qb, lo:hi + 1] = 1
    mask[1, 0, :] = 0  # a (head, query block) that sees nothing
    q = np.zeros((M, H, d), np.float32)
    k = W.round_bf16(rng.standard_normal((Nctx, Hkv, d)).astype(np.float32))
    bounds = [(a, min(a + chunk, kv_end)) for a in range(kv_begin, kv_end, chunk)]
    j = np.arange(Nctx)
    for code in (j % 128, j // 128):
        v = np.zeros((Nctx, Hkv, d), np.float32)
        v[j, :, code] = 1.0
        case = W.BlockSparseCase(q=q, k=k, v=v, mask=mask, q_pos0=q_pos0, chunk=chunk,
                                 scale=d ** -0.5, dtype="bf16" if dt == torch.bfloat16 else "f32")
        qd, kd, vd, md = dev(q, dt), dev(k, dt), dev(v, dt), dev(mask, torch.uint8)
        o_all, l_all = sa.block_sparse_chunks_fwd(qd, kd, vd, md, q_pos0, kv_begin, kv_end, chunk,
                                                  True, case.scale)
        sa.check_device()
        for c, (a, b) in enumerate(bounds):
            ro, rl = oracle.block_sparse(q, k, v, mask, q_pos0, a, b, 1, case.scale)
            n_ref, h_ref = _support_counts(ro.reshape(M, H, d), rl.reshape(M, H))
            o1, l1 = sa.block_sparse_fwd(qd, kd, vd, md, q_pos0, a, b, True, case.scale)
            sa.check_device()
            for what, (og, lg) in (("one chunk", (o1, l1)), ("all chunks", (o_all[c], l_all[c]))):
                n_got, h_got = _support_counts(og.cpu().numpy(), lg.cpu().numpy())
                assert np.array_equal(n_got, n_ref), "%s %d: |S| differs" % (what, c)
                assert np.array_equal(h_got, h_ref), "%s %d: visible keys differ" % (what, c)
        # the partials merged over [kv_begin, kv_end) against the one-shot oracle
        C = len(bounds)
        o, lse = sa.merge_lse(o_all.reshape(C, M * H, d), l_all.reshape(C, M * H), H,
                              out_dtype=torch.float32)
        ro, rl = oracle.block_sparse(q, k, v, mask, q_pos0, kv_begin, kv_end, 1, case.scale)
        n_ref, h_ref = _support_counts(ro.reshape(M, H, d), rl.reshape(M, H))
        n_got, h_got = _support_counts(o.reshape(M, H, d).cpu().numpy(),
                                       lse.reshape(M, H).cpu().numpy())
        assert np.array_equal(n_got, n_ref) and np.array_equal(h_got, h_ref), "merged"
        # the case exercises what it claims: empty rows, rows cut by the
        # chunk edges, and rows whose diagonal block is partly visible
        assert (n_ref == 0).any() and (n_ref > 0).any()
