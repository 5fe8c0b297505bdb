"""GPU parity of the block-selection stages ("XAttention Offload Stream
Synchronization Fix", technical details) with the oracle.

Tolerances: partial stats m within 1e-4 (fp32 scores of order 1), l and the
block sums within 1e-4 relative (sums of ex2-approximated exponentials); the
selection is compared bit for bit with the oracle's selection run on the
kernel's own fp32 block sums (the decision is taken in the same precision on
both sides)."""
import numpy as np
import pytest
import torch

import oracle
import windowed_attention_sinks_gb300 as sa
from windowed_attention_sinks_gb300 import workloads as W

from gpu_helpers import dev

pytestmark = pytest.mark.gpu


def _qk(seed, M, Nctx, H, Hkv, d=128, qscale=1.0):
    r = np.random.default_rng(seed)
    q = W.round_bf16((r.standard_normal((M, H, d)) * qscale).astype(np.float32))
    k = W.round_bf16(r.standard_normal((Nctx, Hkv, d)).astype(np.float32))
    return q, k


def _cmp_stats(m, l, wm, wl):
    m, l = m.cpu().numpy(), l.cpu().numpy()
    assert np.array_equal(np.isneginf(m), np.isneginf(wm))
    fin = np.isfinite(wm)
    assert np.abs(m[fin] - wm[fin]).max(initial=0) <= 1e-4
    assert np.all(l[~fin] == 0)
    assert np.abs(l[fin] - wl[fin]).max(initial=0) <= 1e-4 * np.abs(wl[fin]).max(initial=1)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("M,Nctx,H,Hkv,q_pos0", [(300, 700, 4, 2, 400), (128, 256, 2, 2, 128),
                                                 (77, 1000, 3, 1, 923)])
def test_stats_chunks_and_merge(causal, M, Nctx, H, Hkv, q_pos0):
    q, k = _qk(M + Nctx, M, Nctx, H, Hkv)
    scale = 128 ** -0.5
    qd, kd = dev(q, torch.bfloat16), dev(k, torch.bfloat16)
    chunks = [(a, min(a + 256, Nctx)) for a in range(0, Nctx, 256)]
    mp = torch.empty((len(chunks), M, H), device="cuda")
    lp = torch.empty_like(mp)
    wparts = []
    for c, (a, b) in enumerate(chunks):
        sa.xattn_partial_stats(qd, kd, q_pos0, a, b, causal, scale, m=mp[c], l=lp[c])
        wparts.append(oracle.xattn_partial_stats(q, k, q_pos0, a, b, causal, scale))
    sa.check_device()
    for c in range(len(chunks)):
        _cmp_stats(mp[c], lp[c], *wparts[c])
    m, l = sa.xattn_merge_stats(mp, lp)
    sa.check_device()
    wm, wl = oracle.xattn_merge_stats([p[0] for p in wparts], [p[1] for p in wparts])
    _cmp_stats(m, l, wm, wl)
    # block sums chunk by chunk with the merged stats, then the selection
    bs = torch.zeros((H, -(-M // 128), -(-Nctx // 128)), device="cuda")
    for a, b in chunks:
        sa.xattn_block_sum(qd, kd, m, l, q_pos0, a, b, causal, scale, block_sum=bs)
    sa.check_device()
    want = sum(oracle.xattn_block_sum(q, k, wm, wl, q_pos0, a, b, causal, scale) for a, b in chunks)
    got = bs.cpu().numpy()
    np.testing.assert_allclose(got, want, rtol=1e-4, atol=1e-5)
    for thr in (0.5, 0.9, 1.0):
        mask = sa.xattn_find_blocks(bs, thr).cpu().numpy()
        assert np.array_equal(mask, oracle.xattn_find_blocks(got, thr)), thr


def test_rows_that_see_nothing():
    # causal rows at positions 0..63 see no key of the chunk [128, 384)
    q, k = _qk(5, 64, 384, 2, 2)
    m, l = sa.xattn_partial_stats(dev(q, torch.bfloat16), dev(k, torch.bfloat16), 0, 128, 384,
                                  True, 0.1)
    sa.check_device()
    assert torch.all(torch.isneginf(m)) and torch.all(l == 0)


def test_peaked_scores():
    # sharper softmax (q scaled by 4): the online max moves often within rows
    q, k = _qk(6, 256, 1024, 2, 1, qscale=4.0)
    scale = 128 ** -0.5
    mask, bs = sa.xattn_select_blocks(dev(q, torch.bfloat16), dev(k, torch.bfloat16), 768, True,
                                      0.9, scale, chunk=512)
    sa.check_device()
    wm, wl = oracle.xattn_partial_stats(q, k, 768, 0, 1024, True, scale)
    want = oracle.xattn_block_sum(q, k, wm, wl, 768, 0, 1024, True, scale)
    np.testing.assert_allclose(bs.cpu().numpy(), want, rtol=1e-4, atol=1e-5)
    assert np.array_equal(mask.cpu().numpy(), oracle.xattn_find_blocks(bs.cpu().numpy(), 0.9))


def test_full_size_sampled():
    # the chunked block-sparse workload's shape: the last 4096 positions of a
    # 32768-token context, 32 heads over 8 KV heads, 4096-key chunks
    case = W.block_sparse_bf16(0)
    q, k = case.q, case.k
    M, H = q.shape[0], q.shape[1]
    Nctx, Hkv = k.shape[0], k.shape[1]
    scale = case.scale
    mask, bs = sa.xattn_select_blocks(dev(q, torch.bfloat16), dev(k, torch.bfloat16), case.q_pos0,
                                      True, 0.9, scale, chunk=4096)
    sa.check_device()
    got = bs.cpu().numpy()
    rng = np.random.default_rng(0)
    for h, qb in [(0, 0), (31, 31)] + [tuple(x) for x in rng.integers(0, 32, (4, 2))]:
        rows = slice(qb * 128, (qb + 1) * 128)
        g = h // (H // Hkv)
        q1 = q[rows, h:h + 1]
        k1 = k[:, g:g + 1]
        wm, wl = oracle.xattn_partial_stats(q1, k1, case.q_pos0 + qb * 128, 0, Nctx, True, scale)
        want = oracle.xattn_block_sum(q1, k1, wm, wl, case.q_pos0 + qb * 128, 0, Nctx, True,
                                      scale)[0, 0]
        np.testing.assert_allclose(got[h, qb], want, rtol=1e-4, atol=1e-5, err_msg=str((h, qb)))
    assert np.array_equal(mask.cpu().numpy(), oracle.xattn_find_blocks(got, 0.9))


@pytest.mark.parametrize("M,Nctx,q_pos0", [(5, 60, 55), (128, 100, 0), (40, 130, 90)])
def test_tiny_and_partial_blocks(M, Nctx, q_pos0):
    # fewer rows than a query block, fewer keys than a key block, ragged tails
    q, k = _qk(7 + M, M, Nctx, 2, 1)
    scale = 128 ** -0.5
    mask, bs = sa.xattn_select_blocks(dev(q, torch.bfloat16), dev(k, torch.bfloat16), q_pos0,
                                      True, 0.9, scale, chunk=128)
    sa.check_device()
    wm, wl = oracle.xattn_partial_stats(q, k, q_pos0, 0, Nctx, True, scale)
    want = oracle.xattn_block_sum(q, k, wm, wl, q_pos0, 0, Nctx, True, scale)
    np.testing.assert_allclose(bs.cpu().numpy(), want, rtol=1e-4, atol=1e-5)
    assert np.array_equal(mask.cpu().numpy(), oracle.xattn_find_blocks(bs.cpu().numpy(), 0.9))


def test_empty_chunk_leaves_stats_empty_and_sums_untouched():
    q, k = _qk(8, 64, 256, 2, 2)
    qd, kd = dev(q, torch.bfloat16), dev(k, torch.bfloat16)
    m, l = sa.xattn_partial_stats(qd, kd, 200, 128, 128, True, 0.1)
    bs = torch.full((2, 1, 2), 5.0, device="cuda")
    sa.xattn_block_sum(qd, kd, m, l, 200, 128, 128, True, 0.1, block_sum=bs)
    sa.check_device()
    assert torch.all(torch.isneginf(m)) and torch.all(l == 0)
    assert torch.all(bs == 5.0)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("M,Nctx,H,Hkv,q_pos0,chunk", [(300, 5000, 4, 2, 4700, 1024),
                                                       (200, 700, 3, 3, 500, 256),
                                                       (129, 9000, 6, 2, 8871, 4096),
                                                       (64, 4224, 8, 1, 4160, 640)])
def test_one_call_equals_the_stages(causal, M, Nctx, H, Hkv, q_pos0, chunk):
    # the one-call selection (stage 1 over all chunks in one launch, stage 3
    # over 4096-key pieces) reproduces the four stage calls made chunk by
    # chunk, bit for bit; groups of 1, 2, 3 and 8 heads per KV head
    q, k = _qk(11 + M, M, Nctx, H, Hkv)
    scale = 128 ** -0.5
    qd, kd = dev(q, torch.bfloat16), dev(k, torch.bfloat16)
    mask, bs = sa.xattn_select_blocks(qd, kd, q_pos0, causal, 0.9, scale, chunk=chunk)
    chunks = [(a, min(a + chunk, Nctx)) for a in range(0, Nctx, chunk)]
    mp = torch.empty((len(chunks), M, H), device="cuda")
    lp = torch.empty_like(mp)
    for c, (a, b) in enumerate(chunks):
        sa.xattn_partial_stats(qd, kd, q_pos0, a, b, causal, scale, m=mp[c], l=lp[c])
    m, l = sa.xattn_merge_stats(mp, lp)
    bs2 = torch.full_like(bs, float("nan"))
    for a, b in chunks:
        sa.xattn_block_sum(qd, kd, m, l, q_pos0, a, b, causal, scale, block_sum=bs2)
    mask2 = sa.xattn_find_blocks(bs2, 0.9)
    sa.check_device()
    assert torch.equal(bs, bs2) and torch.equal(mask, mask2)
    # and the oracle on the whole range
    wm, wl = oracle.xattn_partial_stats(q, k, q_pos0, 0, Nctx, causal, scale)
    want = oracle.xattn_block_sum(q, k, wm, wl, q_pos0, 0, Nctx, causal, scale)
    np.testing.assert_allclose(bs.cpu().numpy(), want, rtol=1e-4, atol=1e-5)


def test_one_call_reuses_caller_buffers():
    q, k = _qk(12, 256, 2048, 4, 2)
    qd, kd = dev(q, torch.bfloat16), dev(k, torch.bfloat16)
    ws = torch.empty(sa.xattn_select_workspace_bytes(256, 4, 2048, 512), dtype=torch.uint8,
                     device="cuda")
    bs = torch.full((4, 2, 16), float("nan"), device="cuda")
    mask = torch.full((4, 2, 16), 7, dtype=torch.uint8, device="cuda")
    m1, b1 = sa.xattn_select_blocks(qd, kd, 1792, True, 0.8, None, chunk=512, workspace=ws,
                                    block_sum=bs, mask=mask)
    sa.check_device()
    assert m1.data_ptr() == mask.data_ptr() and b1.data_ptr() == bs.data_ptr()
    assert not torch.isnan(bs).any() and torch.all(mask <= 1)
    m2, b2 = sa.xattn_select_blocks(qd, kd, 1792, True, 0.8, None, chunk=512)
    sa.check_device()
    assert torch.equal(b1, b2) and torch.equal(m1, m2)


def test_find_blocks_counts_negative_and_nan_sums_as_zero():
    # caller-supplied sums may hold values a probability mass cannot take;
    # the kernel and the oracle both count negatives, -0 and NaN as 0
    rng = np.random.default_rng(11)
    H, QB, KB = 3, 5, 37
    bs = rng.random((H, QB, KB)).astype(np.float32)
    neg = rng.random((H, QB, KB)) < 0.3
    bs[neg] = -rng.random(int(neg.sum())).astype(np.float32) * 2
    bs[0, 0, :] = -1.0            # a row with nothing positive: nothing selected
    bs[0, 1, 3] = np.float32(-0.0)
    bs[0, 1, 4] = np.nan
    bs[1, 2, :5] = [0.4, -3.0, 0.4, np.nan, 0.2]
    for thr in (0.0, 0.5, 0.9, 1.0):
        mask = sa.xattn_find_blocks(torch.from_numpy(bs).cuda(), thr)
        sa.check_device()
        want = oracle.xattn_find_blocks(bs, thr)
        assert np.array_equal(mask.cpu().numpy(), want), thr
        assert not want[0, 0].any()


@pytest.mark.parametrize("kind,KB", [("narrow", 200), ("narrow", 256), ("wide", 200),
                                     ("subnormal", 256), ("ties", 256), ("narrow", 300)])
def test_find_blocks_exact_on_both_paths(kind, KB):
    """Rows of at most 256 blocks whose masses lie within 2^21 of each other
    take the kernel's parallel integer prefix sums; wider spans and longer
    rows the sequential float64 walk. Both must match the oracle decision for
    decision, ties and exact boundaries included (the threshold is passed to
    the oracle rounded to float32, as the kernel receives it)."""
    rng = np.random.default_rng(KB + len(kind))
    H, QB = 3, 7
    if kind == "narrow":
        bs = (rng.random((H, QB, KB)) + 0.01).astype(np.float32)
    elif kind == "wide":
        bs = (10.0 ** rng.uniform(-30, 0, (H, QB, KB))).astype(np.float32)
    elif kind == "subnormal":  # masses below the smallest normal float, and a few just above
        bs = (rng.random((H, QB, KB)) * 1e-39).astype(np.float32)
        bs[:, :, ::17] = np.float32(2e-38)
    else:  # equal masses and running sums that hit the target exactly
        bs = rng.choice(np.float32([0.0, 0.125, 0.25, 0.5]), (H, QB, KB))
    bs[0, 0, :] = 0.0  # a row with no mass
    for thr in (0.0, 0.25, 0.3, 0.5, 0.75, 0.9, 0.999, 1.0):
        t32 = float(np.float32(thr))
        mask = sa.xattn_find_blocks(torch.from_numpy(bs).cuda(), t32)
        sa.check_device()
        want = oracle.xattn_find_blocks(bs, t32)
        assert np.array_equal(mask.cpu().numpy(), want), (kind, KB, thr)
        assert not want[0, 0].any()


def test_selection_flips_against_fp64_block_sums():
    # the kernel's fp32 block sums against the oracle's fp64 ones: thresholding
    # is discontinuous, so a block whose cumulative mass sits at the threshold
    # may flip; count how many decisions differ end to end
    case = W.block_sparse_bf16(0, Nctx=4096, M=1024, chunk=1024)
    q, k = case.q, case.k
    scale = case.scale
    mask, bs = sa.xattn_select_blocks(dev(q, torch.bfloat16), dev(k, torch.bfloat16), case.q_pos0,
                                      True, 0.9, scale, chunk=1024)
    sa.check_device()
    wm, wl = oracle.xattn_partial_stats(q, k, case.q_pos0, 0, case.Nctx, True, scale)
    want_bs = oracle.xattn_block_sum(q, k, wm, wl, case.q_pos0, 0, case.Nctx, True, scale)
    want = oracle.xattn_find_blocks(want_bs, 0.9)
    got = mask.cpu().numpy()
    flips = int((got != want).sum())
    # stage by stage the decisions are exact (the oracle on the kernel's sums)
    assert np.array_equal(got, oracle.xattn_find_blocks(bs.cpu().numpy(), 0.9))
    print("selection decisions that differ from the fp64 chain: %d of %d (%d selected)" % (
        flips, got.size, int(want.sum())))
    assert flips <= max(2, got.size // 200)
