"""Pins of the oracle's block-selection stages ("XAttention Offload Stream
Synchronization Fix", technical details: partial softmax stats per KV chunk,
their merge, block sums of the normalised probabilities, and the threshold
selection of key blocks).

Expected values come from counting (q = 0 makes every visible key equally
likely), from hand arithmetic on tiny inputs, from a direct fp64 softmax over
explicitly listed keys, and from invariants (chunked stats merged equal
one-shot stats; every row's probabilities sum to one), so that a wrong causal
bound, a swapped block index, a GQA head map error or a lost chunk fails one.
"""
import math

import numpy as np
import pytest

import oracle


def _rand(seed, M, Nctx, H, Hkv, d):
    r = np.random.default_rng(seed)
    return r.standard_normal((M, H, d)), r.standard_normal((Nctx, Hkv, d))


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_count_visible_keys(causal):
    M, Nctx, H, d, q_pos0, blk = 40, 100, 2, 4, 60, 16
    q = np.zeros((M, H, d))
    k = np.random.default_rng(0).standard_normal((Nctx, 1, d))
    m, l = oracle.xattn_partial_stats(q, k, q_pos0, 0, Nctx, causal, 0.5)
    for i in range(M):
        n = min(Nctx, q_pos0 + i + 1) if causal else Nctx
        assert np.all(m[i] == 0.0) and np.all(l[i] == n)
    bs = oracle.xattn_block_sum(q, k, m, l, q_pos0, 0, Nctx, causal, 0.5, blk=blk)
    for h in range(H):
        for qb in range(-(-M // blk)):
            for kb in range(-(-Nctx // blk)):
                want = 0.0
                for i in range(qb * blk, min(M, qb * blk + blk)):
                    n = min(Nctx, q_pos0 + i + 1) if causal else Nctx
                    seen = [j for j in range(kb * blk, min(Nctx, kb * blk + blk))
                            if not causal or j <= q_pos0 + i]
                    want += len(seen) / n
                assert abs(bs[h, qb, kb] - want) < 1e-12


def test_two_queries_three_keys_by_hand():
    q = np.array([[[1.0]], [[2.0]]])            # M = 2, H = 1, d = 1
    k = np.array([[[0.5]], [[-1.0]], [[3.0]]])  # Nctx = 3
    m, l = oracle.xattn_partial_stats(q, k, 1, 0, 3, True, 1.0)
    # row 0 (position 1) sees keys 0, 1; row 1 (position 2) sees all three
    assert m[0, 0] == 0.5 and abs(l[0, 0] - (1 + math.exp(-1.5))) < 1e-15
    assert m[1, 0] == 6.0 and abs(l[1, 0] - (math.exp(-5) + math.exp(-8) + 1)) < 1e-15
    bs = oracle.xattn_block_sum(q, k, m, l, 1, 0, 3, True, 1.0, blk=2)
    p0 = [1 / (1 + math.exp(-1.5)), math.exp(-1.5) / (1 + math.exp(-1.5))]
    z = math.exp(1) + math.exp(-2) + math.exp(6)
    p1 = [math.exp(1) / z, math.exp(-2) / z, math.exp(6) / z]
    assert abs(bs[0, 0, 0] - (p0[0] + p0[1] + p1[0] + p1[1])) < 1e-14
    assert abs(bs[0, 0, 1] - p1[2]) < 1e-14


def test_stats_against_a_listed_softmax_with_gqa():
    M, Nctx, H, Hkv, d = 9, 30, 4, 2, 8
    q, k = _rand(1, M, Nctx, H, Hkv, d)
    m, l = oracle.xattn_partial_stats(q, k, 20, 5, 27, True, 0.3)
    for i in range(M):
        for h in range(H):
            keys = [j for j in range(5, 27) if j <= 20 + i]
            s = [0.3 * sum(q[i, h, c] * k[j, h // 2, c] for c in range(d)) for j in keys]
            mm = max(s)
            assert abs(m[i, h] - mm) < 1e-13
            assert abs(l[i, h] - sum(math.exp(x - mm) for x in s)) < 1e-12


def test_rows_seeing_nothing():
    q, k = _rand(2, 4, 50, 1, 1, 4)
    m, l = oracle.xattn_partial_stats(q, k, 0, 10, 50, True, 1.0)
    # rows at positions 0..3 see no key of [10, 50)
    assert np.all(np.isneginf(m)) and np.all(l == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_chunked_stats_merge_to_one_shot(causal):
    M, Nctx, H, Hkv, d = 33, 200, 2, 1, 8
    q, k = _rand(3, M, Nctx, H, Hkv, d)
    m1, l1 = oracle.xattn_partial_stats(q, k, 150, 0, Nctx, causal, 0.4)
    parts = [oracle.xattn_partial_stats(q, k, 150, a, min(a + 64, Nctx), causal, 0.4)
             for a in range(0, Nctx, 64)]
    m, l = oracle.xattn_merge_stats([p[0] for p in parts], [p[1] for p in parts])
    assert np.array_equal(m, m1)
    np.testing.assert_allclose(l, l1, rtol=1e-13)


def test_block_sums_of_a_row_block_sum_to_its_rows():
    M, Nctx, H, Hkv, d, blk = 70, 300, 2, 2, 8, 32
    q, k = _rand(4, M, Nctx, H, Hkv, d)
    m, l = oracle.xattn_partial_stats(q, k, 230, 0, Nctx, True, 0.5)
    total = np.zeros((H, -(-M // blk), -(-Nctx // blk)))
    for a in range(0, Nctx, 96):  # chunk by chunk, as the pages do
        total += oracle.xattn_block_sum(q, k, m, l, 230, a, min(a + 96, Nctx), True, 0.5, blk=blk)
    rows = np.array([min(blk, M - qb * blk) for qb in range(-(-M // blk))], dtype=np.float64)
    np.testing.assert_allclose(total.sum(axis=2), np.broadcast_to(rows, (H, len(rows))),
                               rtol=1e-12)


def test_a_dominant_key_takes_its_block():
    M, Nctx, H, d, blk = 16, 64, 1, 4, 16
    q = np.zeros((M, H, d))
    q[:, 0, 0] = 10.0
    k = np.zeros((Nctx, 1, d))
    k[37, 0, 0] = 10.0  # key block 2
    m, l = oracle.xattn_partial_stats(q, k, 48, 0, Nctx, True, 1.0)
    bs = oracle.xattn_block_sum(q, k, m, l, 48, 0, Nctx, True, 1.0, blk=blk)
    assert bs[0, 0, 2] > 16 * (1 - 1e-12)
    sel = oracle.xattn_find_blocks(bs, 0.9)
    assert sel[0, 0].tolist() == [0, 0, 1, 0]


@pytest.mark.parametrize("sums,thr,want", [
    ([0.5, 0.3, 0.2], 0.75, [1, 1, 0]),
    ([0.2, 0.2, 0.6], 0.75, [1, 0, 1]),   # equal masses: the lower block first
    ([0.2, 0.2, 0.6], 0.8, [1, 0, 1]),    # 0.6 + 0.2 = 0.8 reaches 0.8 exactly
    ([0.2, 0.2, 0.6], 0.81, [1, 1, 1]),
    ([0.1, 0.0, 0.9], 1.0, [1, 0, 1]),    # zero mass never needed
    ([0.1, 0.0, 0.9], 0.0, [0, 0, 1]),    # the first block always
    ([0.0, 0.0, 0.0], 0.9, [0, 0, 0]),    # nothing to select
    # a mass is never negative: given negative or NaN sums count as 0
    ([0.5, -1.0, 0.3], 0.9, [1, 0, 1]),   # total 0.8, not -0.2
    ([-0.5, -0.1, 0.0], 0.5, [0, 0, 0]),  # total 0: nothing
    ([float("nan"), 0.4, 0.6], 1.0, [0, 1, 1]),
    ([-0.0, 0.3, -2.0], 1.0, [0, 1, 0]),
])
def test_selection_by_hand(sums, thr, want):
    got = oracle.xattn_find_blocks(np.array([[sums]]), thr)
    assert got[0, 0].tolist() == want
