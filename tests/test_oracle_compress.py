"""Pins of the oracle's compressor gated pooling ("DeepSeek-V4 CSA/HCA
walkthrough", sections 5.1-5.2).

Each expected value is built here without the oracle's reshape/softmax path:
identity and mean-pooling closed forms, the limit of one dominant score, hand
arithmetic on a few numbers, and invariances (a score shift common to a
window's entries, the tail tokens, recomputing a window from the tokens of it
and its predecessor only), so that a dropped ape, a wrong half of the overlap
split, a softmax over the wrong axis or an off-by-one window fails one of them.
"""
import math

import numpy as np
import pytest

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


def _inputs(seed, B, S, d, ratio, overlap):
    r = _rng(seed)
    W = (2 if overlap else 1) * d
    return (r.standard_normal((B, S, W)), r.standard_normal((B, S, W)),
            r.standard_normal((ratio, W)))


def test_ratio_one_without_overlap_is_the_identity():
    kv, score, ape = _inputs(0, 2, 7, 5, 1, False)
    out = oracle.compress_kv(kv, score, ape, 1, False)
    np.testing.assert_allclose(out, kv, rtol=0, atol=1e-15)


@pytest.mark.parametrize("ratio", [2, 4, 8])
def test_equal_scores_give_the_window_mean(ratio):
    B, S, d = 2, 5 * ratio + 3, 6
    kv = _rng(1).standard_normal((B, S, d))
    out = oracle.compress_kv(kv, np.zeros((B, S, d)), np.zeros((ratio, d)), ratio, False)
    assert out.shape == (B, S // ratio, d)
    for b in range(B):
        for w in range(S // ratio):
            want = [sum(kv[b, w * ratio + i, j] for i in range(ratio)) / ratio for j in range(d)]
            np.testing.assert_allclose(out[b, w], want, rtol=0, atol=1e-13)


@pytest.mark.parametrize("ratio", [1, 2, 4])
def test_equal_scores_with_overlap_average_both_halves(ratio):
    # window w averages the first d columns of window w-1's tokens and the last
    # d columns of its own tokens; window 0 has only its own tokens
    B, n, d = 1, 6, 3
    S = n * ratio
    kv = _rng(2).standard_normal((B, S, 2 * d))
    out = oracle.compress_kv(kv, np.zeros((B, S, 2 * d)), np.zeros((ratio, 2 * d)), ratio, True)
    for w in range(n):
        for j in range(d):
            own = [kv[0, w * ratio + i, d + j] for i in range(ratio)]
            prev = [kv[0, (w - 1) * ratio + i, j] for i in range(ratio)] if w > 0 else []
            want = sum(own + prev) / len(own + prev)
            assert abs(out[0, w, j] - want) < 1e-13


def test_ape_is_added_per_window_entry():
    # ape alone (scores 0) sets the weights: entry i of every window gets
    # exp(ape[i]) / sum_k exp(ape[k])
    ratio, d = 3, 2
    kv = _rng(3).standard_normal((1, 2 * ratio, d))
    ape = np.array([[0.5, -1.0], [2.0, 0.0], [-0.25, 1.5]])
    out = oracle.compress_kv(kv, np.zeros((1, 2 * ratio, d)), ape, ratio, False)
    for w in range(2):
        for j in range(d):
            z = sum(math.exp(ape[i, j]) for i in range(ratio))
            want = sum(math.exp(ape[i, j]) / z * kv[0, w * ratio + i, j] for i in range(ratio))
            assert abs(out[0, w, j] - want) < 1e-13


@pytest.mark.parametrize("overlap", [False, True])
def test_a_dominant_score_selects_its_token(overlap):
    ratio, n, d = 4, 5, 3
    S = n * ratio
    coff = 2 if overlap else 1
    r = _rng(4)
    kv = r.standard_normal((1, S, coff * d))
    score = np.zeros((1, S, coff * d))
    pick = r.integers(0, ratio, size=(n, d))
    for w in range(n):
        for j in range(d):
            score[0, w * ratio + pick[w, j], (coff - 1) * d + j] = 1000.0
    out = oracle.compress_kv(kv, score, np.zeros((ratio, coff * d)), ratio, overlap)
    for w in range(n):
        for j in range(d):
            assert abs(out[0, w, j] - kv[0, w * ratio + pick[w, j], (coff - 1) * d + j]) < 1e-12


def test_two_tokens_by_hand():
    # one window of two tokens, one column: (e^a k0 + e^b k1) / (e^a + e^b)
    kv = np.array([[[3.0], [-1.0]]])
    score = np.array([[[0.2], [1.1]]])
    ape = np.array([[0.3], [-0.4]])
    a, b = 0.2 + 0.3, 1.1 - 0.4
    want = (math.exp(a) * 3.0 + math.exp(b) * -1.0) / (math.exp(a) + math.exp(b))
    assert abs(oracle.compress_kv(kv, score, ape, 2, False)[0, 0, 0] - want) < 1e-13


def test_overlap_by_hand():
    # ratio 1, d = 1, two tokens: row 1 mixes token 0's first column and token
    # 1's second column
    kv = np.array([[[1.0, 10.0], [2.0, 20.0]]])
    score = np.array([[[0.0, 5.0], [0.7, -0.3]]])
    ape = np.array([[0.1, 0.2]])
    out = oracle.compress_kv(kv, score, ape, 1, True)
    assert abs(out[0, 0, 0] - 10.0) < 1e-15  # window 0: only its own second column
    a, b = 0.0 + 0.1, -0.3 + 0.2
    want = (math.exp(a) * 1.0 + math.exp(b) * 20.0) / (math.exp(a) + math.exp(b))
    assert abs(out[0, 1, 0] - want) < 1e-13


def test_a_shift_common_to_a_window_column_changes_nothing():
    ratio, d = 4, 5
    kv, score, ape = _inputs(5, 2, 6 * ratio, d, ratio, False)
    shift = _rng(6).standard_normal((2, 6, 1, d)) * 50
    shifted = (score.reshape(2, 6, ratio, d) + shift).reshape(score.shape)
    np.testing.assert_allclose(oracle.compress_kv(kv, shifted, ape, ratio, False),
                               oracle.compress_kv(kv, score, ape, ratio, False),
                               rtol=0, atol=1e-12)


def test_tail_tokens_do_not_matter():
    ratio, d = 4, 3
    kv, score, ape = _inputs(7, 1, 5 * ratio + 3, d, ratio, True)
    out = oracle.compress_kv(kv, score, ape, ratio, True)
    kv2, score2 = kv.copy(), score.copy()
    kv2[:, 5 * ratio:] = 1e3
    score2[:, 5 * ratio:] = -7.0
    assert out.shape == (1, 5, d)
    np.testing.assert_array_equal(oracle.compress_kv(kv2, score2, ape, ratio, True), out)


def test_a_window_needs_only_itself_and_its_predecessor():
    # the decode step compresses a window from the tokens of the current and
    # the previous window; the row equals the one computed over the sequence
    ratio, d, n = 4, 3, 7
    kv, score, ape = _inputs(8, 1, n * ratio, d, ratio, True)
    full = oracle.compress_kv(kv, score, ape, ratio, True)
    for w in range(1, n):
        sl = slice((w - 1) * ratio, (w + 1) * ratio)
        part = oracle.compress_kv(kv[:, sl], score[:, sl], ape, ratio, True)
        np.testing.assert_allclose(part[0, 1], full[0, w], rtol=0, atol=1e-14)


def test_rows_are_convex_combinations():
    ratio, d = 8, 4
    kv, score, ape = _inputs(9, 3, 10 * ratio, d, ratio, True)
    out = oracle.compress_kv(kv, 4 * score, ape, ratio, True)
    for w in range(1, 10):
        for j in range(d):
            vals = np.concatenate([kv[:, (w - 1) * ratio:w * ratio, j],
                                   kv[:, w * ratio:(w + 1) * ratio, d + j]], axis=1)
            assert np.all(out[:, w, j] <= vals.max(axis=1) + 1e-12)
            assert np.all(out[:, w, j] >= vals.min(axis=1) - 1e-12)
