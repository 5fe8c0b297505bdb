"""Pins of the oracle's cache bookkeeping (topk index lists, ring write).

Both are checked against a token-by-token simulation of the ring ("DeepSeek-V4
CSA/HCA walkthrough", section 3.3: a decode step writes its token at row
start_pos % win, older tokens are overwritten), which shares no formula with
the oracle's block split.
"""
import numpy as np
import pytest

import oracle


def _simulated_ring(p, win):
    """ring[row] = token stored there after tokens 0..p were written one by one."""
    ring = [-1] * win
    for t in range(p + 1):
        ring[t % win] = t
    return ring


@pytest.mark.parametrize("p", [0, 3, 7, 8, 9, 100, 1023])
def test_window_entries_point_at_the_latest_tokens(p):
    win = 8
    ix = oracle.topk_idxs([p], 1, win, win, 0)[0, 0]
    ring = _simulated_ring(p, win)
    for k in range(win):
        t = p - win + 1 + k  # the k-th most recent-but-(win-1-k) token
        if t < 0:
            assert ix[k] == -1
        else:
            assert ring[ix[k]] == t


@pytest.mark.parametrize("p,ratio,K", [(0, 4, 16), (5, 4, 16), (63, 4, 16), (1000, 4, 40),
                                       (17, 1, 12), (30, 0, 16)])
def test_compressed_part_counts_and_order(p, ratio, K):
    win = 8
    ix = oracle.topk_idxs([p], 1, K, win, ratio)[0, 0]
    comp = ix[win:]
    valid = comp[comp >= 0]
    if ratio == 0:
        assert valid.size == 0
        return
    visible = p // ratio + 1
    assert valid.size == min(visible, K - win)
    assert np.all(np.diff(valid) == 1)              # ascending, consecutive
    assert valid[-1] == win + p // ratio            # includes the newest visible row
    assert np.all(comp[valid.size:] == -1)           # padding after


def test_start_pos_shifts_positions():
    a = oracle.topk_idxs([0], 10, 24, 8, 4)
    b = oracle.topk_idxs([3], 7, 24, 8, 4)
    assert np.array_equal(a[0, 3:], b[0])


@pytest.mark.parametrize("start,S,win", [(0, 1, 8), (5, 1, 8), (0, 8, 8), (3, 10, 8),
                                         (13, 3, 8), (0, 30, 8), (7, 5, 4)])
def test_ring_write_matches_token_by_token_writes(start, S, win):
    rng = np.random.default_rng(start * 100 + S)
    B, N, d = 2, win + 5, 3
    cache = rng.standard_normal((B, N, d))
    new = rng.standard_normal((B, S, d))
    starts = [start, start + 2]
    got = oracle.kv_ring_write(cache, new, starts, win)
    for b in range(B):
        want = cache[b].copy()
        for i in range(S):  # one decode-style write per token
            want[(starts[b] + i) % win] = new[b, i]
        assert np.array_equal(got[b], want)
        assert np.array_equal(got[b, win:], cache[b, win:])  # compressed rows untouched
