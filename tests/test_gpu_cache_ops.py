"""GPU parity of the cache bookkeeping kernels (index lists, ring write) with
the oracle: bit-exact (integers and copies)."""
import numpy as np
import pytest
import torch

import oracle
import windowed_attention_sinks_gb300 as sa

pytestmark = pytest.mark.gpu


def _starts(*v):
    return torch.tensor(v, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("K,win,ratio", [(2048, 128, 4), (645, 128, 4), (64, 16, 1), (40, 8, 0),
                                         (6, 8, 4)])
def test_topk_idxs_small(K, win, ratio):
    starts = [0, 5, 1000, 127]
    got = sa.build_topk_idxs(_starts(*starts), 37, K, win, ratio)
    want = oracle.topk_idxs(starts, 37, K, win, ratio)
    assert np.array_equal(got.cpu().numpy(), want)


def test_topk_idxs_prefill_size_sampled():
    # one sequence of 8192 queries from position 0, K = 2048 (the prefill layout)
    M, K, win, ratio = 8192, 2048, 128, 4
    got = sa.build_topk_idxs(_starts(0), M, K, win, ratio).cpu().numpy()[0]
    rng = np.random.default_rng(0)
    for p in sorted(set(rng.integers(0, M, 48).tolist()) | {0, 126, 127, 128, 7679, 7680, M - 1}):
        want = oracle.topk_idxs([p], 1, K, win, ratio)[0, 0]
        assert np.array_equal(got[p], want), p


def test_topk_idxs_decode_size():
    # 64 requests, one query each, at scattered positions up to 32767
    rng = np.random.default_rng(1)
    starts = rng.integers(0, 32768, 64).tolist()
    got = sa.build_topk_idxs(_starts(*starts), 1, 640, 128, 4)
    want = oracle.topk_idxs(starts, 1, 640, 128, 4)
    assert np.array_equal(got.cpu().numpy(), want)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("S", [1, 5, 128, 300])
def test_ring_write(dtype, S):
    win, N, d, B = 128, 128 + 40, 128, 3
    g = torch.Generator().manual_seed(S)
    cache = torch.randn((B, N, d), generator=g).to(dtype)
    new = torch.randn((B, S, d), generator=g).to(dtype)
    starts = [0, 77, 5000]
    want = oracle.kv_ring_write(cache.float().numpy(), new.float().numpy(), starts, win)
    c = cache.cuda()
    sa.kv_ring_write(c, new.cuda(), _starts(*starts), win)
    sa.check_device()
    assert np.array_equal(c.float().cpu().numpy(), want)


def test_negative_start_pos_is_reported():
    out = sa.build_topk_idxs(_starts(-3), 2, 16, 8, 4)
    with pytest.raises(sa.SattnError):
        sa.check_device()
    assert (out.cpu().numpy() == -1).all()
