"""GPU parity of the compressor gated pooling (sattn_compress_kv) with the
oracle. Tolerances: fp32 output 1e-5 absolute (fp32 arithmetic with ex2 over
values of order 1); bf16 output 1e-2 (the row's own bf16 rounding included)."""
import numpy as np
import pytest
import torch

import oracle
import windowed_attention_sinks_gb300 as sa
from windowed_attention_sinks_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-2}


def _dev(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).cuda()


def _run(case, in_dtype, out_dtype):
    kv = _dev(case.kv, in_dtype)
    score = _dev(case.score, in_dtype)
    ape = _dev(case.ape, torch.float32)
    out = sa.compress_kv(kv, score, ape, case.ratio, case.overlap, out_dtype=out_dtype)
    sa.check_device()
    return out.float().cpu().numpy()


@pytest.mark.parametrize("ratio", [1, 2, 4, 7])
@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("in_dtype,out_dtype", [(torch.float32, torch.float32),
                                                (torch.bfloat16, torch.bfloat16),
                                                (torch.bfloat16, torch.float32),
                                                (torch.float32, torch.bfloat16)])
def test_small(ratio, overlap, in_dtype, out_dtype):
    # three sequences with a ragged tail of 3 tokens, d = 64
    case = W.compress_case(ratio, B=3, S=5 * ratio + 3, d=64, ratio=ratio, overlap=overlap,
                           bf16=in_dtype == torch.bfloat16)
    got = _run(case, in_dtype, out_dtype)
    want = oracle.compress_kv(case.kv, case.score, case.ape, ratio, overlap)
    assert got.shape == want.shape
    assert np.abs(got - want).max() <= TOL[out_dtype]


@pytest.mark.parametrize("d", [4, 12, 128, 132, 512])
def test_head_dims(d):
    # d/4 threads per window: below, at and across a warp, and a whole block
    case = W.compress_case(11, B=2, S=40, d=d, ratio=4, overlap=True)
    got = _run(case, torch.float32, torch.float32)
    want = oracle.compress_kv(case.kv, case.score, case.ape, 4, True)
    assert np.abs(got - want).max() <= 1e-5


def test_large_ratio_with_overlap():
    # a long window (HCA-style ratio 128): 256 entries per column
    case = W.compress_case(12, B=2, S=128 * 6 + 5, d=128, ratio=128, overlap=True)
    got = _run(case, torch.float32, torch.float32)
    want = oracle.compress_kv(case.kv, case.score, case.ape, 128, True)
    assert np.abs(got - want).max() <= 1e-5


def test_rows_land_in_the_compressed_region_of_a_cache():
    # out = the rows win .. win + S/ratio - 1 of a [B, N, d] bf16 cache; the
    # window rows and the rows past the written ones keep their contents
    B, S, d, ratio, win, N = 3, 64, 128, 4, 16, 40
    case = W.compress_case(13, B=B, S=S, d=d, ratio=ratio, overlap=True, bf16=True)
    cache = torch.full((B, N, d), 7.0, dtype=torch.bfloat16, device="cuda")
    view = cache[:, win:win + S // ratio]
    sa.compress_kv(_dev(case.kv, torch.bfloat16), _dev(case.score, torch.bfloat16),
                   _dev(case.ape, torch.float32), ratio, True, out=view)
    sa.check_device()
    c = cache.float().cpu().numpy()
    want = oracle.compress_kv(case.kv, case.score, case.ape, ratio, True)
    assert np.abs(c[:, win:win + S // ratio] - want).max() <= 1e-2
    assert np.all(c[:, :win] == 7.0) and np.all(c[:, win + S // ratio:] == 7.0)


def test_decode_step_matches_prefill_row():
    # compressing the tokens of window w-1 and w alone gives row w of the prefill
    case = W.compress_case(14, B=2, S=4 * 50, d=128, ratio=4, overlap=True)
    full = _run(case, torch.float32, torch.float32)
    for w in (1, 17, 49):
        sl = slice((w - 1) * 4, (w + 1) * 4)
        part = W.CompressCase(kv=case.kv[:, sl], score=case.score[:, sl], ape=case.ape, ratio=4,
                              overlap=True)
        got = _run(part, torch.float32, torch.float32)
        assert np.array_equal(got[:, 1], full[:, w])


def test_fewer_tokens_than_a_window_write_nothing():
    case = W.compress_case(15, B=2, S=3, d=64, ratio=4, overlap=False)
    out = torch.full((2, 1, 64), 3.0, device="cuda")
    kv, score = _dev(case.kv, torch.float32), _dev(case.score, torch.float32)
    res = sa.compress_kv(kv, score, _dev(case.ape, torch.float32), 4, False)
    assert res.shape == (2, 0, 64)
    sa.check_device()
    assert torch.all(out == 3.0)


def test_full_size_sampled_windows():
    # the bench workload (8 sequences x 32768 tokens, ratio 4, overlap, fp32 in,
    # bf16 out), checked on sampled windows (each needs only its own and the
    # previous window's tokens)
    case = W.compress_case(0)
    got = _run(case, torch.float32, torch.bfloat16)
    n = case.kv.shape[1] // case.ratio
    rng = np.random.default_rng(0)
    for b in range(case.kv.shape[0]):
        for w in sorted(set(rng.integers(1, n, 6).tolist()) | {1, n - 1}):
            sl = slice((w - 1) * 4, (w + 1) * 4)
            want = oracle.compress_kv(case.kv[b:b + 1, sl], case.score[b:b + 1, sl], case.ape,
                                      4, True)[0, 1]
            assert np.abs(got[b, w] - want).max() <= 1e-2, (b, w)
        want0 = oracle.compress_kv(case.kv[b:b + 1, :4], case.score[b:b + 1, :4], case.ape, 4,
                                   True)[0, 0]
        assert np.abs(got[b, 0] - want0).max() <= 1e-2
