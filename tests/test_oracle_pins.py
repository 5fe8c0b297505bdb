"""Pins for the fp64 oracle against facts fixed by the pages and by mathematics.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, an off-by-one window, a sink in
the numerator) fails at least one of them:
  * hand-worked examples (tests/golden/hand_examples.json);
  * q = 0 closed forms, whose zero pattern recovers the visible key set;
  * sink reductions: key-0 bias with sink 0 and null logit with sink -inf are
    plain attention; very large sinks pin the limits;
  * the null-logit identity o_null = o_none * Z / (Z + e^s);
  * textbook special cases computed with torch (fp64, CPU): full attention,
    causal attention, dense attention over all rows, GQA via repeat_interleave;
  * -1 entries and list order do not change the sparse result;
  * chunked partials merged by LSE equal the one-shot result.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from windowed_attention_sinks_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")
MODES = {"none": 0, "key0_bias": 1, "null_logit": 2}


def _ev(x):
    """Evaluate a fixture expression: numbers, fractions, ln(...), -inf."""
    if isinstance(x, (int, float)):
        return float(x)
    if x == "-inf":
        return -math.inf
    return float(eval(x, {"__builtins__": {}}, {"ln": math.log}))


def _arr(x, dtype=np.float64):
    if isinstance(x, list):
        return np.array([_arr(e, dtype) for e in x], dtype=dtype)
    return _ev(x)


# ---------------------------------------------------------------- golden cases

def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_hand_examples(oracle_mod, case):
    tol = 1e-6
    if case["kind"] == "window":
        q, k, v = (_arr(case[n]).astype(np.float32) for n in ("q", "k", "v"))
        for mode, exp in case["expect"].items():
            sinks = _arr(exp["sinks"]).astype(np.float32) if "sinks" in exp else None
            o, lse = oracle_mod.window(q, k, v, case["cu_seqlens"], case["H"], case["Hkv"],
                                       case["d"], case["window"], case["window"], case["causal"],
                                       sinks, MODES[mode], 1.0)
            np.testing.assert_allclose(o, _arr(exp["o"]), atol=tol, rtol=0)
            np.testing.assert_allclose(lse, _arr(exp["lse"]), atol=tol, rtol=0)
    elif case["kind"] == "sparse":
        q, kv = _arr(case["q"]).astype(np.float32), _arr(case["kv"]).astype(np.float32)
        idx = np.array(case["idx"], dtype=np.int32)
        for mode, exp in case["expect"].items():
            sinks = _arr(exp["sinks"]).astype(np.float32) if "sinks" in exp else None
            o, lse = oracle_mod.sparse(q, kv, idx, sinks, MODES[mode], 1.0)
            np.testing.assert_allclose(o, _arr(exp["o"]), atol=tol, rtol=0)
            np.testing.assert_allclose(lse, _arr(exp["lse"]), atol=tol, rtol=0)
    elif case["kind"] == "block":
        q, k, v = (_arr(case[n]).astype(np.float32) for n in ("q", "k", "v"))
        mask = np.array(case["mask"], dtype=np.uint8)
        for ch in case["expect"]["chunks"]:
            o, lse = oracle_mod.block_sparse(q, k, v, mask, case["q_pos0"], ch["kv"][0],
                                             ch["kv"][1], case["causal"], 1.0, blk=case["blk"])
            np.testing.assert_allclose(o, _arr(ch["o"]), atol=tol, rtol=0)
            np.testing.assert_array_equal(np.isinf(lse), np.isinf(_arr(ch["lse"])))
            fin = np.isfinite(lse)
            np.testing.assert_allclose(lse[fin], _arr(ch["lse"])[fin], atol=tol, rtol=0)
    elif case["kind"] == "merge":
        op, lp = _arr(case["o_parts"]), _arr(case["lse_parts"])
        for mode, exp in case["expect"].items():
            sinks = _arr(exp["sinks"]).astype(np.float32) if "sinks" in exp else None
            o, lse = oracle_mod.merge(op, lp, case["H"], sinks)
            np.testing.assert_allclose(o, _arr(exp["o"]), atol=tol, rtol=0)
            np.testing.assert_allclose(lse, _arr(exp["lse"]), atol=tol, rtol=0)
    else:
        raise AssertionError(case["kind"])


# ---------------------------------------------------------------- helpers

def _rand_window(seed, lens, H, Hkv, d, std=1.0):
    rng = np.random.default_rng(seed)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    T = int(cu[-1])
    q = (rng.standard_normal((T, H, d)) * std).astype(np.float32)
    k = (rng.standard_normal((T, Hkv, d)) * std).astype(np.float32)
    v = rng.standard_normal((T, Hkv, d)).astype(np.float32)
    sinks = rng.standard_normal(H).astype(np.float32)
    return q, k, v, cu, sinks


def _torch_attention(q, k, v, scale, mask=None):
    """Textbook softmax attention with torch in fp64 (library routine).

    q[Lq,d], k/v[Lk,d]; mask[Lq,Lk] boolean (True = visible)."""
    qt, kt, vt = (torch.from_numpy(np.asarray(a, dtype=np.float64)) for a in (q, k, v))
    s = (qt @ kt.T) * scale
    if mask is not None:
        s = s.masked_fill(~torch.from_numpy(mask), -math.inf)
    lse = torch.logsumexp(s, dim=-1)
    return (torch.softmax(s, dim=-1) @ vt).numpy(), lse.numpy()


# ---------------------------------------------------------------- q = 0 closed forms

@pytest.mark.parametrize("wl,wr,causal", [(8, 8, 0), (0, 0, 0), (3, 5, 0), (7, 7, 1), (-1, 2, 0),
                                          (4, -1, 1), (-1, -1, 0)])
def test_window_zero_query_recovers_visible_set(oracle_mod, wl, wr, causal):
    """With q = 0 every visible key has weight 1/|S| and v_j = one-hot(j), so the
    support of o is exactly S. S is enumerated here from the pages' rule
    (same sequence, -wl <= j-i <= wr, j <= i if causal)."""
    lens = [5, 37, 1, 12]
    H, Hkv, d = 2, 1, 64
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    T = int(cu[-1])
    q = np.zeros((T, H, d), dtype=np.float32)
    k = np.random.default_rng(0).standard_normal((T, Hkv, d)).astype(np.float32)
    v = np.zeros((T, Hkv, d), dtype=np.float32)
    for s in range(len(lens)):
        for j in range(lens[s]):
            v[cu[s] + j, 0, j % d] = 1.0
    o, lse = oracle_mod.window(q, k, v, cu, H, Hkv, d, wl, wr, causal, None, 0, 0.125)
    o = o.reshape(T, H, d)
    lse = lse.reshape(T, H)
    for s in range(len(lens)):
        for i in range(lens[s]):
            S = [j for j in range(lens[s])
                 if (wl < 0 or j >= i - wl) and (wr < 0 or j <= i + wr) and (not causal or j <= i)]
            want = np.zeros(d)
            for j in S:
                want[j % d] += 1.0 / len(S)
            for h in range(H):
                np.testing.assert_allclose(o[cu[s] + i, h], want, atol=1e-14)
                assert abs(lse[cu[s] + i, h] - math.log(len(S))) < 1e-13


def test_window_zero_query_sink_closed_forms(oracle_mod):
    """q = 0: key-0 weight e^s/(e^s+|S|-1) when key 0 is visible; null logit gives
    every key 1/(|S|+e^s) and lse = ln(|S|+e^s)."""
    lens, w = [37], 8
    H, d = 3, 64
    cu = np.array([0, 37], dtype=np.int32)
    q = np.zeros((37, H, d), dtype=np.float32)
    k = np.random.default_rng(1).standard_normal((37, 1, d)).astype(np.float32)
    v = np.zeros((37, 1, d), dtype=np.float32)
    for j in range(37):
        v[j, 0, j] = 1.0
    sinks = np.array([0.7, -1.3, 2.5], dtype=np.float32)
    ok, lk = oracle_mod.window(q, k, v, cu, H, 1, d, w, w, 0, sinks, 1, 1.0)
    on, ln_ = oracle_mod.window(q, k, v, cu, H, 1, d, w, w, 0, sinks, 2, 1.0)
    ok, on = ok.reshape(37, H, d), on.reshape(37, H, d)
    lk, ln_ = lk.reshape(37, H), ln_.reshape(37, H)
    for i in range(37):
        S = list(range(max(0, i - w), min(36, i + w) + 1))
        for h in range(H):
            es = math.exp(float(sinks[h]))
            if 0 in S:
                Z = es + len(S) - 1
                assert abs(ok[i, h, 0] - es / Z) < 1e-14
                assert abs(lk[i, h] - math.log(Z)) < 1e-13
            else:
                assert abs(lk[i, h] - math.log(len(S))) < 1e-13
            Zn = len(S) + es
            for j in S:
                assert abs(on[i, h, j] - 1.0 / Zn) < 1e-14
            assert abs(ln_[i, h] - math.log(Zn)) < 1e-13


# ---------------------------------------------------------------- sink reductions

def test_sink_reductions_to_plain_attention(oracle_mod):
    """key-0 bias with sink 0 and null logit with sink -inf both equal no sink."""
    q, k, v, cu, _ = _rand_window(3, [5, 37, 64], 8, 4, 64)
    args = (q, k, v, cu, 8, 4, 64, 8, 8, 0)
    o0, l0 = oracle_mod.window(*args, None, 0, 0.125)
    ok, lk = oracle_mod.window(*args, np.zeros(8, np.float32), 1, 0.125)
    on, ln_ = oracle_mod.window(*args, np.full(8, -np.inf, np.float32), 2, 0.125)
    np.testing.assert_array_equal(ok, o0)
    np.testing.assert_array_equal(lk, l0)
    np.testing.assert_array_equal(on, o0)
    np.testing.assert_array_equal(ln_, l0)


def test_sink_large_limits(oracle_mod):
    """A huge key-0 sink makes rows that see key 0 copy v[key 0]; a huge null
    sink drives o to 0 and lse to the sink."""
    q, k, v, cu, _ = _rand_window(4, [5, 37], 8, 2, 64)
    T = int(cu[-1])
    big = np.full(8, 80.0, np.float32)
    ok, lk = oracle_mod.window(q, k, v, cu, 8, 2, 64, 8, 8, 0, big, 1, 0.125)
    on, ln_ = oracle_mod.window(q, k, v, cu, 8, 2, 64, 8, 8, 0, big, 2, 0.125)
    ok, on = ok.reshape(T, 8, 64), on.reshape(T, 8, 64)
    ln_ = ln_.reshape(T, 8)
    for s in range(2):
        for i in range(cu[s + 1] - cu[s]):
            t = cu[s] + i
            for h in range(8):
                if i <= 8:
                    np.testing.assert_allclose(ok[t, h], v[cu[s], h // 4], atol=1e-12)
                assert np.abs(on[t, h]).max() < 1e-20
                assert abs(ln_[t, h] - 80.0) < 1e-12


def test_null_logit_identity(oracle_mod):
    """o_null = o_none * Z / (Z + e^s) and lse_null = ln(e^lse_none + e^s)."""
    q, k, v, cu, sinks = _rand_window(5, [5, 37, 100], 8, 8, 64)
    args = (q, k, v, cu, 8, 8, 64, 16, 16, 0)
    o0, l0 = oracle_mod.window(*args, None, 0, 0.125)
    on, ln_ = oracle_mod.window(*args, sinks, 2, 0.125)
    s = np.tile(sinks.astype(np.float64), int(cu[-1]))
    Z = np.exp(l0)
    np.testing.assert_allclose(on, o0 * (Z / (Z + np.exp(s)))[:, None], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(ln_, np.log(Z + np.exp(s)), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- textbook special cases

def test_window_wider_than_sequence_is_full_attention(oracle_mod):
    lens = [5, 37, 64]
    q, k, v, cu, _ = _rand_window(6, lens, 8, 8, 32)
    o, lse = oracle_mod.window(q, k, v, cu, 8, 8, 32, 100, 100, 0, None, 0, 0.3)
    o, lse = o.reshape(-1, 8, 32), lse.reshape(-1, 8)
    for s in range(len(lens)):
        a, b = cu[s], cu[s + 1]
        for h in range(8):
            ref, rl = _torch_attention(q[a:b, h], k[a:b, h], v[a:b, h], 0.3)
            np.testing.assert_allclose(o[a:b, h], ref, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(lse[a:b, h], rl, rtol=1e-12, atol=1e-13)


def test_window_band_and_causal_match_torch_mask(oracle_mod):
    lens = [37, 70]
    q, k, v, cu, _ = _rand_window(7, lens, 4, 4, 32)
    for wl, wr, causal in [(8, 8, 0), (3, 11, 0), (16, 16, 1)]:
        o, _ = oracle_mod.window(q, k, v, cu, 4, 4, 32, wl, wr, causal, None, 0, 0.2)
        o = o.reshape(-1, 4, 32)
        for s in range(len(lens)):
            a, b = cu[s], cu[s + 1]
            L = b - a
            pos = torch.arange(L)
            diff = pos.view(1, -1) - pos.view(-1, 1)  # j - i
            m = (diff >= -wl) & (diff <= wr)
            if causal:
                m &= torch.ones(L, L, dtype=torch.bool).tril()
            for h in range(4):
                ref, _ = _torch_attention(q[a:b, h], k[a:b, h], v[a:b, h], 0.2, m.numpy())
                np.testing.assert_allclose(o[a:b, h], ref, rtol=1e-12, atol=1e-13)


def test_window_gqa_equals_repeat_interleave(oracle_mod):
    """GQA: head h reads KV head h // (H/Hkv), i.e. repeat_interleave of the KV heads."""
    q, k, v, cu, sinks = _rand_window(8, [5, 37], 8, 2, 64)
    kr = torch.from_numpy(k).repeat_interleave(4, dim=1).numpy()
    vr = torch.from_numpy(v).repeat_interleave(4, dim=1).numpy()
    for mode in (0, 1, 2):
        a = oracle_mod.window(q, k, v, cu, 8, 2, 64, 8, 8, 0, sinks, mode, 0.125)
        b = oracle_mod.window(q, kr, vr, cu, 8, 8, 64, 8, 8, 0, sinks, mode, 0.125)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


def test_sparse_all_rows_is_dense_attention(oracle_mod):
    rng = np.random.default_rng(9)
    B, M, H, d, N = 2, 3, 4, 32, 40
    q = rng.standard_normal((B, M, H, d)).astype(np.float32)
    kv = rng.standard_normal((B, N, d)).astype(np.float32)
    idx = np.tile(np.arange(N, dtype=np.int32), (B, M, 1))
    o, lse = oracle_mod.sparse(q, kv, idx, None, 0, 0.17)
    o, lse = o.reshape(B, M, H, d), lse.reshape(B, M, H)
    for b in range(B):
        for m in range(M):
            ref, rl = _torch_attention(q[b, m], kv[b], kv[b], 0.17)
            np.testing.assert_allclose(o[b, m], ref, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(lse[b, m], rl, rtol=1e-12, atol=1e-13)


def test_sparse_invalid_entries_and_order_are_irrelevant(oracle_mod):
    rng = np.random.default_rng(10)
    B, M, H, d, N, K = 2, 4, 4, 64, 300, 96
    q = rng.standard_normal((B, M, H, d)).astype(np.float32)
    kv = rng.standard_normal((B, N, d)).astype(np.float32)
    idx = rng.integers(0, N, size=(B, M, K)).astype(np.int32)
    idx[rng.random((B, M, K)) < 0.3] = -1
    sinks = rng.standard_normal(H).astype(np.float32)
    for mode in (0, 2):
        o, lse = oracle_mod.sparse(q, kv, idx, sinks, mode, 0.125)
        perm = idx[:, :, rng.permutation(K)]
        o2, l2 = oracle_mod.sparse(q, kv, perm, sinks, mode, 0.125)
        np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(l2, lse, rtol=1e-12, atol=1e-14)
        # dropping the -1 entries (compacted lists, padded at the end) changes nothing
        comp = np.full_like(idx, -1)
        for b in range(B):
            for m in range(M):
                valid = idx[b, m][idx[b, m] >= 0]
                comp[b, m, :len(valid)] = valid
        o3, l3 = oracle_mod.sparse(q, kv, comp, sinks, mode, 0.125)
        np.testing.assert_allclose(o3, o, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(l3, lse, rtol=1e-12, atol=1e-14)


def test_sparse_all_invalid_row(oracle_mod):
    """A list of only -1: o = 0, lse = -inf (no sink) or lse = sink (null logit)."""
    q = np.ones((1, 1, 2, 8), np.float32)
    kv = np.ones((1, 4, 8), np.float32)
    idx = np.full((1, 1, 5), -1, np.int32)
    sinks = np.array([0.5, -2.0], np.float32)
    o, lse = oracle_mod.sparse(q, kv, idx, sinks, 0, 1.0)
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    o, lse = oracle_mod.sparse(q, kv, idx, sinks, 2, 1.0)
    assert np.all(o == 0)
    np.testing.assert_allclose(lse, sinks.astype(np.float64), atol=1e-7)


def test_window_with_one_kv_head_equals_sparse_band_lists(oracle_mod):
    """Window attention with Hkv = 1 is gathered attention over each query's band."""
    lens = [5, 37, 20]
    H, d, w = 4, 32, 6
    q, k, v, cu, sinks = _rand_window(11, lens, H, 1, d)
    kv_same = k  # make key == value for the sparse view
    ow, lw = oracle_mod.window(q, kv_same, kv_same, cu, H, 1, d, w, w, 0, sinks, 2, 0.2)
    T = int(cu[-1])
    K = 2 * w + 1
    idx = np.full((1, T, K), -1, np.int32)
    for s in range(len(lens)):
        for i in range(lens[s]):
            band = [cu[s] + j for j in range(max(0, i - w), min(lens[s] - 1, i + w) + 1)]
            idx[0, cu[s] + i, :len(band)] = band
    os_, ls = oracle_mod.sparse(q[None], k[:, 0][None], idx, sinks, 2, 0.2)
    np.testing.assert_allclose(os_, ow, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ls, lw, rtol=1e-12, atol=1e-14)


def test_block_sparse_full_mask_is_causal_attention(oracle_mod):
    rng = np.random.default_rng(12)
    M, Nctx, H, Hkv, d, blk = 96, 256, 4, 2, 32, 32
    q_pos0 = Nctx - M
    q = rng.standard_normal((M, H, d)).astype(np.float32)
    k = rng.standard_normal((Nctx, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((Nctx, Hkv, d)).astype(np.float32)
    mask = np.ones((H, M // blk, Nctx // blk), np.uint8)
    o, lse = oracle_mod.block_sparse(q, k, v, mask, q_pos0, 0, Nctx, 1, 0.18, blk=blk)
    o, lse = o.reshape(M, H, d), lse.reshape(M, H)
    pos = np.arange(q_pos0, Nctx)[:, None]
    vis = np.arange(Nctx)[None, :] <= pos
    for h in range(H):
        ref, rl = _torch_attention(q[:, h], k[:, h // 2], v[:, h // 2], 0.18, vis)
        np.testing.assert_allclose(o[:, h], ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[:, h], rl, rtol=1e-12, atol=1e-13)


def test_block_sparse_mask_matches_torch_kron(oracle_mod):
    """Block mask expanded to token level with torch.kron (query blocks local,
    key blocks global), combined with causality."""
    rng = np.random.default_rng(13)
    M, Nctx, H, Hkv, d, blk = 64, 256, 2, 1, 16, 16
    q_pos0 = 160
    q = rng.standard_normal((M, H, d)).astype(np.float32)
    k = rng.standard_normal((Nctx, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((Nctx, Hkv, d)).astype(np.float32)
    mask = (rng.random((H, M // blk, Nctx // blk)) < 0.4).astype(np.uint8)
    for qb in range(M // blk):
        mask[:, qb, (q_pos0 // blk) + qb] = 1
    o, _ = oracle_mod.block_sparse(q, k, v, mask, q_pos0, 0, Nctx, 1, 0.25, blk=blk)
    o = o.reshape(M, H, d)
    causal = torch.arange(Nctx).view(1, -1) <= torch.arange(q_pos0, q_pos0 + M).view(-1, 1)
    for h in range(H):
        tok = torch.kron(torch.from_numpy(mask[h]).to(torch.int64),
                         torch.ones(blk, blk, dtype=torch.int64)).bool()
        ref, _ = _torch_attention(q[:, h], k[:, 0], v[:, 0], 0.25, (tok & causal).numpy())
        np.testing.assert_allclose(o[:, h], ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- merge

def test_chunked_merge_equals_one_shot(oracle_mod):
    case = W.block_sparse_bf16(0, Nctx=1024, M=256, H=4, Hkv=2, d=32, chunk=256, blk=64,
                               density=0.3)
    parts = [oracle_mod.block_sparse(case.q, case.k, case.v, case.mask, case.q_pos0, a, b, 1,
                                     case.scale, blk=case.blk) for a, b in case.chunks]
    o_parts = np.stack([p[0] for p in parts])
    lse_parts = np.stack([p[1] for p in parts])
    assert np.isneginf(lse_parts).any()  # some chunks see nothing for some rows
    om, lm = oracle_mod.merge(o_parts, lse_parts, case.H)
    o1, l1 = oracle_mod.block_sparse(case.q, case.k, case.v, case.mask, case.q_pos0, 0,
                                     case.Nctx, 1, case.scale, blk=case.blk)
    np.testing.assert_allclose(om, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lm, l1, rtol=1e-12, atol=1e-13)


def test_merge_with_sinks_equals_null_logit_one_shot(oracle_mod):
    """Chunks run without sinks, the null-logit term added once in the merge."""
    rng = np.random.default_rng(14)
    B, M, H, d, N, K = 1, 6, 4, 32, 200, 120
    q = rng.standard_normal((B, M, H, d)).astype(np.float32)
    kv = rng.standard_normal((B, N, d)).astype(np.float32)
    idx = rng.integers(0, N, size=(B, M, K)).astype(np.int32)
    idx[:, :, 100:] = -1  # the last chunk sees nothing
    sinks = rng.standard_normal(H).astype(np.float32)
    chunks = [(0, 40), (40, 80), (80, 120)]
    parts = [oracle_mod.sparse(q, kv, np.ascontiguousarray(idx[:, :, a:b]), None, 0, 0.2)
             for a, b in chunks]
    om, lm = oracle_mod.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]),
                              H, sinks)
    o1, l1 = oracle_mod.sparse(q, kv, idx, sinks, 2, 0.2)
    np.testing.assert_allclose(om, o1, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lm, l1, rtol=1e-12, atol=1e-14)


def test_merge_all_empty(oracle_mod):
    o, l = oracle_mod.merge(np.zeros((3, 2, 4)), np.full((3, 2), -np.inf), 2)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_threads_do_not_change_results(oracle_mod):
    q, k, v, cu, sinks = _rand_window(15, [37, 64, 5], 8, 4, 64)
    n0 = oracle_mod.get_threads()
    try:
        oracle_mod.set_threads(1)
        a = oracle_mod.window(q, k, v, cu, 8, 4, 64, 8, 8, 0, sinks, 1, 0.125)
        oracle_mod.set_threads(3)
        b = oracle_mod.window(q, k, v, cu, 8, 4, 64, 8, 8, 0, sinks, 1, 0.125)
    finally:
        oracle_mod.set_threads(0 if n0 <= 0 else n0)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_sampled_rows_match_full(oracle_mod):
    case = W.window_tiny_f32(0, 4)
    full = oracle_mod.window(case.q, case.k, case.v, case.cu_seqlens, case.H, case.Hkv, case.d,
                             8, 8, 0, case.sinks, 1, case.scale)
    rows = np.array([0, 7, 41 * 8 + 3, 100, 5 * 8], dtype=np.int64)
    part = oracle_mod.window(case.q, case.k, case.v, case.cu_seqlens, case.H, case.Hkv, case.d,
                             8, 8, 0, case.sinks, 1, case.scale, rows=rows)
    np.testing.assert_array_equal(part[0], full[0][rows])
    np.testing.assert_array_equal(part[1], full[1][rows])


# ---------------------------------------------------------------- pages' sanity (not a pin)

def test_sink_semantics_differ_on_tiny_workload(oracle_mod):
    """Sanity, not a pin: on the tiny 5/37-token workload dropping the sinks moves
    the output by O(1e-1) and swapping key-0 for null-logit semantics moves it
    noticeably too (the PR report quotes errors of this order)."""
    case = W.window_tiny_f32(0, 4)
    args = (case.q, case.k, case.v, case.cu_seqlens, case.H, case.Hkv, case.d, 8, 8, 0)
    ok, _ = oracle_mod.window(*args, case.sinks, 1, case.scale)
    o0, _ = oracle_mod.window(*args, None, 0, case.scale)
    on, _ = oracle_mod.window(*args, case.sinks, 2, case.scale)
    assert np.abs(ok - o0).max() > 1e-2
    assert np.abs(ok - on).max() > 1e-2
