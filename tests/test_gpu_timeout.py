"""GPU test of the bounded waits: every tensor-core kernel family takes its
timeout path once, on a tiny input, and the context stays usable.

With the test hook on (sattn_set_test_wait_stall) and a 2 ms wait limit, the
MMA-issuing thread of each launch waits for a barrier phase that nothing
completes. The wait runs out, the kernel records SATTN_ERR_TIMEOUT, every role
of the CTA stops, the copies and MMAs in flight drain (bounded) and tensor
memory is freed. The test then turns the hook off, restores the limit, and
checks that a normal call of the same family matches the oracle. No GPU
fault, trap or hang is involved: a wait that nothing satisfies returns an
error status (the XAttention stream-synchronisation page is about work that
waits on the wrong stream; here every wait is bounded instead).
"""
import numpy as np
import pytest
import torch

import oracle
import windowed_attention_sinks_gb300 as sa
from windowed_attention_sinks_gb300 import workloads as W

from gpu_helpers import TOL_BF16_O, compare, dev

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000  # copies in flight land within microseconds


def _window():
    case = W.window_vision_bf16(3, 8, num_seqs=2)
    q, k, v = (dev(x, torch.bfloat16) for x in (case.q, case.k, case.v))
    cu, s = dev(case.cu_seqlens, torch.int32), dev(case.sinks, torch.float32)

    def call():
        return sa.window_fwd(q, k, v, cu, case.max_seqlen, case.window_left, case.window_right,
                             False, s, sa.SINK_NULL_LOGIT, case.scale)

    def ref():
        return oracle.window(case.q, case.k, case.v, case.cu_seqlens, case.H, case.Hkv, case.d,
                             case.window_left, case.window_right, 0, case.sinks, 2, case.scale)
    return call, ref


def _block():
    case = W.block_sparse_bf16(1, Nctx=1024, M=256, chunk=512, density=0.4)
    q, k, v = (dev(x, torch.bfloat16) for x in (case.q, case.k, case.v))
    mask = dev(case.mask, torch.uint8)

    def call():
        return sa.block_sparse_fwd(q, k, v, mask, case.q_pos0, 0, case.Nctx, True, case.scale)

    def ref():
        return oracle.block_sparse(case.q, case.k, case.v, case.mask, case.q_pos0, 0, case.Nctx,
                                   1, case.scale)
    return call, ref


def _sparse(B):
    # B = 4: the cluster kernel; B = 100: the persistent kernel with split lists
    case = W.sparse_decode_bf16(4, B=B)
    q, kv = dev(case.q, torch.bfloat16), dev(case.kv, torch.bfloat16)
    idx, s = dev(case.idx, torch.int32), dev(case.sinks, torch.float32)
    ws = torch.empty(max(1, sa.sparse_workspace_bytes(case.B, case.M, case.H, case.d, case.K)),
                     dtype=torch.uint8, device="cuda")

    def call():
        return sa.sparse_fwd(q, kv, idx, s, case.sink_mode, case.scale, workspace=ws)

    def ref():
        return oracle.sparse(case.q, case.kv, case.idx, case.sinks, case.sink_mode, case.scale)
    return call, ref


def _sparse_fp8(B):
    # B = 4: the cluster kernel; B = 100: the persistent kernel with split lists
    case = W.sparse_decode_bf16(5, B=B)
    q, idx = dev(case.q, torch.bfloat16), dev(case.idx, torch.int32)
    s = dev(case.sinks, torch.float32)
    nope, rope, scl = sa.quantize_kv_fp8(dev(case.kv, torch.bfloat16), case.d // 2)
    torch.cuda.synchronize()
    # the kernel multiplies the rows as gathered: e4m3 value x scale rounded to bf16
    deq = oracle.bf16_round(oracle.dequantize_kv_fp8(
        nope.cpu().numpy(), rope.float().cpu().numpy(), scl.cpu().numpy()).astype(np.float32))

    ws = torch.empty(max(1, sa.sparse_workspace_bytes(case.B, case.M, case.H, case.d, case.K)),
                     dtype=torch.uint8, device="cuda")

    def call():
        return sa.sparse_fp8_fwd(q, nope, rope, scl, idx, s, case.sink_mode, case.scale,
                                 workspace=ws)

    def ref():
        return oracle.sparse(case.q, deq, case.idx, case.sinks, case.sink_mode, case.scale)
    return call, ref


def _xattn():
    rng = np.random.default_rng(9)
    M, Nctx, H, Hkv, d = 256, 768, 2, 1, 128
    q = W.round_bf16(rng.standard_normal((M, H, d)).astype(np.float32))
    k = W.round_bf16(rng.standard_normal((Nctx, Hkv, d)).astype(np.float32))
    qd, kd = dev(q, torch.bfloat16), dev(k, torch.bfloat16)

    def call():
        return sa.xattn_partial_stats(qd, kd, 512, 0, Nctx, True, d ** -0.5)

    def ref():
        return oracle.xattn_partial_stats(q, k, 512, 0, Nctx, True, d ** -0.5)
    return call, ref


FAMILIES = {"window": _window, "block": _block, "sparse_cluster": lambda: _sparse(4),
            "sparse_persistent": lambda: _sparse(100), "sparse_fp8_cluster": lambda: _sparse_fp8(4),
            "sparse_fp8_persistent": lambda: _sparse_fp8(100),
            "xattn_stats": _xattn}


@pytest.mark.parametrize("family", list(FAMILIES))
def test_wait_runs_out_and_context_recovers(family):
    call, ref = FAMILIES[family]()
    sa.check_device()
    try:
        sa.set_wait_limit_ns(LIMIT_NS)
        sa.set_test_wait_stall(True)
        call()
        with pytest.raises(sa.SattnError) as e:
            sa.check_device()
        assert e.value.code == 5, "expected SATTN_ERR_TIMEOUT, got %d" % e.value.code
    finally:
        sa.set_test_wait_stall(False)
        sa.set_wait_limit_ns(0)
    # the same call again, normally: the context is usable and the result right
    out = call()
    sa.check_device()
    want = ref()
    if family == "xattn_stats":
        m, l = (x.cpu().numpy() for x in out)
        wm, wl = want
        assert np.array_equal(np.isneginf(m), np.isneginf(wm))
        fin = np.isfinite(wm)
        assert np.abs(m[fin] - wm[fin]).max(initial=0) <= 1e-4
        assert np.abs(l[fin] - wl[fin]).max(initial=0) <= 1e-4 * np.abs(wl[fin]).max(initial=1)
    else:
        o, lse = out
        ro, rl = want
        compare(o, lse, ro, rl, TOL_BF16_O, what=family)
