"""Helpers shared by the GPU parity tests: device copies of workload tensors
and comparison against the oracle."""
import numpy as np
import torch

TOL_F32_O = 1e-4
TOL_BF16_O = 1e-2
TOL_LSE = 1e-3


def dev(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).cuda()


def tdtype(name):
    return torch.float32 if name == "f32" else torch.bfloat16


# Half an ulp of bf16, relative: the final round-to-nearest of o into bf16
# (the output has q's dtype) may add this on top of the computation error.
BF16_OUT_REL = 2.0 ** -8


# Every comparison's plain errors, for the end-of-run parity table that
# tests/conftest.py prints: (test, what, dtype, tol_o, max |o - oracle| with no
# rounding allowance, the largest share of tol_o that any element used after
# its allowance, max |lse - oracle|).
PARITY_LOG = []


def compare(o_gpu, lse_gpu, o_ref, lse_ref, tol_o, tol_lse=TOL_LSE, what=""):
    """Element-wise comparison; lse -inf must match exactly.

    bf16 outputs may differ by tol_o plus their own final rounding."""
    import os

    import torch

    o = o_gpu.float().cpu().numpy().reshape(o_ref.shape).astype(np.float64)
    assert np.isfinite(o).all(), "%s: non-finite output" % what
    allowance = BF16_OUT_REL * np.abs(o_ref) if o_gpu.dtype == torch.bfloat16 else 0.0
    diff = np.abs(o - o_ref)
    excess = diff - (tol_o + allowance)
    err = diff.max() if o.size else 0.0
    used = float(np.max(np.maximum(diff - allowance, 0.0)) / tol_o) if o.size else 0.0
    entry = [os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], what,
             str(o_gpu.dtype).replace("torch.", ""), tol_o, float(err), used, None]
    PARITY_LOG.append(entry)
    assert (excess <= 0).all(), "%s: max |o - oracle| = %.3g beyond bound (tol %.1g)" % (
        what, err, tol_o)
    if lse_gpu is not None:
        l = lse_gpu.float().cpu().numpy().reshape(lse_ref.shape).astype(np.float64)
        inf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(l), inf_ref), "%s: -inf pattern of lse differs" % what
        fin = ~inf_ref
        lerr = np.abs(l[fin] - lse_ref[fin]).max() if fin.any() else 0.0
        entry[6] = float(lerr)
        assert lerr <= tol_lse, "%s: max |lse - oracle| = %.3g > %.1g" % (what, lerr, tol_lse)
        return err, lerr
    return err, 0.0
