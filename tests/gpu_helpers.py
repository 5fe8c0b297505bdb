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


def compare(o_gpu, lse_gpu, o_ref, lse_ref, tol_o, tol_lse=TOL_LSE, what=""):
    """Element-wise comparison; lse -inf must match exactly.

    bf16 outputs may differ by tol_o plus their own final rounding."""
    import torch

    o = o_gpu.float().cpu().numpy().reshape(o_ref.shape).astype(np.float64)
    assert np.isfinite(o).all(), "%s: non-finite output" % what
    bound = tol_o + (BF16_OUT_REL * np.abs(o_ref) if o_gpu.dtype == torch.bfloat16 else 0.0)
    excess = np.abs(o - o_ref) - bound
    err = np.abs(o - o_ref).max() if o.size else 0.0
    assert (excess <= 0).all(), "%s: max |o - oracle| = %.3g beyond bound (tol %.1g)" % (
        what, err, tol_o)
    if lse_gpu is not None:
        l = lse_gpu.float().cpu().numpy().reshape(lse_ref.shape).astype(np.float64)
        inf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(l), inf_ref), "%s: -inf pattern of lse differs" % what
        fin = ~inf_ref
        lerr = np.abs(l[fin] - lse_ref[fin]).max() if fin.any() else 0.0
        assert lerr <= tol_lse, "%s: max |lse - oracle| = %.3g > %.1g" % (what, lerr, tol_lse)
        return err, lerr
    return err, 0.0
