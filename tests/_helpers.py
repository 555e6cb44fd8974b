"""Shared helpers for the GPU parity tests (no attention arithmetic here)."""

import numpy as np
import torch

OUT_TOL = 1e-2   # max |out - oracle|, fp32 output
LSE_TOL = 1e-3   # max |lse - oracle|


def dev():
    return torch.device("cuda:0")


def status_word():
    return torch.zeros(1, dtype=torch.int32, device=dev())


def to_np(t):
    return t.detach().cpu().double().numpy()


def max_err(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    fa, fb = np.isfinite(a), np.isfinite(b)
    assert np.array_equal(fa, fb), "finite / non-finite pattern differs"
    assert np.array_equal(a[~fa], b[~fb]), "non-finite values differ"
    return float(np.max(np.abs(a[fa] - b[fb]))) if fa.any() else 0.0


def assert_close(out, lse, ref_out, ref_lse, out_tol=OUT_TOL, lse_tol=LSE_TOL, what=""):
    eo = max_err(to_np(out) if torch.is_tensor(out) else out, ref_out)
    assert eo <= out_tol, f"{what}: max |out err| {eo:.3e} > {out_tol}"
    if lse is not None:
        el = max_err(to_np(lse) if torch.is_tensor(lse) else lse, ref_lse)
        assert el <= lse_tol, f"{what}: max |lse err| {el:.3e} > {lse_tol}"


def bf16_half_ulp(x):
    """Half a bf16 ulp of |x| (the rounding bound of a bf16 output)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 0.5 * 2.0 ** (e - 7)
