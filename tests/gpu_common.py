"""Shared helpers of the GPU parity tests (CUDA path through the C ABI vs the oracle)."""

import numpy as np
import torch

# max-abs tolerances (out, lse).  bf16 and fp8 are the stated bars; fp32 is
# derived from fp32 accumulation over a few hundred tokens (errors ~1e-6).
TOL = {"f32": (1e-4, 1e-5), "bf16": (1e-2, 1e-3), "fp8": (3e-2, 3e-3)}


def tol_for(cfg):
    if cfg["kv_dtype"] == "fp8":
        return TOL["fp8"]
    return TOL[cfg["out_dtype"]]


def f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def assert_close_rows(out, lse, ref_out, ref_lse, tol, what=""):
    """Element-wise comparison; -inf LSE must match exactly (and outputs are then 0)."""
    to, tl = tol
    out = np.asarray(out, dtype=np.float64).reshape(ref_out.shape)
    lse = np.asarray(lse, dtype=np.float64).reshape(ref_lse.shape)
    ninf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), ninf), f"{what}: -inf pattern differs"
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    if ninf.any():
        assert np.all(out[ninf] == 0.0), f"{what}: empty rows must be zero"
    fin = ~ninf
    if fin.any():
        eo = np.abs(out[fin] - ref_out[fin]).max()
        el = np.abs(lse[fin] - ref_lse[fin]).max()
        assert eo <= to, f"{what}: max |out - oracle| = {eo:.3g} > {to}"
        assert el <= tl, f"{what}: max |lse - oracle| = {el:.3g} > {tl}"
        return eo, el
    return 0.0, 0.0
