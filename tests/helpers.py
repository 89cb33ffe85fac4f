"""Shared comparison helpers for the GPU parity tests (no attention arithmetic here)."""
import math

import numpy as np
import torch

# Tolerances of the parity bar: bf16 inputs, fp32 accumulation, bf16 output.
TOL_O = 2e-2
TOL_LSE = 5e-3


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def assert_out_close(gpu, ref, tol=TOL_O, what="out"):
    g = to_np(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{what}: shape {g.shape} vs {r.shape}"
    assert np.isfinite(g).all(), f"{what}: non-finite values from the GPU"
    err = np.abs(g - r)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= tol, f"{what}: max |dO| = {worst:.3e} > {tol} at {np.unravel_index(err.argmax(), err.shape)}"
    return worst


def assert_lse_close(gpu, ref, tol=TOL_LSE, what="lse"):
    g = to_np(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{what}: shape {g.shape} vs {r.shape}"
    ninf_g, ninf_r = np.isneginf(g), np.isneginf(r)
    assert (ninf_g == ninf_r).all(), f"{what}: -inf pattern differs ({int(ninf_g.sum())} vs {int(ninf_r.sum())})"
    assert not np.isnan(g).any(), f"{what}: NaN from the GPU"
    fin = ~ninf_r
    worst = float(np.abs(g[fin] - r[fin]).max()) if fin.any() else 0.0
    assert worst <= tol, f"{what}: max |dLSE| = {worst:.3e} > {tol}"
    return worst


def dev():
    return torch.device("cuda", torch.cuda.current_device())
