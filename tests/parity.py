"""Comparison helpers for GPU-vs-oracle parity tests.

Metric (per tensor): max |x_gpu - x_ref| / RMS(x_ref), with x_ref the fp64 oracle's
result on the same (already rounded) inputs.  Bounds: 1e-4 for fp32 inputs,
1e-2 for bf16 inputs with fp32 accumulation and state.

When the GPU result is *stored* in bf16, its own final rounding (at most half a
bf16 ulp, i.e. 2^-8 |x|) is not arithmetic error; it is allowed on top of the
bound, element by element:  |x_gpu - x_ref| <= tol * RMS + 2^-8 (|x_ref| + tol * RMS).
"""
from __future__ import annotations

import numpy as np
import torch

TOL_F32 = 1e-4
TOL_BF16 = 1e-2
BF16_HALF_ULP_REL = 2.0 ** -8


def to64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def rel_err(gpu, ref) -> float:
    g, r = to64(gpu), to64(ref)
    rms = float(np.sqrt(np.mean(r * r)))
    if rms == 0.0:
        return float(np.max(np.abs(g - r))) if g.size else 0.0
    return float(np.max(np.abs(g - r))) / rms if g.size else 0.0


def assert_close(name: str, gpu, ref, tol: float, stored_bf16: bool = False) -> float:
    g, r = to64(gpu), to64(ref)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values in GPU result"
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    err = np.abs(g - r)
    bound = tol * rms + (BF16_HALF_ULP_REL * (np.abs(r) + tol * rms) if stored_bf16 else 0.0)
    ok = err <= bound
    if not np.all(ok):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{name}: max|err|/rms = {err.max() / max(rms, 1e-300):.3e} > tol {tol:g}"
            f" (worst at {i}: gpu {g[i]:.6g} ref {r[i]:.6g}, rms {rms:.3g})")
    return float(err.max() / rms) if rms else 0.0
