"""GPU decode step (efla_step through the C ABI) vs the fp64 oracle, step after step."""
import numpy as np
import pytest
import torch

import efla_workloads as wl
import exact_flow_recurrence_gb300 as efla
import oracle
from parity import TOL_BF16, TOL_F32, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(w, steps, out_dtype, heads=None, euler=False, check_every=1):
    ds = wl.DecodeStream(w)
    S = torch.zeros((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=DEV)
    sel = heads or [(b, h) for b in range(w.B) for h in range(w.H)]
    bs = np.array([b for b, _ in sel])
    hs = np.array([h for _, h in sel])
    S_ref = np.zeros((len(sel), 1, w.dk, w.dv))
    tol = TOL_F32 if w.dtype == torch.float32 else TOL_BF16
    for t in range(steps):
        x = ds.next()
        o = efla.efla_step(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), x["beta"].to(DEV), S,
                           out_dtype=out_dtype, mode=efla.EULER if euler else efla.EXACT)
        # oracle on the sampled sequences, arranged as a [n,1,...] batch
        o_ref, S_ref = oracle.step(x["q"][bs, hs][:, None], x["k"][bs, hs][:, None],
                                   x["v"][bs, hs][:, None], x["beta"][bs, hs][:, None], S_ref,
                                   euler=euler)
        if t % check_every == 0 or t == steps - 1:
            assert_close(f"o[step {t}]", o[bs, hs][:, None], o_ref, tol,
                         stored_bf16=out_dtype == torch.bfloat16)
    efla.efla_get_status()
    assert_close("S_final", S[bs, hs][:, None], S_ref, tol)


@pytest.mark.parametrize("dv", [16, 32, 48, 64, 80, 96, 112, 128])
def test_value_widths(dv):
    w = wl.resized(wl.DECODE, B=3, H=2, dk=64, dv=dv)
    _run(w, 12, torch.float32)


def test_tiny_fp32_inputs_strict_tolerance():
    w = wl.resized(wl.DECODE, B=2, H=2, dk=16, dv=16, dtype=torch.float32)
    _run(w, 40, torch.float32)
    _run(w, 10, torch.float32, euler=True)


def test_bf16_outputs():
    _run(wl.resized(wl.DECODE, B=4, H=4), 20, torch.bfloat16)


def test_full_decode_sampled_heads():
    """Full B256 H16 d128 state (268 MB) through 1024 successive steps; oracle on 6 sequences."""
    _run(wl.DECODE, wl.DECODE.steps, torch.bfloat16,
         heads=[(0, 0), (17, 3), (100, 15), (128, 8), (200, 1), (255, 15)], check_every=64)


def test_d128_fp32_inputs_and_euler():
    """dk = dv = 128 (the shared-memory-staged step) with fp32 inputs and outputs."""
    w = wl.resized(wl.DECODE, B=2, H=3, dtype=torch.float32)
    _run(w, 16, torch.float32)
    _run(w, 8, torch.float32, euler=True)


def test_d128_many_sequences_per_sm():
    """1024 sequences: each persistent CTA of the staged step cycles its three stages several
    times per step; every sequence checked."""
    _run(wl.resized(wl.DECODE, B=64, H=16), 6, torch.float32)
