"""GPU chunked backward (efla_bwd through the C ABI) vs the fp64 oracle's reverse-mode
gradient of sum(o * dO) + sum(S_final * dS_final)."""
import pytest
import torch

import efla_workloads as wl
import exact_flow_recurrence_gb300 as efla
import oracle
from parity import TOL_BF16, TOL_F32, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check(w, out_dtype, dS_final=False, euler=False, heads=None):
    x = wl.make_inputs(w)
    if x["dO"] is None:
        g = torch.Generator().manual_seed(99)
        x["dO"] = torch.randn(x["v"].shape, generator=g, dtype=torch.float64).to(w.dtype)
    dSf = None
    if dS_final:
        g = torch.Generator().manual_seed(98)
        dSf = torch.randn((w.B, w.H, w.dk, w.dv), generator=g, dtype=torch.float64).float()
    d = {k: (v.to(DEV) if v is not None else None) for k, v in x.items()}
    dSf_d = dSf.to(DEV) if dSf is not None else None
    grads = efla.efla_bwd(d["q"], d["k"], d["v"], d["beta"], d["dO"], d["S0"], dSf_d,
                          chunk=w.chunk, out_dtype=out_dtype,
                          mode=efla.EULER if euler else efla.EXACT)
    efla.efla_get_status()
    tol = TOL_F32 if w.dtype == torch.float32 else TOL_BF16
    bf_out = out_dtype == torch.bfloat16
    sel = heads or [(b, h) for b in range(w.B) for h in range(w.H)]
    for b, h in sel:
        sl = (slice(b, b + 1), slice(h, h + 1))
        S0 = x["S0"][sl] if x["S0"] is not None else None
        ref = oracle.bwd(x["q"][sl], x["k"][sl], x["v"][sl], x["beta"][sl], x["dO"][sl], S0,
                         dSf[sl] if dSf is not None else None, euler=euler)
        for name, gg, r, stored in zip(("dq", "dk", "dv", "dbeta", "dS0"), grads, ref,
                                       (bf_out, bf_out, bf_out, False, False)):
            assert_close(f"{name}[{b},{h}]", gg[sl], r, tol, stored_bf16=stored)


def test_tiny_fp32():
    _check(wl.TINY_FP32, torch.float32)


def test_tiny_fp32_with_state_gradient_and_euler():
    w = wl.resized(wl.TINY_FP32, B=1, H=2, L=50)
    _check(w, torch.float32, dS_final=True)
    _check(w, torch.float32, dS_final=True, euler=True)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_lm1p3b_distribution_ragged(out_dtype):
    _check(wl.resized(wl.LM1P3B_FWDBWD, B=1, H=2, L=300), out_dtype, dS_final=True)


def test_stiff_distribution():
    _check(wl.resized(wl.STIFF_LONG, H=2, L=400), torch.float32)


@pytest.mark.parametrize("dk,dv,chunk,L", [(16, 16, 16, 37), (64, 32, 32, 100), (32, 80, 64, 70)])
def test_shapes_and_chunks(dk, dv, chunk, L):
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=1, L=L, dk=dk, dv=dv, chunk=chunk)
    _check(w, torch.float32, dS_final=True)


def test_full_lm1p3b_sampled_heads():
    """Full B4 H16 L4096 d128 fwd+bwd workload; oracle on 2 sequences."""
    _check(wl.LM1P3B_FWDBWD, torch.bfloat16, heads=[(0, 3), (3, 14)])


@pytest.mark.parametrize("dv,euler", [(64, False), (64, True), (128, True)])
def test_tensor_pipe_gradients_value_width_and_euler(dv, euler):
    """bf16 inputs at d_k = 128, chunk 64: the per-chunk gradients run on the tensor pipe
    (tf32 operands); one and two 64-column value slices, exact and Euler updates."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=2, L=200, dv=dv)
    _check(w, torch.bfloat16, dS_final=True, euler=euler)


def test_fp32_inputs_at_d128_stay_fp32():
    """fp32 inputs at d_k = 128, chunk 64 keep fp32 arithmetic (fp32 tolerance)."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=1, L=130, dtype=torch.float32)
    _check(w, torch.float32, dS_final=True)


def test_simt_path_keeps_fp32_products():
    """path=SIMT on a shape the tensor-pipe kernels take: every product stays fp32, so the
    gradients meet the fp32 bound even for bf16 inputs (outputs stored in fp32)."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=1, L=130)
    x = wl.make_inputs(w)
    g = torch.Generator().manual_seed(97)
    dO = torch.randn(x["v"].shape, generator=g, dtype=torch.float64).to(w.dtype)
    d = {k: (v.to(DEV) if v is not None else None) for k, v in x.items()}
    grads = efla.efla_bwd(d["q"], d["k"], d["v"], d["beta"], dO.to(DEV), d["S0"], None,
                          chunk=w.chunk, out_dtype=torch.float32, path=efla.SIMT)
    efla.efla_get_status()
    ref = oracle.bwd(x["q"], x["k"], x["v"], x["beta"], dO, x["S0"], None)
    for name, gg, r in zip(("dq", "dk", "dv", "dbeta", "dS0"), grads, ref):
        assert_close(name, gg, r, TOL_F32)
