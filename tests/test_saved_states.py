"""Training with a recorded forward: efla_fwd_save writes every chunk's entering state S_c
and corrected values U' beside o and S_final; efla_bwd_saved computes the backward from
that record instead of re-running the state scan.  Against the fp64 oracle (gradients,
and S_c against the oracle's state after each chunk's prefix), on the tensor-core forward
(fused, segment-parallel, and the fp32 recomputation of an out-of-range sequence) and on
the fp32 CUDA-core path."""
import numpy as np
import pytest
import torch

import efla_workloads as wl
import exact_flow_recurrence_gb300 as efla
import oracle
from parity import TOL_BF16, TOL_F32, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
GRADS = ("dq", "dk", "dv", "dbeta", "dS0")


def _dev(x):
    return {k: (v.to(DEV) if v is not None else None) for k, v in x.items()}


def _dO(x, w):
    if x["dO"] is not None:
        return x["dO"]
    g = torch.Generator().manual_seed(99)
    return torch.randn(x["v"].shape, generator=g, dtype=torch.float64).to(w.dtype)


def _run(w, x, out_dtype, tol, heads, euler=False, check_states=True):
    x = dict(x)
    x["dO"] = _dO(x, w)
    d = _dev(x)
    mode = efla.EULER if euler else efla.EXACT
    o, Sf, rec = efla.efla_fwd_save(d["q"], d["k"], d["v"], d["beta"], d["S0"], chunk=w.chunk,
                                    out_dtype=out_dtype, mode=mode)
    o2, Sf2 = efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], chunk=w.chunk,
                            out_dtype=out_dtype, mode=mode)
    efla.efla_get_status()
    assert torch.equal(o, o2) and torch.equal(Sf, Sf2)       # recording changes no result
    grads = efla.efla_bwd_saved(d["q"], d["k"], d["v"], d["beta"], d["dO"], rec, None, chunk=w.chunk,
                                out_dtype=out_dtype, mode=mode)
    efla.efla_get_status()
    NC = (w.L + w.chunk - 1) // w.chunk
    Sc = rec[: w.B * w.H * NC * w.dk * w.dv].view(w.B, w.H, NC, w.dk, w.dv)
    for b, h in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        S0 = x["S0"][sl] if x["S0"] is not None else None
        ref = oracle.bwd(x["q"][sl], x["k"][sl], x["v"][sl], x["beta"][sl], x["dO"][sl], S0, euler=euler)
        for name, g_, r in zip(GRADS, grads, ref):
            assert_close(f"{name}[{b},{h}]", g_[sl], r, tol, stored_bf16=out_dtype == torch.bfloat16
                         and name in ("dq", "dk", "dv"))
        if check_states:   # the state entering chunk c = the oracle's state after c chunks
            for c in sorted({1, NC // 2, NC - 1}):
                if c < 1:
                    continue
                t = c * w.chunk
                cut = lambda a: a[sl][:, :, :t]   # noqa: E731
                _, S_ref = oracle.fwd(cut(x["q"]), cut(x["k"]), cut(x["v"]), cut(x["beta"]), S0, euler=euler)
                assert_close(f"S_c[{b},{h},{c}]", Sc[b, h, c], S_ref[0, 0], tol)
    return grads


def test_tensor_forward_record_ragged():
    w = wl.resized(wl.LM1P3B_FWDBWD, B=2, H=2, L=200)
    _run(w, wl.make_inputs(w), torch.float32, TOL_BF16, [(0, 0), (0, 1), (1, 0), (1, 1)])


def test_tensor_forward_record_euler_bf16_outputs():
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=2, L=257)
    _run(w, wl.make_inputs(w), torch.bfloat16, TOL_BF16, [(0, 0), (0, 1)], euler=True)


def test_saved_equals_recompute_backward():
    """Same gradients (within the bound) as the backward that recomputes the states."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=3, L=300)
    x = _dev(wl.make_inputs(w))
    _, _, rec = efla.efla_fwd_save(x["q"], x["k"], x["v"], x["beta"], x["S0"], out_dtype=torch.float32)
    gs = efla.efla_bwd_saved(x["q"], x["k"], x["v"], x["beta"], x["dO"], rec, out_dtype=torch.float32)
    gr = efla.efla_bwd(x["q"], x["k"], x["v"], x["beta"], x["dO"], x["S0"], out_dtype=torch.float32)
    efla.efla_get_status()
    for name, a, b in zip(GRADS, gs, gr):
        assert_close(name, a, b.double().cpu().numpy(), TOL_BF16)


def test_full_lm1p3b_recorded_training_step():
    """The full B4 H16 L4096 workload: forward with record, backward from it; oracle on two
    sequences."""
    w = wl.LM1P3B_FWDBWD
    _run(w, wl.make_inputs(w), torch.bfloat16, TOL_BF16, [(0, 3), (3, 14)], check_states=False)


def test_segment_parallel_forward_record():
    """B1 H2 L16384: the output pass of the segment-parallel form writes the record."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=2, L=16384)
    _run(w, wl.make_inputs(w), torch.float32, TOL_BF16, [(0, 1)])


def test_recomputed_sequence_writes_the_record():
    """A sequence the fp16 staging cannot hold (v of 1e5) is recomputed in fp32, record
    included; the other one keeps the tensor-core record."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=2, L=150)
    x = wl.make_inputs(w)
    x["v"][0, 1] = (x["v"][0, 1].double() * 1e5).to(w.dtype)
    _run(w, x, torch.float32, TOL_BF16, [(0, 0), (0, 1)])


def test_simt_forward_record():
    w = wl.resized(wl.TINY_FP32, B=1, H=2, L=90, dk=32, dv=32, chunk=32)
    _run(w, wl.make_inputs(w), torch.float32, TOL_F32, [(0, 0), (0, 1)])


def test_record_rejects_a_short_buffer():
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=1, L=100)
    x = _dev(wl.make_inputs(w))
    small = torch.empty(16, dtype=torch.float32, device=DEV)
    with pytest.raises(efla.EflaError, match="states"):
        efla.efla_fwd_save(x["q"], x["k"], x["v"], x["beta"], x["S0"], states=small)
    with pytest.raises(efla.EflaError, match="states"):
        efla.efla_bwd_saved(x["q"], x["k"], x["v"], x["beta"], x["dO"], small)


def test_recorded_backward_with_a_marked_sequence():
    """From a record the backward skips its preparation kernel; a sequence the tcgen05
    reverse scan marks (dO far below its fp16 range) gets its W and P prepared and its
    reverse scan redone in tf32.  Every sequence against the oracle."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=3, L=200)
    x = wl.make_inputs(w)
    x["dO"][0, 2] = (x["dO"][0, 2].double() * 1e-5).to(w.dtype)
    _run(w, x, torch.float32, TOL_BF16, [(0, 0), (0, 1), (0, 2)], check_states=False)


def test_record_holds_T_and_alpha():
    """The record's T and alpha blocks: T unit lower triangular, alpha = 0 past L; used by
    the backward in place of its own preparation."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=2, L=100)
    x = _dev(wl.make_inputs(w))
    _, _, rec = efla.efla_fwd_save(x["q"], x["k"], x["v"], x["beta"], x["S0"])
    efla.efla_get_status()
    NC, C = 2, 64
    al = lambda n: (n + 63) // 64 * 64   # noqa: E731  (256-byte alignment in floats)
    o_T = al(2 * NC * 128 * 128) + al(2 * NC * C * 128)
    o_a = o_T + al(2 * NC * C * C)
    T = rec[o_T:o_T + 2 * NC * C * C].view(2, NC, C, C).cpu()
    alpha = rec[o_a:o_a + 2 * NC * C].view(2, NC, C).cpu()
    assert torch.all(torch.diagonal(T, dim1=2, dim2=3) == 1.0)
    assert torch.all(torch.triu(T, 1) == 0)
    assert torch.all(alpha[:, 1, 100 - 64:] == 0) and torch.all(alpha[:, 0] > 0)
