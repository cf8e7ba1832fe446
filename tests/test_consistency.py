"""Cross-path consistency of the GPU entry points, edge cases, and failure handling."""
import numpy as np
import pytest
import torch

import efla_workloads as wl
import exact_flow_recurrence_gb300 as efla
import oracle
from parity import TOL_F32, assert_close, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(B=1, H=2, L=150, d=32, dtype=torch.float32, seed=5):
    w = wl.resized(wl.LM1P3B_FWDBWD, B=B, H=H, L=L, dk=d, dv=d, dtype=dtype, chunk=32)
    x = wl.make_inputs(w, seed=seed)
    return w, {k: (v.to(DEV) if v is not None else None) for k, v in x.items()}


def test_step_loop_equals_chunked_forward():
    w, x = _inputs()
    o, Sf = efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], x["S0"], chunk=32)
    S = x["S0"].clone()
    outs = []
    for t in range(w.L):
        outs.append(efla.efla_step(x["q"][:, :, t].contiguous(), x["k"][:, :, t].contiguous(),
                                   x["v"][:, :, t].contiguous(), x["beta"][:, :, t].contiguous(), S))
    o2 = torch.stack(outs, 2)
    assert rel_err(o2, o) < 1e-4 and rel_err(S, Sf) < 1e-4


def test_resume_chaining_and_in_place_state():
    w, x = _inputs(L=200)
    o, Sf = efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], x["S0"], chunk=32)
    L1 = 77
    cut = lambda t, a, b: t[:, :, a:b].contiguous()  # noqa: E731
    oa, Sa = efla.efla_fwd(cut(x["q"], 0, L1), cut(x["k"], 0, L1), cut(x["v"], 0, L1),
                           cut(x["beta"], 0, L1), x["S0"], chunk=32)
    S = Sa.clone()
    ob, _ = efla.efla_fwd(cut(x["q"], L1, 200), cut(x["k"], L1, 200), cut(x["v"], L1, 200),
                          cut(x["beta"], L1, 200), S, S_final=S, chunk=32)   # S0 aliases S_final
    assert rel_err(torch.cat([oa, ob], 2), o) < 1e-4
    assert rel_err(S, Sf) < 1e-4


def test_chunk_size_invariance():
    w, x = _inputs(L=130, d=64)
    res = [efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], x["S0"], chunk=c) for c in (16, 32, 64)]
    for o, Sf in res[1:]:
        assert rel_err(o, res[0][0]) < 1e-4 and rel_err(Sf, res[0][1]) < 1e-4


def test_bitwise_determinism():
    w, x = _inputs(B=2, H=2, L=300, d=128, dtype=torch.bfloat16)
    o1, S1 = efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], x["S0"])
    o2, S2 = efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], x["S0"])
    assert torch.equal(o1, o2) and torch.equal(S1, S2)
    dO = torch.randn_like(x["v"])
    g1 = efla.efla_bwd(x["q"], x["k"], x["v"], x["beta"], dO, x["S0"])
    g2 = efla.efla_bwd(x["q"], x["k"], x["v"], x["beta"], dO, x["S0"])
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_empty_inputs():
    _, x = _inputs(L=0)
    o, Sf = efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], x["S0"])
    torch.cuda.synchronize()
    assert o.numel() == 0 and torch.equal(Sf, x["S0"])
    o, Sf = efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(Sf) == 0
    dSf = torch.randn_like(x["S0"])
    g = efla.efla_bwd(x["q"], x["k"], x["v"], x["beta"], torch.empty_like(x["v"]), x["S0"], dSf)
    torch.cuda.synchronize()
    assert torch.equal(g[4], dSf)
    _, x = _inputs(B=0, L=10)
    o, Sf = efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], None)
    assert o.numel() == 0


def test_outputs_stay_in_bounds():
    """The kernels write exactly [B,H,L,dv] of o: a sentinel just past it survives."""
    w, x = _inputs(L=45, d=32)
    n = x["v"].numel()
    buf = torch.full((n + 1024,), 12345.0, device=DEV)
    o = buf[:n].view_as(x["v"])
    efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], x["S0"], o=o, chunk=32)
    torch.cuda.synchronize()
    assert torch.all(buf[n:] == 12345.0)
    assert torch.all(torch.isfinite(o))


def test_nan_propagates_without_trapping():
    w, x = _inputs(B=1, H=2, L=100)
    v = x["v"].clone()
    v[0, 1, 40, 3] = float("nan")
    o, Sf = efla.efla_fwd(x["q"], x["k"], v, x["beta"], x["S0"], chunk=32)
    efla.efla_get_status()                      # no device fault
    assert torch.all(torch.isfinite(o[0, 0])) and torch.all(torch.isfinite(Sf[0, 0]))
    assert torch.isnan(o[0, 1, 40:]).any()
    assert torch.all(torch.isfinite(o[0, 1, :32]))


def test_errors_raise_with_message():
    _, x = _inputs(d=32)
    with pytest.raises(efla.EflaError, match="chunk"):
        efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], chunk=48)
    with pytest.raises(efla.EflaError, match="workspace"):
        efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], workspace=torch.empty(1, device=DEV))


def test_euler_mode_matches_oracle_delta_rule():
    w = wl.resized(wl.TINY_FP32, B=1, H=2, L=70, dk=16, dv=16)
    xc = wl.make_inputs(w)
    d = {k: (v.to(DEV) if v is not None else None) for k, v in xc.items()}
    o, Sf = efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], None, chunk=16, mode=efla.EULER)
    o_ref, Sf_ref = oracle.fwd(xc["q"], xc["k"], xc["v"], xc["beta"], euler=True)
    assert_close("o", o, o_ref, TOL_F32)
    assert_close("S_final", Sf, Sf_ref, TOL_F32)
