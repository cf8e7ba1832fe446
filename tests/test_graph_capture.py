"""The tensor-core backward captured in a CUDA graph and replayed gives the eager results bit
for bit.  Captured: the chunk preparation, the recording forward and the reverse scan on two
streams (fork and join by events), the per-chunk gradients, and the list-driven fallbacks
after them, which are launched as programmatic dependents of the kernel before them.  The
marked scenarios make those fallbacks do work inside the graph."""
import pytest
import torch

import efla_workloads as wl
import exact_flow_recurrence_gb300 as efla

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(scenario):
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=4, L=1024)
    x = wl.make_inputs(w, seed=11)
    f64 = lambda t: t.to(torch.float64)   # noqa: E731
    if scenario == "dO_tiny_one_sequence":   # the reverse scan marks sequence 1 (tf32 redo)
        x["dO"][0, 1] = (f64(x["dO"][0, 1]) * 1e-5).to(w.dtype)
    elif scenario == "v_large_one_sequence":   # fp32 forward record and gradient chunks to redo
        x["v"][0, 2] = (f64(x["v"][0, 2]) * 1e5).to(w.dtype)
    return w, {k: (v.to(DEV) if v is not None else None) for k, v in x.items()}


@pytest.mark.parametrize("scenario", ["plain", "dO_tiny_one_sequence", "v_large_one_sequence"])
def test_backward_graph_replay_equals_eager(scenario):
    w, d = _inputs(scenario)
    args = (d["q"], d["k"], d["v"], d["beta"], d["dO"], d["S0"], None)
    kw = dict(chunk=64, out_dtype=torch.float32)
    eager = efla.efla_bwd(*args, **kw)
    efla.efla_get_status()
    shape = efla.make_shape(w.B, w.H, w.L, w.dk, w.dv, 64, w.dtype, torch.float32)
    ws = torch.empty(efla.efla_bwd_workspace_size(shape), dtype=torch.uint8, device=DEV)
    side = torch.cuda.Stream()   # warm-up off the default stream, then capture
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        efla.efla_bwd(*args, workspace=ws, **kw)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = efla.efla_bwd(*args, workspace=ws, **kw)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    efla.efla_get_status()
    for name, a, b in zip(("dq", "dk", "dv", "dbeta", "dS0"), out, eager):
        assert torch.equal(a, b), name


def test_fused_forward_graph_replay_tracks_new_inputs():
    """The fused forward (flag clearing, then the cooperative launch that depends on it)
    captured once and replayed on inputs rewritten in place between replays: every replay
    equals an eager call on the same inputs, so the image-ready flags are cleared again on
    each replay (stale flags would let the sequences take the previous replay's images)."""
    w = wl.resized(wl.LM340M_FWD, B=2, H=4, L=1024)
    xs = [wl.make_inputs(w, seed=s) for s in (21, 22)]
    d = {n: xs[0][n].to(DEV).clone() for n in ("q", "k", "v", "beta")}
    kw = dict(chunk=64)
    shape = efla.make_shape(w.B, w.H, w.L, w.dk, w.dv, 64, w.dtype, w.dtype)
    ws = torch.empty(efla.efla_fwd_workspace_size(shape), dtype=torch.uint8, device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], None, workspace=ws, **kw)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        o, S_final = efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], None, workspace=ws, **kw)
    for x in (xs[1], xs[0], xs[1]):
        for n in d:
            d[n].copy_(x[n])
        g.replay()
        torch.cuda.synchronize()
        efla.efla_get_status()
        o_e, S_e = efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], None, **kw)
        assert torch.equal(o, o_e) and torch.equal(S_final, S_e)
