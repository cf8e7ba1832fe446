"""The debug build (libefla_gb300_debug.so, compiled with -DEFLA_DEBUG): every global write
of the tensor-core kernels is checked tile by tile against its buffer, and a write outside
would be skipped and reported by efla_get_status as EFLA_ERR_BOUNDS.  The tensor-core
forward (fused, segment-parallel, recording), the backward (recomputing and from a record,
with a marked sequence and marked chunks) and the shared-memory-staged decode step run
through it with no violation and give the release library's results bit for bit."""
import pytest
import torch

import efla_workloads as wl
import exact_flow_recurrence_gb300 as efla

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def libs():
    return efla.load_library(), efla.load_library(efla.DEBUG_LIB_PATH)


def _with(lib, fn):
    """Run fn with the binding's calls routed to `lib`; the status must come back clean."""
    old = efla._lib
    efla._lib = lib
    try:
        out = fn()
        efla.efla_get_status()   # raises EflaError (EFLA_ERR_BOUNDS) on a skipped write
        return out
    finally:
        efla._lib = old


def _same(a, b):
    if isinstance(a, (tuple, list)):
        for x, y in zip(a, b):
            _same(x, y)
    elif a is not None:
        assert torch.equal(a, b)


def _dev(x):
    return {k: (v.to(DEV) if v is not None else None) for k, v in x.items()}


@pytest.mark.parametrize("L", [200, 4096])
def test_fused_forward_and_backward(libs, L):
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=3, L=L)
    x = _dev(wl.make_inputs(w))
    fwd = lambda: efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], x["S0"])   # noqa: E731
    bwd = lambda: efla.efla_bwd(x["q"], x["k"], x["v"], x["beta"], x["dO"], x["S0"])   # noqa: E731
    rel, dbg = libs
    _same(_with(rel, fwd), _with(dbg, fwd))
    _same(_with(rel, bwd), _with(dbg, bwd))


def test_segment_parallel_forward(libs):
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=2, L=16384)
    x = _dev(wl.make_inputs(w))
    fwd = lambda: efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], x["S0"], out_dtype=torch.float32)   # noqa: E731
    rel, dbg = libs
    _same(_with(rel, fwd), _with(dbg, fwd))


def test_recorded_training_with_marked_work(libs):
    """v of 1e5 in one sequence (fp32 recomputation of the forward, marked gradient chunks)
    and dO of 1e-5 in another (the reverse scan marks it): every fallback path writes."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=3, L=300)
    x = wl.make_inputs(w)
    x["v"][0, 1] = (x["v"][0, 1].double() * 1e5).to(w.dtype)
    x["dO"][0, 2] = (x["dO"][0, 2].double() * 1e-5).to(w.dtype)
    x = _dev(x)

    def step():
        o, Sf, rec = efla.efla_fwd_save(x["q"], x["k"], x["v"], x["beta"], x["S0"], out_dtype=torch.float32)
        g = efla.efla_bwd_saved(x["q"], x["k"], x["v"], x["beta"], x["dO"], rec, out_dtype=torch.float32)
        return (o, Sf, rec) + tuple(g)

    rel, dbg = libs
    _same(_with(rel, step), _with(dbg, step))


def test_decode_step(libs):
    """The shared-memory-staged decode step (dk = dv = 128): several steps from the same state
    through both libraries, bit for bit, with no bounds violation."""
    w = wl.resized(wl.DECODE, B=8, H=40)   # 320 sequences: every CTA cycles its stages
    ds = wl.DecodeStream(w)
    xs = [_dev(ds.next()) for _ in range(3)]
    rel, dbg = libs
    outs = []
    for lib in (rel, dbg):
        S = torch.zeros((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=DEV)
        os_ = [_with(lib, lambda x=x: efla.efla_step(x["q"], x["k"], x["v"], x["beta"], S)) for x in xs]
        outs.append((os_, S))
    _same(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])
