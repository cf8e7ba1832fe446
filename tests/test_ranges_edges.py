"""Input range and edge cases of the tensor-core forward and the tensor-pipe backward,
against the fp64 oracle.

The tcgen05 forward stages its MMA operands in fp16.  A sequence whose values leave the
range that staging represents (large values overflow, tiny ones lose precision; the
bounds are stated beside kStageKMax in fwd_tc.cu), or whose outputs come out non-finite,
is recomputed token by token in fp32 inside the same call.  So the default path must give
the oracle's result for any finite input: large v, S0 and k, tiny v, q and k are checked
here, in the plain, segment-parallel and two-kernel forms.  Also: keys exactly zero
(lambda = 0, alpha = beta), negative beta, a NaN confined to its own sequence, outputs
written exactly inside their buffers, and full-size runs with fp32 outputs (no bf16
output rounding allowance)."""
import numpy as np
import pytest
import torch

import efla_workloads as wl
import exact_flow_recurrence_gb300 as efla
import oracle
from parity import TOL_BF16, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(x):
    return {k: (v.to(DEV) if v is not None else None) for k, v in x.items()}


def _scaled(w, scenario, seq=(0, 0), seed=None):
    """Workload inputs with one sequence pushed out of the fp16 staging range."""
    x = wl.make_inputs(w, seed=seed)
    b, h = seq
    f32 = lambda t: t.to(torch.float64)   # noqa: E731
    if scenario == "v_large":
        x["v"][b, h] = (f32(x["v"][b, h]) * 1e5).to(w.dtype)
    elif scenario == "S0_large":
        S0 = x["S0"] if x["S0"] is not None else torch.zeros((w.B, w.H, w.dk, w.dv))
        g = torch.Generator().manual_seed(5)
        S0[b, h] = 1e5 * torch.randn((w.dk, w.dv), generator=g)
        x["S0"] = S0
    elif scenario == "k_large":
        x["k"][b, h] = (f32(x["k"][b, h]) * 300.0).to(w.dtype)
    elif scenario == "v_tiny":     # v and S0 both tiny, so the whole state is
        x["v"][b, h] = (f32(x["v"][b, h]) * 1e-5).to(w.dtype)
        if x["S0"] is not None:
            x["S0"][b, h] *= 1e-5
    elif scenario == "q_tiny":
        x["q"][b, h] = (f32(x["q"][b, h]) * 1e-4).to(w.dtype)
    elif scenario == "k_tiny":
        x["k"][b, h] = (f32(x["k"][b, h]) * 1e-4).to(w.dtype)
    else:
        raise ValueError(scenario)
    return x


def _check_fwd(w, x, o, Sf, heads, tol=TOL_BF16):
    for b, h in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        S0 = x["S0"][sl] if x["S0"] is not None else None
        o_ref, Sf_ref = oracle.fwd(x["q"][sl], x["k"][sl], x["v"][sl], x["beta"][sl], S0)
        assert_close(f"o[{b},{h}]", o[sl], o_ref, tol)
        if Sf is not None:
            assert_close(f"S_final[{b},{h}]", Sf[sl], Sf_ref, tol)


SCENARIOS = ["v_large", "S0_large", "k_large", "v_tiny", "q_tiny", "k_tiny"]


@pytest.mark.parametrize("path", [efla.AUTO, efla.TENSOR])
@pytest.mark.parametrize("scenario", SCENARIOS)
def test_tensor_forward_out_of_staging_range(scenario, path):
    """B2 H2 L200 (fused launch): sequence (0,0) out of range, the others ordinary; every
    sequence against the oracle with fp32 outputs (plain 1e-2 bound)."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=2, H=2, L=200)
    x = _scaled(w, scenario)
    d = _dev(x)
    o, Sf = efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], chunk=64,
                          out_dtype=torch.float32, path=path)
    efla.efla_get_status()
    _check_fwd(w, x, o, Sf, [(b, h) for b in range(2) for h in range(2)])


def test_tensor_forward_out_of_range_resume_in_place():
    """A recomputed sequence still honours S_final aliasing S0 (S0 is read again by the
    recomputation, so S_final must not have been written before it)."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=2, L=150)
    x = _scaled(w, "v_large", seq=(0, 1))
    d = _dev(x)
    S = d["S0"].clone()
    o, _ = efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], S, chunk=64, out_dtype=torch.float32,
                         S_final=S)
    efla.efla_get_status()
    _check_fwd(w, x, o, S, [(0, 0), (0, 1)])


def test_two_kernel_form_out_of_range():
    """B*H = 144 leaves too few SMs for a fused launch: preparation kernel, then the
    sequence kernel; two sequences out of range (large v, tiny q)."""
    w = wl.resized(wl.LM340M_FWD, B=2, H=72, L=130)
    x = _scaled(w, "v_large", seq=(0, 3))
    x["q"][1, 70] = (x["q"][1, 70].to(torch.float64) * 1e-4).to(w.dtype)
    d = _dev(x)
    o, Sf = efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], None, chunk=64, out_dtype=torch.float32,
                          path=efla.TENSOR)
    efla.efla_get_status()
    _check_fwd(w, x, o, Sf, [(0, 3), (1, 70), (0, 0), (1, 71)])


@pytest.mark.parametrize("scenario", ["v_large", "k_large"])
def test_segment_parallel_form_out_of_range(scenario):
    """B1 H2 L16384 runs as 16 segments per sequence; head 1 out of range is recomputed
    whole, from its S0, after the segments ran; head 0 keeps the segment result."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=2, L=16384)
    x = _scaled(w, scenario, seq=(0, 1))
    d = _dev(x)
    S = d["S0"].clone()
    o, _ = efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], S, chunk=64, out_dtype=torch.float32,
                         S_final=S)
    efla.efla_get_status()
    _check_fwd(w, x, o, S, [(0, 0), (0, 1)])


def _zero_keys_negative_beta(w):
    x = wl.make_inputs(w)
    x["k"][0, 0, 5:9] = 0
    x["k"][0, 0, 100] = 0
    x["k"][0, 2, 64:128] = 0          # a whole chunk of zero keys
    g = torch.Generator().manual_seed(11)
    neg = -0.2 * torch.rand((w.L,), generator=g)
    x["beta"][0, 1, ::7] = neg[::7]   # every 7th token of head 1: beta in (-0.2, 0]
    return x


def test_tensor_paths_zero_keys_and_negative_beta():
    """lambda = 0 gives alpha = beta (the limit of the closed form); beta < 0 is accepted
    as given.  Forward on the tcgen05 kernels, backward on the tensor-pipe kernels."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=3, L=200)
    x = _zero_keys_negative_beta(w)
    d = _dev(x)
    o, Sf = efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], chunk=64,
                          out_dtype=torch.float32, path=efla.TENSOR)
    efla.efla_get_status()
    _check_fwd(w, x, o, Sf, [(0, 0), (0, 1), (0, 2)])
    grads = efla.efla_bwd(d["q"], d["k"], d["v"], d["beta"], d["dO"], d["S0"], None, chunk=64,
                          out_dtype=torch.float32)
    efla.efla_get_status()
    for h in range(3):
        sl = (slice(0, 1), slice(h, h + 1))
        ref = oracle.bwd(x["q"][sl], x["k"][sl], x["v"][sl], x["beta"][sl], x["dO"][sl], x["S0"][sl])
        for name, g_, r in zip(("dq", "dk", "dv", "dbeta", "dS0"), grads, ref):
            assert_close(f"{name}[0,{h}]", g_[sl], r, TOL_BF16)


def test_tensor_backward_large_values():
    """The tensor-pipe backward keeps fp32's exponent range (tf32 operands): v of 1e5 and
    an S0 of 1e5 in one sequence."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=2, L=150)
    x = _scaled(w, "v_large", seq=(0, 1))
    x["S0"][0, 1] *= 5e6
    d = _dev(x)
    grads = efla.efla_bwd(d["q"], d["k"], d["v"], d["beta"], d["dO"], d["S0"], None, chunk=64,
                          out_dtype=torch.float32)
    efla.efla_get_status()
    for h in range(2):
        sl = (slice(0, 1), slice(h, h + 1))
        ref = oracle.bwd(x["q"][sl], x["k"][sl], x["v"][sl], x["beta"][sl], x["dO"][sl], x["S0"][sl])
        for name, g_, r in zip(("dq", "dk", "dv", "dbeta", "dS0"), grads, ref):
            assert_close(f"{name}[0,{h}]", g_[sl], r, TOL_BF16)


def _nan_equal_close(name, gpu, ref, tol):
    g = gpu.detach().double().cpu().numpy()
    r = np.asarray(ref, dtype=np.float64)
    assert np.array_equal(np.isnan(g), np.isnan(r)), f"{name}: NaN pattern differs"
    fin = np.isfinite(r)
    rms = float(np.sqrt(np.mean(r[fin] ** 2)))
    assert np.all(np.isfinite(g[fin]))
    err = float(np.max(np.abs(g[fin] - r[fin]))) / rms
    assert err <= tol, f"{name}: {err:.3e}"


def test_tensor_forward_nan_stays_in_its_sequence():
    """One NaN in v (token 70, value column 5) of sequence (0,1): the other sequences are
    unaffected, and that sequence matches the oracle's NaN propagation exactly (only value
    column 5 from token 70 on) -- a non-finite output sends it to the fp32 recomputation."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=3, L=200)
    x = wl.make_inputs(w)
    x["v"][0, 1, 70, 5] = float("nan")
    d = _dev(x)
    o, Sf = efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], chunk=64,
                          out_dtype=torch.float32, path=efla.TENSOR)
    efla.efla_get_status()
    _check_fwd(w, x, o, Sf, [(0, 0), (0, 2)])
    sl = (slice(0, 1), slice(1, 2))
    o_ref, Sf_ref = oracle.fwd(x["q"][sl], x["k"][sl], x["v"][sl], x["beta"][sl], x["S0"][sl])
    assert np.isnan(o_ref[0, 0, 70:, 5]).all() and np.isfinite(o_ref[0, 0, :, :5]).all()
    _nan_equal_close("o[0,1]", o[sl], o_ref, TOL_BF16)
    _nan_equal_close("S_final[0,1]", Sf[sl], Sf_ref, TOL_BF16)
    grads = efla.efla_bwd(d["q"], d["k"], d["v"], d["beta"], d["dO"], d["S0"], None, chunk=64,
                          out_dtype=torch.float32)
    efla.efla_get_status()
    for h in (0, 2):
        sl = (slice(0, 1), slice(h, h + 1))
        ref = oracle.bwd(x["q"][sl], x["k"][sl], x["v"][sl], x["beta"][sl], x["dO"][sl], x["S0"][sl])
        for name, g_, r in zip(("dq", "dk", "dv", "dbeta", "dS0"), grads, ref):
            assert_close(f"{name}[0,{h}]", g_[sl], r, TOL_BF16)


# ------------------------------------------------------------------ guarded outputs
_MARGIN = 4096   # elements before and after each output (keeps 16-byte alignment)
_SENT = {torch.float32: (torch.int32, 0x7FC0DEAD), torch.bfloat16: (torch.int16, 0x7FCD)}


def _guarded(shape, dtype):
    """An output view inside a buffer prefilled with a NaN sentinel on both sides."""
    n = int(np.prod(shape))
    ity, bits = _SENT[dtype]
    buf = torch.full((n + 2 * _MARGIN,), bits, dtype=ity, device=DEV).view(dtype)
    return buf, buf[_MARGIN:_MARGIN + n].view(shape)


def _check_guard(name, buf, n, dtype):
    ity, bits = _SENT[dtype]
    raw = buf.view(ity)
    assert torch.all(raw[:_MARGIN] == bits) and torch.all(raw[_MARGIN + n:] == bits), \
        f"{name}: a write landed outside the output"
    inner = raw[_MARGIN:_MARGIN + n]
    assert not torch.any(inner == bits), f"{name}: some output elements were never written"
    assert torch.all(torch.isfinite(buf[_MARGIN:_MARGIN + n])), f"{name}: non-finite output"


@pytest.mark.parametrize("form,B,H,L,out_dtype", [
    ("fused", 2, 2, 200, torch.bfloat16),
    ("fused", 1, 3, 129, torch.float32),
    ("two-kernel", 2, 72, 130, torch.bfloat16),
    ("segment-parallel", 1, 2, 16384, torch.bfloat16),
])
def test_forward_outputs_written_exactly_in_place(form, B, H, L, out_dtype):
    w = wl.resized(wl.LM1P3B_FWDBWD, B=B, H=H, L=L)
    x = _dev(wl.make_inputs(w))
    ob, o = _guarded((B, H, L, 128), out_dtype)
    sb, Sf = _guarded((B, H, 128, 128), torch.float32)
    efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], x["S0"], chunk=64, o=o, S_final=Sf,
                  out_dtype=out_dtype, path=efla.TENSOR)
    efla.efla_get_status()
    _check_guard("o", ob, o.numel(), out_dtype)
    _check_guard("S_final", sb, Sf.numel(), torch.float32)


@pytest.mark.parametrize("dv,out_dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_backward_outputs_written_exactly_in_place(dv, out_dtype):
    """The four tensor-pipe backward kernels (bf16, d_k = 128, chunk 64, ragged tail)."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=2, L=200, dv=dv)
    x = _dev(wl.make_inputs(w))
    shape = efla.make_shape(1, 2, 200, 128, dv, 64, torch.bfloat16, out_dtype)
    ws = torch.empty(efla.efla_bwd_workspace_size(shape), dtype=torch.uint8, device=DEV)
    bufs = {n: _guarded(s, t) for n, s, t in (
        ("dq", (1, 2, 200, 128), out_dtype), ("dk", (1, 2, 200, 128), out_dtype),
        ("dv", (1, 2, 200, dv), out_dtype), ("dbeta", (1, 2, 200), torch.float32),
        ("dS0", (1, 2, 128, dv), torch.float32))}
    lib = efla.load_library()
    import ctypes
    rc = lib.efla_bwd(ctypes.byref(shape), x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                      x["beta"].data_ptr(), x["S0"].data_ptr(), x["dO"].data_ptr(), None,
                      *(bufs[n][1].data_ptr() for n in ("dq", "dk", "dv", "dbeta", "dS0")),
                      ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.efla_last_error().decode()
    efla.efla_get_status()
    for n, (buf, view) in bufs.items():
        _check_guard(n, buf, view.numel(), view.dtype)


# ----------------------------------------------------------- full size, fp32 outputs
def test_full_lm340m_fp32_outputs():
    """The benchmarked B8 H8 L2048 launch with fp32 outputs: the plain 1e-2 bound."""
    w = wl.LM340M_FWD
    x = wl.make_inputs(w)
    d = _dev(x)
    o, Sf = efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], None, chunk=64, out_dtype=torch.float32)
    efla.efla_get_status()
    _check_fwd(w, x, o, Sf, [(0, 0), (3, 5), (7, 7)])


def test_full_lm1p3b_fp32_outputs_fwd_and_bwd():
    w = wl.LM1P3B_FWDBWD
    x = wl.make_inputs(w)
    d = _dev(x)
    o, Sf = efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], chunk=64, out_dtype=torch.float32)
    efla.efla_get_status()
    _check_fwd(w, x, o, Sf, [(0, 0), (3, 15)])
    del o, Sf
    grads = efla.efla_bwd(d["q"], d["k"], d["v"], d["beta"], d["dO"], d["S0"], None, chunk=64,
                          out_dtype=torch.float32)
    efla.efla_get_status()
    for b, h in [(0, 3), (3, 14)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.bwd(x["q"][sl], x["k"][sl], x["v"][sl], x["beta"][sl], x["dO"][sl], x["S0"][sl])
        for name, g_, r in zip(("dq", "dk", "dv", "dbeta", "dS0"), grads, ref):
            assert_close(f"{name}[{b},{h}]", g_[sl], r, TOL_BF16)


@pytest.mark.parametrize("scale", [1e-5, 1e4])
def test_tensor_backward_gradient_scale_out_of_staging_range(scale):
    """The tcgen05 reverse scan stages dO and the state gradient in fp16: a sequence whose
    dO is far below (or whose gradients overflow) that range is marked and recomputed by the
    tf32 reverse scan; the other sequences keep the tensor-core result.  All against the
    oracle (fp32 outputs)."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=3, L=200)
    x = wl.make_inputs(w)
    x["dO"][0, 1] = (x["dO"][0, 1].double() * scale).to(w.dtype)
    d = _dev(x)
    grads = efla.efla_bwd(d["q"], d["k"], d["v"], d["beta"], d["dO"], d["S0"], None, chunk=64,
                          out_dtype=torch.float32)
    efla.efla_get_status()
    for h in range(3):
        sl = (slice(0, 1), slice(h, h + 1))
        ref = oracle.bwd(x["q"][sl], x["k"][sl], x["v"][sl], x["beta"][sl], x["dO"][sl], x["S0"][sl])
        for name, g_, r in zip(("dq", "dk", "dv", "dbeta", "dS0"), grads, ref):
            assert_close(f"{name}[0,{h}]", g_[sl], r, TOL_BF16)


def test_tensor_backward_two_kernel_form():
    """B*H = 144: the reverse scan's chunk preparation runs as its own kernel first."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=2, H=72, L=130)
    x = wl.make_inputs(w)
    d = _dev(x)
    grads = efla.efla_bwd(d["q"], d["k"], d["v"], d["beta"], d["dO"], d["S0"], None, chunk=64,
                          out_dtype=torch.float32)
    efla.efla_get_status()
    for b, h in [(0, 0), (1, 71)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.bwd(x["q"][sl], x["k"][sl], x["v"][sl], x["beta"][sl], x["dO"][sl], x["S0"][sl])
        for name, g_, r in zip(("dq", "dk", "dv", "dbeta", "dS0"), grads, ref):
            assert_close(f"{name}[{b},{h}]", g_[sl], r, TOL_BF16)


def test_tensor_backward_every_sequence_marked():
    """dO of 1e-5 in all 8 sequences: the tcgen05 reverse scan marks every one, so the tf32
    preparation walks its list of 8 x 64 chunks on a grid of two CTAs per SM (several chunks
    per CTA, shared memory reused) and the tf32 reverse scan redoes every sequence."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=8, L=4096)
    x = wl.make_inputs(w)
    x["dO"] = (x["dO"].double() * 1e-5).to(w.dtype)
    d = _dev(x)
    grads = efla.efla_bwd(d["q"], d["k"], d["v"], d["beta"], d["dO"], d["S0"], None, chunk=64,
                          out_dtype=torch.float32)
    efla.efla_get_status()
    for h in (0, 7):
        sl = (slice(0, 1), slice(h, h + 1))
        ref = oracle.bwd(x["q"][sl], x["k"][sl], x["v"][sl], x["beta"][sl], x["dO"][sl], x["S0"][sl])
        for name, g_, r in zip(("dq", "dk", "dv", "dbeta", "dS0"), grads, ref):
            assert_close(f"{name}[0,{h}]", g_[sl], r, TOL_BF16)


def test_tensor_backward_many_marked_chunks():
    """v of 1e5 over L = 16384: U' leaves fp16's range in the chunks of the gradient kernel,
    which lists them (up to 256, more than one per SM); the widening kernel and the tf32
    gradient kernel walk that list, several chunks per CTA."""
    w = wl.resized(wl.LM1P3B_FWDBWD, B=1, H=1, L=16384)
    x = _scaled(w, "v_large", seq=(0, 0))
    d = _dev(x)
    grads = efla.efla_bwd(d["q"], d["k"], d["v"], d["beta"], d["dO"], d["S0"], None, chunk=64,
                          out_dtype=torch.float32)
    efla.efla_get_status()
    ref = oracle.bwd(x["q"], x["k"], x["v"], x["beta"], x["dO"], x["S0"])
    for name, g_, r in zip(("dq", "dk", "dv", "dbeta", "dS0"), grads, ref):
        assert_close(name, g_, r, TOL_BF16)
