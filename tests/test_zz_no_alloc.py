"""efla_fwd_noalloc, the forward pass for callers that cannot allocate device memory
(plugins whose host application owns the allocator, real-time loops that may not
allocate once running): its scratch is the library's own device array, so the only
device memory the caller provides is inputs and outputs.

Both entry points run the same deterministic kernels, so efla_fwd_noalloc must return
exactly what efla_fwd (the entry point with a caller workspace) returns, bit for bit, on
two calls in a row with different inputs, since every call reuses the same array (the
second call runs on whatever the first one left there).  The cases cover the fused
tensor-core launch, whose image-ready flags live in the array; the segment-parallel form,
which also keeps its chained states and per-sequence out-of-range words there; and the
fp32 CUDA-core path.  This file is collected last on purpose."""
import ctypes

import pytest
import torch

import efla_workloads as wl
import exact_flow_recurrence_gb300 as efla

pytestmark = pytest.mark.gpu
DEV = "cuda"
NOALLOC_BYTES = 40 << 20


def _call_noalloc(lib, x, w, out_dtype):
    """Direct C-ABI call; o and S_final are allocated here, by the caller."""
    shape = efla.make_shape(w.B, w.H, w.L, w.dk, w.dv, w.chunk, w.dtype, out_dtype)
    o = torch.empty((w.B, w.H, w.L, w.dv), dtype=out_dtype, device=DEV)
    Sf = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=DEV)
    S0 = x["S0"]
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.efla_fwd_noalloc(ctypes.byref(shape), x["q"].data_ptr(), x["k"].data_ptr(),
                              x["v"].data_ptr(), x["beta"].data_ptr(),
                              S0.data_ptr() if S0 is not None else None, o.data_ptr(),
                              Sf.data_ptr(), stream)
    assert rc == 0, lib.efla_last_error().decode()
    return o, Sf


@pytest.mark.parametrize("base,out_dtype", [
    (wl.resized(wl.LM1P3B_FWDBWD, B=2, H=4, L=300), torch.bfloat16),
    (wl.resized(wl.LM1P3B_FWDBWD, B=1, H=2, L=16384), torch.bfloat16),
    (wl.resized(wl.TINY_FP32, B=1, H=3, L=100), torch.float32),
])
def test_noalloc_matches_efla_fwd_two_calls_in_a_row(base, out_dtype):
    lib = efla.load_library()
    shape = efla.make_shape(base.B, base.H, base.L, base.dk, base.dv, base.chunk, base.dtype,
                            out_dtype)
    need = efla.efla_fwd_workspace_size(shape)
    assert 0 < need <= NOALLOC_BYTES
    if base.L == 16384:   # segment-parallel: chained states follow the images and flags
        nc = base.L // 64
        assert need > base.B * base.H * nc * (4096 * 4 + 4 + 8)
    for seed in (101, 202):        # second call runs on scratch left by the first
        x = {k: (v.to(DEV) if v is not None else None)
             for k, v in wl.make_inputs(base, seed=seed).items()}
        o_na, S_na = _call_noalloc(lib, x, base, out_dtype)
        o_ref, S_ref = efla.efla_fwd(x["q"], x["k"], x["v"], x["beta"], x["S0"],
                                     chunk=base.chunk, out_dtype=out_dtype)
        efla.efla_get_status()
        assert torch.equal(o_na, o_ref), seed
        assert torch.equal(S_na, S_ref), seed


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = efla.load_library()
    shape = efla.make_shape(16, 16, 4096, 128, 128, 64, torch.bfloat16)
    assert efla.efla_fwd_workspace_size(shape) > NOALLOC_BYTES
    fake = 0x7f0000000000          # never dereferenced: the size check comes first
    rc = lib.efla_fwd_noalloc(ctypes.byref(shape), fake, fake + (1 << 30), fake + (2 << 30),
                              fake + (3 << 30), None, fake + (4 << 30), None, None)
    assert rc == 2                 # EFLA_ERR_UNSUPPORTED
    msg = lib.efla_last_error().decode()
    assert "EFLA_NOALLOC_SCRATCH_BYTES" in msg and str(NOALLOC_BYTES) in msg
