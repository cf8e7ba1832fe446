"""Python binding of the EFLA GB300 library (libefla_gb300.so, C ABI in include/efla.h).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (torch supplies device memory and
the stream); each call passes ``data_ptr()`` values and the current stream to
the C entry point of the same name.  There is no fallback: if the compiled
library is missing or a call fails, an exception is raised.

Method (gist.science summary of arXiv 2512.12602, "Exact Flow Linear Attention:
Exact Solution from Continuous-Time Dynamics", page es, Metodologia item 3):
    S_t = (I - alpha_t k_t k_t^T) S_{t-1} + alpha_t k_t v_t^T,
    alpha_t = (1 - exp(-beta_t ||k_t||^2)) / ||k_t||^2,      o_t = S_t^T q_t.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "EflaError", "load_library", "library_path", "efla_fwd", "efla_fwd_noalloc", "efla_bwd",
    "efla_step",
    "efla_fwd_workspace_size", "efla_bwd_workspace_size", "efla_get_status",
    "efla_fwd_save", "efla_bwd_saved", "efla_fwd_states_size", "efla_bwd_saved_workspace_size",
    "efla_bwd_plan", "efla_mixer_proj", "MixerShape",
    "F32", "BF16", "EXACT", "EULER", "AUTO", "SIMT", "TENSOR", "efla_tc_selftest", "efla_wait_selftest",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libefla_gb300.so")
# the same library with -DEFLA_DEBUG: tile-level bounds checks on the tensor-core kernels'
# global writes (EFLA_ERR_BOUNDS from efla_get_status); built beside it by build.py
DEBUG_LIB_PATH = os.path.join(_HERE, "libefla_gb300_debug.so")

F32, BF16 = 0, 1
EXACT, EULER = 0, 1
AUTO, SIMT, TENSOR = 0, 1, 2
_STATUS = {0: "EFLA_OK", 1: "EFLA_ERR_INVALID_ARG", 2: "EFLA_ERR_UNSUPPORTED",
           3: "EFLA_ERR_ALIGNMENT", 4: "EFLA_ERR_WORKSPACE", 5: "EFLA_ERR_CUDA",
           6: "EFLA_ERR_TIMEOUT", 7: "EFLA_ERR_BOUNDS"}


class EflaError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS.get(status, status)}: {msg}")


class MixerShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("L", ctypes.c_int), ("D", ctypes.c_int), ("H", ctypes.c_int),
                ("dk", ctypes.c_int)]


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("L", ctypes.c_int),
                ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("chunk", ctypes.c_int),
                ("dtype", ctypes.c_int), ("out_dtype", ctypes.c_int), ("mode", ctypes.c_int),
                ("path", ctypes.c_int)]


_lib = None
_vp = ctypes.c_void_p


def library_path() -> str:
    return _LIB_PATH


def load_library(path: Optional[str] = None):
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} is missing: build it first (python -m exact_flow_recurrence_gb300.build)")
    lib = ctypes.CDLL(p)
    sp = ctypes.POINTER(Shape)
    lib.efla_fwd_workspace_size.restype = ctypes.c_size_t
    lib.efla_fwd_workspace_size.argtypes = [sp]
    lib.efla_bwd_workspace_size.restype = ctypes.c_size_t
    lib.efla_bwd_workspace_size.argtypes = [sp]
    lib.efla_fwd.restype = ctypes.c_int
    lib.efla_fwd.argtypes = [sp] + [_vp] * 8 + [ctypes.c_size_t, _vp]
    lib.efla_bwd.restype = ctypes.c_int
    lib.efla_bwd.argtypes = [sp] + [_vp] * 13 + [ctypes.c_size_t, _vp]
    lib.efla_fwd_states_size.restype = ctypes.c_size_t
    lib.efla_fwd_states_size.argtypes = [sp]
    lib.efla_bwd_saved_workspace_size.restype = ctypes.c_size_t
    lib.efla_bwd_saved_workspace_size.argtypes = [sp]
    lib.efla_bwd_plan.restype = ctypes.c_int
    lib.efla_bwd_plan.argtypes = [sp, ctypes.c_size_t]
    lib.efla_fwd_save.restype = ctypes.c_int
    lib.efla_fwd_save.argtypes = [sp] + [_vp] * 8 + [ctypes.c_size_t, _vp, ctypes.c_size_t, _vp]
    lib.efla_bwd_saved.restype = ctypes.c_int
    lib.efla_bwd_saved.argtypes = [sp] + [_vp] * 5 + [ctypes.c_size_t] + [_vp] * 8 + [ctypes.c_size_t, _vp]
    lib.efla_mixer_proj.restype = ctypes.c_int
    lib.efla_mixer_proj.argtypes = [ctypes.POINTER(MixerShape)] + [_vp] * 7
    lib.efla_fwd_noalloc.restype = ctypes.c_int
    lib.efla_fwd_noalloc.argtypes = [sp] + [_vp] * 8
    lib.efla_step.restype = ctypes.c_int
    lib.efla_step.argtypes = [sp] + [_vp] * 7
    lib.efla_wait_selftest.restype = ctypes.c_int
    lib.efla_wait_selftest.argtypes = [ctypes.c_int, ctypes.c_int, _vp]
    lib.efla_tc_selftest.restype = ctypes.c_int
    lib.efla_tc_selftest.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int] + [_vp] * 5
    lib.efla_get_status.restype = ctypes.c_int
    lib.efla_get_status.argtypes = [_vp]
    lib.efla_status_string.restype = ctypes.c_char_p
    lib.efla_status_string.argtypes = [ctypes.c_int]
    lib.efla_last_error.restype = ctypes.c_char_p
    lib.efla_last_error.argtypes = []
    if path is None:
        _lib = lib
    return lib


def _check(rc: int, where: str):
    if rc != 0:
        raise EflaError(rc, where, load_library().efla_last_error().decode())


def _dt(t: torch.dtype) -> int:
    if t == torch.float32:
        return F32
    if t == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t} (float32 or bfloat16)")


def _tdt(code: int) -> torch.dtype:
    return torch.bfloat16 if code == BF16 else torch.float32


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _out(t: Optional[torch.Tensor], shape, dtype: torch.dtype, device, name: str) -> torch.Tensor:
    """A caller-supplied output as given (its shape and dtype must be the ones the call
    writes), else a fresh one."""
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    if t.dtype != dtype or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")
    return t


def make_shape(B, H, L, dk, dv, chunk=64, dtype=torch.bfloat16, out_dtype=None,
               mode: int = EXACT, path: int = AUTO) -> Shape:
    out_dtype = dtype if out_dtype is None else out_dtype
    return Shape(B, H, L, dk, dv, chunk, _dt(dtype), _dt(out_dtype), mode, path)


def efla_fwd_workspace_size(shape: Shape) -> int:
    return load_library().efla_fwd_workspace_size(ctypes.byref(shape))


def efla_bwd_workspace_size(shape: Shape) -> int:
    return load_library().efla_bwd_workspace_size(ctypes.byref(shape))


def _workspace(nbytes: int, device, ws: Optional[torch.Tensor]) -> torch.Tensor:
    """The caller's workspace as given (the library checks its size), else a fresh one."""
    if ws is not None:
        return ws
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


def efla_fwd(q, k, v, beta, S0=None, *, chunk: int = 64, out_dtype=None, mode: int = EXACT,
             o=None, S_final=None, workspace=None, want_state: bool = True, stream=None,
             path: int = AUTO):
    """Chunked EFLA forward.  q,k [B,H,L,dk]; v [B,H,L,dv]; beta [B,H,L] fp32; S0 [B,H,dk,dv] fp32.

    Returns (o [B,H,L,dv], S_final [B,H,dk,dv] fp32 or None)."""
    B, H, L, dk = k.shape
    dv = v.shape[-1]
    shape = make_shape(B, H, L, dk, dv, chunk, q.dtype, out_dtype, mode, path)
    o = _out(o, (B, H, L, dv), _tdt(shape.out_dtype), q.device, "o")
    if S_final is not None or want_state:
        S_final = _out(S_final, (B, H, dk, dv), torch.float32, q.device, "S_final")
    ws = _workspace(efla_fwd_workspace_size(shape), q.device, workspace)
    rc = load_library().efla_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                 _ptr(S0), _ptr(o), _ptr(S_final), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "efla_fwd")
    return o, S_final


def efla_fwd_states_size(shape: Shape) -> int:
    return load_library().efla_fwd_states_size(ctypes.byref(shape))


def efla_bwd_saved_workspace_size(shape: Shape) -> int:
    return load_library().efla_bwd_saved_workspace_size(ctypes.byref(shape))


def efla_bwd_plan(shape: Shape, free_bytes: int) -> int:
    """1: record the forward's chunk states (efla_fwd_save + efla_bwd_saved); 0: recompute
    them (efla_fwd + efla_bwd); -1: neither fits in free_bytes."""
    return load_library().efla_bwd_plan(ctypes.byref(shape), free_bytes)


def efla_fwd_save(q, k, v, beta, S0=None, *, chunk: int = 64, out_dtype=None, mode: int = EXACT,
                  o=None, S_final=None, states=None, workspace=None, want_state: bool = True,
                  stream=None, path: int = AUTO):
    """efla_fwd that also records every chunk's entering state and corrected values for
    efla_bwd_saved.  Returns (o, S_final or None, states) with states a flat fp32 tensor
    of efla_fwd_states_size bytes."""
    B, H, L, dk = k.shape
    dv = v.shape[-1]
    shape = make_shape(B, H, L, dk, dv, chunk, q.dtype, out_dtype, mode, path)
    o = _out(o, (B, H, L, dv), _tdt(shape.out_dtype), q.device, "o")
    if S_final is not None or want_state:
        S_final = _out(S_final, (B, H, dk, dv), torch.float32, q.device, "S_final")
    nrec = efla_fwd_states_size(shape)
    if states is None:
        states = torch.empty(max(nrec // 4, 4), dtype=torch.float32, device=q.device)
    ws = _workspace(efla_fwd_workspace_size(shape), q.device, workspace)
    rc = load_library().efla_fwd_save(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                      _ptr(S0), _ptr(o), _ptr(S_final), _ptr(states),
                                      states.numel() * states.element_size(), _ptr(ws),
                                      ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "efla_fwd_save")
    return o, S_final, states


def efla_bwd_saved(q, k, v, beta, dO, states, dS_final=None, *, chunk: int = 64, out_dtype=None,
                   mode: int = EXACT, want_dS0: bool = True, workspace=None, stream=None,
                   path: int = AUTO):
    """efla_bwd from the record of efla_fwd_save (same shape, inputs and mode).
    Returns (dq, dk, dv, dbeta, dS0 or None)."""
    B, H, L, dk = k.shape
    dv = v.shape[-1]
    shape = make_shape(B, H, L, dk, dv, chunk, q.dtype, out_dtype, mode, path)
    odt = _tdt(shape.out_dtype)
    dq = torch.empty((B, H, L, dk), dtype=odt, device=q.device)
    dkk = torch.empty((B, H, L, dk), dtype=odt, device=q.device)
    dvv = torch.empty((B, H, L, dv), dtype=odt, device=q.device)
    db = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    dS0 = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device) if want_dS0 else None
    ws = _workspace(efla_bwd_saved_workspace_size(shape), q.device, workspace)
    rc = load_library().efla_bwd_saved(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                       _ptr(states), states.numel() * states.element_size(), _ptr(dO),
                                       _ptr(dS_final), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(db),
                                       _ptr(dS0), _ptr(ws), ws.numel() * ws.element_size(),
                                       _stream(stream))
    _check(rc, "efla_bwd_saved")
    return dq, dkk, dvv, db, dS0


def efla_mixer_proj(x, w, H: int, *, dk: int = 128, q=None, k=None, v=None, beta=None, stream=None):
    """The token mixer's input projections: x [B, L, D] bf16, w [3 H dk + H, D] bf16 ->
    q = (x Wq^T)/sqrt(dk), k, v [B, H, L, dk] bf16 and beta = sigmoid(x Wb^T) [B, H, L] fp32."""
    B, L, D = x.shape
    shape = MixerShape(B, L, D, H, dk)
    q = _out(q, (B, H, L, dk), torch.bfloat16, x.device, "q")
    k = _out(k, (B, H, L, dk), torch.bfloat16, x.device, "k")
    v = _out(v, (B, H, L, dk), torch.bfloat16, x.device, "v")
    beta = _out(beta, (B, H, L), torch.float32, x.device, "beta")
    rc = load_library().efla_mixer_proj(ctypes.byref(shape), _ptr(x), _ptr(w), _ptr(q), _ptr(k), _ptr(v),
                                        _ptr(beta), _stream(stream))
    _check(rc, "efla_mixer_proj")
    return q, k, v, beta


def efla_fwd_noalloc(q, k, v, beta, S0=None, *, chunk: int = 64, out_dtype=None,
                     mode: int = EXACT, o=None, S_final=None, want_state: bool = True,
                     stream=None, path: int = AUTO):
    """efla_fwd for callers that cannot allocate device memory: the scratch is the
    library's own device array (EFLA_NOALLOC_SCRATCH_BYTES), so no workspace is passed.
    Outputs (o, S_final) are still the caller's; pass them in to avoid any allocation here."""
    B, H, L, dk = k.shape
    dv = v.shape[-1]
    shape = make_shape(B, H, L, dk, dv, chunk, q.dtype, out_dtype, mode, path)
    o = _out(o, (B, H, L, dv), _tdt(shape.out_dtype), q.device, "o")
    if S_final is not None or want_state:
        S_final = _out(S_final, (B, H, dk, dv), torch.float32, q.device, "S_final")
    rc = load_library().efla_fwd_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v),
                                         _ptr(beta), _ptr(S0), _ptr(o), _ptr(S_final),
                                         _stream(stream))
    _check(rc, "efla_fwd_noalloc")
    return o, S_final


def efla_bwd(q, k, v, beta, dO, S0=None, dS_final=None, *, chunk: int = 64, out_dtype=None,
             mode: int = EXACT, want_dS0: bool = True, workspace=None, stream=None,
             path: int = AUTO):
    """Backward of efla_fwd.  Returns (dq, dk, dv, dbeta, dS0 or None).
    path=SIMT keeps every product in fp32 on the CUDA cores."""
    B, H, L, dk = k.shape
    dv = v.shape[-1]
    shape = make_shape(B, H, L, dk, dv, chunk, q.dtype, out_dtype, mode, path)
    odt = _tdt(shape.out_dtype)
    dq = torch.empty((B, H, L, dk), dtype=odt, device=q.device)
    dkk = torch.empty((B, H, L, dk), dtype=odt, device=q.device)
    dvv = torch.empty((B, H, L, dv), dtype=odt, device=q.device)
    db = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    dS0 = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device) if want_dS0 else None
    ws = _workspace(efla_bwd_workspace_size(shape), q.device, workspace)
    rc = load_library().efla_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                 _ptr(S0), _ptr(dO), _ptr(dS_final), _ptr(dq), _ptr(dkk),
                                 _ptr(dvv), _ptr(db), _ptr(dS0), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "efla_bwd")
    return dq, dkk, dvv, db, dS0


def efla_step(q, k, v, beta, S, *, out_dtype=None, mode: int = EXACT, o=None, stream=None):
    """One decode step, S [B,H,dk,dv] fp32 updated in place.  q,k [B,H,dk]; v [B,H,dv]; beta [B,H].

    Returns o [B,H,dv]."""
    B, H, dk = k.shape
    dv = v.shape[-1]
    shape = make_shape(B, H, 1, dk, dv, 1, q.dtype, out_dtype, mode)
    o = _out(o, (B, H, dv), _tdt(shape.out_dtype), q.device, "o")
    rc = load_library().efla_step(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                  _ptr(S), _ptr(o), _stream(stream))
    _check(rc, "efla_step")
    return o


def efla_tc_selftest(A, B, C, a_mn_major=False, b_mn_major=False, a_in_tmem=False, stream=None):
    """Diagnostic tile product on tcgen05: returns C + A B^T (A [128,K], B [N,K] fp16; C fp32).

    With a_mn_major / b_mn_major the operand is staged in the MN-major layout (the
    library is handed its transpose); with a_in_tmem, A is read from tensor memory."""
    N, K = B.shape
    D = torch.empty((128, N), dtype=torch.float32, device=A.device)
    a = A.t().contiguous() if a_mn_major else A
    b = B.t().contiguous() if b_mn_major else B
    flags = (1 if a_mn_major else 0) | (2 if b_mn_major else 0) | (4 if a_in_tmem else 0)
    rc = load_library().efla_tc_selftest(N, K, flags, _ptr(a), _ptr(b), _ptr(C), _ptr(D),
                                         _stream(stream))
    _check(rc, "efla_tc_selftest")
    return D


def efla_wait_selftest(kind, limit=4096, stream=None):
    """Diagnostic: a bounded device-side wait that must time out (kind 0: an mbarrier,
    kind 1: a global flag); the next efla_get_status raises EFLA_ERR_TIMEOUT."""
    _check(load_library().efla_wait_selftest(int(kind), int(limit), _stream(stream)), "efla_wait_selftest")


def efla_get_status(stream=None):
    """Synchronise the stream and raise on any asynchronous kernel error."""
    _check(load_library().efla_get_status(_stream(stream)), "efla_get_status")
