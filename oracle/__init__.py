"""fp64 CPU oracle for Exact Flow Linear Attention (EFLA).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product package never imports this
module, and this module never imports the product package.

The arithmetic lives in ``efla_oracle.c`` (plain C, fp64, token by token);
this file only compiles it with gcc, loads it with ctypes and marshals numpy
arrays.  Source of the method: "Exact Flow Linear Attention: Exact Solution
from Continuous-Time Dynamics" (gist.science summary of arXiv 2512.12602),
page es, section "Metodologia", items 1-3 (ODE, rank-1 closed form, update
rule and alpha).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "efla_oracle.c")
_LIB = os.path.join(_HERE, "libefla_oracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile efla_oracle.c into libefla_oracle.so next to it (gcc, OpenMP if it links)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c99", _SRC, "-o", _LIB, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # no libgomp: build single-threaded
        subprocess.run(base, check=True, capture_output=True, text=True)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    i, d = ctypes.c_int, ctypes.c_double
    lib.efla_oracle_alpha.restype = d
    lib.efla_oracle_alpha.argtypes = [d, d, i]
    lib.efla_oracle_dalpha_dbeta.restype = d
    lib.efla_oracle_dalpha_dbeta.argtypes = [d, d, i]
    lib.efla_oracle_dalpha_dlambda.restype = d
    lib.efla_oracle_dalpha_dlambda.argtypes = [d, d, i]
    lib.efla_oracle_max_threads.restype = i
    lib.efla_oracle_max_threads.argtypes = []
    lib.efla_oracle_fwd.restype = i
    lib.efla_oracle_fwd.argtypes = [i, i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, _dp, i, i]
    lib.efla_oracle_step.restype = i
    lib.efla_oracle_step.argtypes = [i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, i, i]
    lib.efla_oracle_bwd.restype = i
    lib.efla_oracle_bwd.argtypes = [i, i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                    _dp, _dp, _dp, _dp, _dp, i, i]
    _lib = lib
    return lib


def _f64(x):
    """Contiguous fp64 numpy copy of an array-like (torch tensors included, any dtype)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: upcast exactly on the CPU
        import torch
        x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def alpha(beta: float, lam: float, euler: bool = False) -> float:
    """alpha = (1 - exp(-beta*lambda))/lambda (page es, Metodologia item 3); beta at lambda = 0."""
    return _load().efla_oracle_alpha(float(beta), float(lam), int(euler))


def dalpha_dbeta(beta: float, lam: float, euler: bool = False) -> float:
    return _load().efla_oracle_dalpha_dbeta(float(beta), float(lam), int(euler))


def dalpha_dlambda(beta: float, lam: float, euler: bool = False) -> float:
    return _load().efla_oracle_dalpha_dlambda(float(beta), float(lam), int(euler))


def max_threads() -> int:
    return _load().efla_oracle_max_threads()


def fwd(q, k, v, beta, S0=None, euler=False, nthreads=0):
    """Token-by-token forward.  q,k [B,H,L,dk]; v [B,H,L,dv]; beta [B,H,L]; S0 [B,H,dk,dv].

    Returns (o [B,H,L,dv], S_final [B,H,dk,dv]) as fp64 numpy arrays."""
    q, k, v, beta, S0 = map(_f64, (q, k, v, beta, S0))
    B, H, L, dk = k.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, L, dv))
    Sf = np.zeros((B, H, dk, dv))
    rc = _load().efla_oracle_fwd(B, H, L, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                 _ptr(S0), _ptr(o), _ptr(Sf), int(euler), int(nthreads))
    if rc:
        raise RuntimeError(f"efla_oracle_fwd failed ({rc})")
    return o, Sf


def step(q, k, v, beta, S, euler=False, nthreads=0):
    """One decode step.  q,k [B,H,dk]; v [B,H,dv]; beta [B,H]; S [B,H,dk,dv].

    Returns (o [B,H,dv], S_new [B,H,dk,dv]); the input S is not modified."""
    q, k, v, beta = map(_f64, (q, k, v, beta))
    Sn = _f64(S).copy()
    B, H, dk = k.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, dv))
    rc = _load().efla_oracle_step(B, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                  _ptr(Sn), _ptr(o), int(euler), int(nthreads))
    if rc:
        raise RuntimeError(f"efla_oracle_step failed ({rc})")
    return o, Sn


def bwd(q, k, v, beta, dO, S0=None, dS_final=None, euler=False, nthreads=0):
    """Reverse-mode gradient of sum(o*dO) + sum(S_final*dS_final).

    Returns (dq, dk, dv, dbeta, dS0) as fp64 numpy arrays."""
    q, k, v, beta, S0, dO, dSf = map(_f64, (q, k, v, beta, S0, dO, dS_final))
    B, H, L, dk = k.shape
    dv = v.shape[-1]
    dq = np.zeros((B, H, L, dk))
    dkk = np.zeros((B, H, L, dk))
    dvv = np.zeros((B, H, L, dv))
    db = np.zeros((B, H, L))
    dS0 = np.zeros((B, H, dk, dv))
    rc = _load().efla_oracle_bwd(B, H, L, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                 _ptr(S0), _ptr(dO), _ptr(dSf), _ptr(dq), _ptr(dkk),
                                 _ptr(dvv), _ptr(db), _ptr(dS0), int(euler), int(nthreads))
    if rc:
        raise RuntimeError(f"efla_oracle_bwd failed ({rc})")
    return dq, dkk, dvv, db, dS0


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
