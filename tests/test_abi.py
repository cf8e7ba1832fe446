"""The C-ABI library builds, loads and exports every symbol include/efla.h declares;
host-side validation rejects bad arguments before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

import exact_flow_recurrence_gb300 as efla
from exact_flow_recurrence_gb300 import build as efla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "efla.h")


@pytest.fixture(scope="module")
def lib():
    efla_build.build()
    return efla.load_library()


def _declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(efla_[a-z_]+)\s*\(", txt)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"efla_fwd", "efla_bwd", "efla_step", "efla_get_status", "efla_status_string",
            "efla_fwd_workspace_size", "efla_bwd_workspace_size", "efla_last_error"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_debug_library_exports_the_same_symbols(lib):
    """The -DEFLA_DEBUG build (tile-level bounds checks) is a drop-in for the release one."""
    dbg = efla.load_library(efla.DEBUG_LIB_PATH)
    for n in _declared_functions():
        assert hasattr(dbg, n), n
    assert dbg.efla_status_string(7).decode() == "EFLA_ERR_BOUNDS"
    s = _shape(dk=128, dv=128, chunk=64)
    assert dbg.efla_bwd_workspace_size(ctypes.byref(s)) == lib.efla_bwd_workspace_size(ctypes.byref(s))


def test_status_strings(lib):
    for code, name in efla._STATUS.items():
        assert lib.efla_status_string(code).decode() == name


def _shape(**kw):
    base = dict(B=2, H=3, L=100, dk=64, dv=32, chunk=64, dtype=efla.BF16, out_dtype=efla.BF16,
                mode=efla.EXACT)
    base.update(kw)
    return efla.Shape(**base)


def test_workspace_size_positive_and_monotone(lib):
    s1 = lib.efla_fwd_workspace_size(ctypes.byref(_shape()))
    s2 = lib.efla_fwd_workspace_size(ctypes.byref(_shape(L=1000)))
    b1 = lib.efla_bwd_workspace_size(ctypes.byref(_shape()))
    assert 0 < s1 < s2 and b1 > s1
    assert lib.efla_fwd_workspace_size(ctypes.byref(_shape(dk=24))) == 0
    assert lib.efla_fwd_workspace_size(None) == 0


# Fake, never-dereferenced device addresses: validation must fail before any launch.
A = 0x7f0000000000


def _fwd(lib, shape, q=A, k=A + 0x10000000, v=A + 0x20000000, beta=A + 0x30000000, S0=None,
         o=A + 0x40000000, Sf=None, ws=A + 0x50000000, wsb=1 << 40):
    return lib.efla_fwd(ctypes.byref(shape) if shape is not None else None, q, k, v, beta, S0, o,
                        Sf, ws, wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(dk=24), 2),
    (dict(dv=144), 2),
    (dict(dk=8), 2),
    (dict(chunk=48), 2),
    (dict(chunk=128), 2),
    (dict(dtype=7), 2),
    (dict(mode=3), 2),
    (dict(B=-1), 1),
    (dict(L=-5), 1),
    (dict(L=64 * 65536), 2),
])
def test_fwd_rejects_bad_shapes(lib, kw, code):
    assert _fwd(lib, _shape(**kw)) == code
    assert lib.efla_last_error().decode() != ""


def test_fwd_rejects_bad_pointers(lib):
    s = _shape()
    assert _fwd(lib, None) == 1
    assert _fwd(lib, s, q=None) == 1
    assert _fwd(lib, s, o=None) == 1
    assert _fwd(lib, s, k=A + 8) == 3                       # misaligned
    assert _fwd(lib, s, S0=A + 0x60000004) == 3
    assert _fwd(lib, s, o=A + 0x20000000) == 1              # o aliases v
    assert _fwd(lib, s, ws=None) == 4                       # no workspace
    assert _fwd(lib, s, wsb=16) == 4                        # too small
    assert _fwd(lib, s, ws=A) == 1                          # workspace overlaps q
    # S_final may alias S0 exactly, but not partially
    assert _fwd(lib, s, S0=A + 0x60000000, Sf=A + 0x60000000 + 256, wsb=16) == 1


def test_step_rejects_bad_args(lib):
    s = _shape(L=2)
    args = [A, A + 0x1000000, A + 0x2000000, A + 0x3000000, A + 0x4000000, A + 0x5000000, None]
    assert lib.efla_step(ctypes.byref(s), *args) == 1       # L != 1
    s = _shape(L=1)
    bad = list(args)
    bad[4] = None                                            # S missing
    assert lib.efla_step(ctypes.byref(s), *bad) == 1
    bad = list(args)
    bad[5] = A + 0x4000000                                   # o aliases S
    assert lib.efla_step(ctypes.byref(s), *bad) == 1


def test_bwd_rejects_aliasing_outputs(lib):
    s = _shape()
    p = [A + i * 0x10000000 for i in range(12)]             # q .. dS0
    p[8] = p[7]                                              # dk aliases dq
    rc = lib.efla_bwd(ctypes.byref(s), *p, A + 0xF0000000, 1 << 40, None)
    assert rc == 1


def test_empty_batch_is_a_no_op(lib):
    assert _fwd(lib, _shape(B=0), q=None, k=None, v=None, beta=None, o=None) == 0


def _al(x):
    return (x + 255) // 256 * 256


def test_segment_parallel_workspace(lib):
    """Few long sequences take the segment-parallel tensor-core form, whose workspace adds
    three [B*H*nseg][128][128] fp32 state arrays, the chained final states [B*H][128][128]
    fp32 and one out-of-range word per sequence to the images, flags and per-chunk norm
    maxima; a chunk count that does not split evenly keeps the plain form."""
    def ws(L, H=16):
        return lib.efla_fwd_workspace_size(ctypes.byref(
            _shape(B=1, H=H, L=L, dk=128, dv=128, chunk=64)))
    bh, nc = 16, 65536 // 64
    plain = _al(bh * nc * 4096 * 4) + _al(bh * nc * 4) + _al(bh * nc * 8)
    assert ws(65536) == plain + 3 * _al(bh * 8 * 128 * 128 * 4) + _al(bh * 65536) + _al(bh * 4)   # 8 segments
    nc2 = 65472 // 64                                                     # 1023 chunks: odd
    assert ws(65472) == _al(bh * nc2 * 4096 * 4) + _al(bh * nc2 * 4) + _al(bh * nc2 * 8)
    nc3 = 16384 // 64                                                     # B*H = 2: 16 segments
    assert ws(16384, H=2) == _al(2 * nc3 * 4096 * 4) + _al(2 * nc3 * 4) + _al(2 * nc3 * 8) \
        + 3 * _al(2 * 16 * 65536) + _al(2 * 65536) + _al(2 * 4)
    nc4 = 8192 // 64                                                      # 128 chunks: too short
    assert ws(8192, H=2) == _al(2 * nc4 * 4096 * 4) + _al(2 * nc4 * 4) + _al(2 * nc4 * 8)


def test_path_selection_is_validated(lib):
    """efla_bwd and efla_step reject EFLA_PATH_TENSOR (the tcgen05 forward kernels) before
    any launch; the forward rejects TENSOR for shapes those kernels do not take; AUTO's
    backward workspace adds, to SIMT's, the tcgen05 reverse scan's images, flags, norms and
    out-of-range words."""
    p = [A + i * 0x10000000 for i in range(12)]
    s_tc = _shape(dk=128, dv=128, chunk=64, path=efla.TENSOR)
    assert lib.efla_bwd(ctypes.byref(s_tc), *p, A + 0xF0000000, 1 << 40, None) == 2
    assert lib.efla_bwd_workspace_size(ctypes.byref(s_tc)) == 0
    s_step = _shape(L=1, dk=128, dv=128, path=efla.TENSOR)
    assert lib.efla_step(ctypes.byref(s_step), A, A + 0x1000000, A + 0x2000000, A + 0x3000000,
                         A + 0x4000000, A + 0x5000000, None) == 2
    assert _fwd(lib, _shape(dk=64, dv=64, chunk=64, path=efla.TENSOR)) == 2   # not a tensor-core shape
    auto = lib.efla_bwd_workspace_size(ctypes.byref(_shape(dk=128, dv=128, chunk=64)))
    simt = lib.efla_bwd_workspace_size(ctypes.byref(_shape(dk=128, dv=128, chunk=64, path=efla.SIMT)))
    nch = 2 * 3 * 2            # B*H*NC of the default shape (L = 100)
    # tcgen05 reverse scan (Ta/P^T images, flags, norms, marked sequences with their count and
    # list, dSc and dU' fp16 images of 32 and 16 KB per chunk), then the tcgen05 gradient
    # kernel's list of chunks to recompute (count, indices) and the forward's per-sequence
    # record-format words
    assert auto == simt + _al(nch * 4096 * 2 * 2) + _al(nch * 4) + _al(nch * 8) + 2 * _al(2 * 3 * 4) + 256 \
        + _al(nch * 32768) + _al(nch * 16384) + 256 + _al(nch * 4) + _al(2 * 3 * 4) > simt > 0


def test_recorded_training_sizes_and_plan(lib):
    """The chunk-state record (S_c then U', fp32) and the backward that reads it: sizes, and
    the choice between recording and recomputing by the memory available (the faster form
    that fits: efla_bwd on one-pass tensor-core shapes, the recorded form elsewhere)."""
    s = _shape(B=4, H=16, L=4096, dk=128, dv=128, chunk=64)
    nc = 4096 // 64
    rec = lib.efla_fwd_states_size(ctypes.byref(s))
    assert rec == _al(64 * nc * 128 * 128 * 4) + _al(64 * nc * 64 * 128 * 4) + _al(64 * nc * 64 * 64 * 4) \
        + _al(64 * nc * 64 * 4)
    saved = lib.efla_bwd_saved_workspace_size(ctypes.byref(s))
    full = lib.efla_bwd_workspace_size(ctypes.byref(s))
    # the record's S_c and U' replace the backward's own Sc and Up arrays
    assert saved + _al(64 * nc * 128 * 128 * 4) + _al(64 * nc * 64 * 128 * 4) == full
    plan = lib.efla_bwd_plan
    plan.restype = ctypes.c_int
    plan.argtypes = [ctypes.POINTER(efla.Shape), ctypes.c_size_t]
    assert full < rec + saved          # the record also keeps T and alpha
    # one-pass tensor-core shape: efla_bwd first, the recorded form only where efla_bwd's
    # workspace does not fit (never here: it needs more)
    assert plan(ctypes.byref(s), rec + saved) == 0
    assert plan(ctypes.byref(s), full) == 0
    assert plan(ctypes.byref(s), full - 1) == -1
    # other shapes (here dv = 64, the tf32 backward): the recorded form first
    s64 = _shape(B=4, H=16, L=4096, dk=128, dv=64, chunk=64)
    rec64 = lib.efla_fwd_states_size(ctypes.byref(s64))
    saved64 = lib.efla_bwd_saved_workspace_size(ctypes.byref(s64))
    full64 = lib.efla_bwd_workspace_size(ctypes.byref(s64))
    assert plan(ctypes.byref(s64), rec64 + saved64) == 1
    if full64 < rec64 + saved64:
        assert plan(ctypes.byref(s64), rec64 + saved64 - 1) == 0
    assert plan(ctypes.byref(s64), min(full64, rec64 + saved64) - 1) == -1
    s2 = _shape(B=1, H=1, L=100, dk=32, dv=16, chunk=16)
    r2 = lib.efla_fwd_states_size(ctypes.byref(s2))
    assert r2 == _al(7 * 32 * 16 * 4) + _al(7 * 16 * 16 * 4) + _al(7 * 16 * 16 * 4) + _al(7 * 16 * 4)
    assert plan(ctypes.byref(_shape(chunk=48)), 1 << 40) == -1


def test_recorded_entry_points_validate_before_launch(lib):
    s = _shape(B=1, H=1, L=100, dk=32, dv=32, chunk=32)
    rec = lib.efla_fwd_states_size(ctypes.byref(s))
    ws = lib.efla_fwd_workspace_size(ctypes.byref(s))
    args = [A, A + (1 << 30), A + (2 << 30), A + (3 << 30), None, A + (4 << 30), None]
    # a record too small, then a misaligned one: rejected before any launch
    rc = lib.efla_fwd_save(ctypes.byref(s), *args, A + (5 << 30), rec - 1, A + (6 << 30), ws, None)
    assert rc == 1 and "states" in lib.efla_last_error().decode()
    rc = lib.efla_fwd_save(ctypes.byref(s), *args, A + (5 << 30) + 4, rec, A + (6 << 30), ws, None)
    assert rc == 3
    bws = lib.efla_bwd_saved_workspace_size(ctypes.byref(s))
    rc = lib.efla_bwd_saved(ctypes.byref(s), A, A + (1 << 30), A + (2 << 30), A + (3 << 30), None, rec,
                            A + (4 << 30), None, *(A + (i << 30) for i in range(5, 10)),
                            A + (10 << 30), bws, None)
    assert rc == 1 and "states" in lib.efla_last_error().decode()


def test_mixer_projection_validates_before_launch(lib):
    sh = efla.MixerShape
    bad = [sh(1, 100, 64, 2, 128),    # L not a multiple of 128
           sh(1, 128, 96, 2, 128),    # D not a multiple of 64
           sh(1, 128, 64, 3, 128),    # odd H
           sh(1, 128, 64, 34, 128),   # H > 32
           sh(1, 128, 64, 2, 64)]     # dk != 128
    for s in bad:
        assert lib.efla_mixer_proj(ctypes.byref(s), A, A + (1 << 30), A + (2 << 30), A + (3 << 30),
                                   A + (4 << 30), A + (5 << 30), None) == 2
    s = sh(1, 128, 64, 2, 128)
    assert lib.efla_mixer_proj(ctypes.byref(s), A, A + (1 << 30), A, A + (3 << 30), A + (4 << 30),
                               A + (5 << 30), None) == 1          # q overlaps x
    assert lib.efla_mixer_proj(ctypes.byref(s), A + 8, A + (1 << 30), A + (2 << 30), A + (3 << 30),
                               A + (4 << 30), A + (5 << 30), None) == 3
    assert lib.efla_mixer_proj(ctypes.byref(sh(0, 128, 64, 2, 128)), None, None, None, None, None, None,
                               None) == 0                          # empty: nothing to do
