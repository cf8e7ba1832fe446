"""The token mixer's input projections on the tensor cores (efla_mixer_proj through the C
ABI) against the fp64 projection oracle: one tile, several tiles, more tiles than SMs
(each CTA walks several, reusing its two accumulators and output boxes), the full
340M- and 1.3B-layer widths (sampled tokens), and the projections feeding efla_fwd.

Tolerance: fp32 accumulation of exact bf16 products over d_model terms, then rounding
to bf16: max|err| <= 1e-3 RMS plus half a bf16 ulp of each element for q, k, v; beta is
stored in fp32 (absolute 1e-4 on a value in (0, 1))."""
import numpy as np
import pytest
import torch

import efla_workloads as wl
import exact_flow_recurrence_gb300 as efla
import oracle
from oracle.mixer import mixer_proj
from parity import TOL_BF16, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_PROJ = 1e-3


def _check(w, rows=None):
    x = wl.mixer_inputs(w)
    xd, wd = x["x"].to(DEV), x["w"].to(DEV)
    q, k, v, beta = efla.efla_mixer_proj(xd, wd, w.H)
    efla.efla_get_status()
    xs = x["x"] if rows is None else x["x"][:, rows]
    q_r, k_r, v_r, b_r = mixer_proj(xs, x["w"], w.H, w.dk)
    sel = (slice(None), slice(None), slice(None) if rows is None else rows)
    for name, g, r in (("q", q, q_r), ("k", k, k_r), ("v", v, v_r)):
        assert_close(name, g[sel], r, TOL_PROJ, stored_bf16=True)
    err = np.abs(beta[sel].double().cpu().numpy() - b_r).max()
    assert err <= 1e-4, err
    return xd, wd, q, k, v, beta


@pytest.mark.parametrize("B,L,D,H", [
    (1, 128, 64, 2),       # one token tile: three q/k/v column tiles and the beta tile
    (2, 256, 512, 4),      # several tiles of each kind
    (2, 2048, 256, 8),     # 416 tiles: more than one per CTA
    (1, 384, 192, 32),     # 32 heads (the most beta columns one tile holds), D not a power of 2
])
def test_projection_tiles(B, L, D, H):
    _check(wl.MixerWorkload("t", 5, B, L, D, H))


@pytest.mark.parametrize("w", [wl.MIXER_340M, wl.MIXER_1P3B])
def test_full_width_sampled_tokens(w):
    rows = [0, 1, 127, 128, 1000, w.L - 1]
    _check(w, rows=rows)


def test_projections_feed_the_forward():
    """x -> projections -> efla_fwd, against the oracle's projections (rounded to bf16 as
    the layer hands them on) and the oracle's recurrence."""
    w = wl.MixerWorkload("t", 6, 1, 256, 256, 2)
    xd, wd, q, k, v, beta = _check(w)
    o, Sf = efla.efla_fwd(q, k, v, beta, None, out_dtype=torch.float32)
    efla.efla_get_status()
    x = wl.mixer_inputs(w)
    q_r, k_r, v_r, b_r = mixer_proj(x["x"], x["w"], w.H, w.dk)
    bf = lambda a: torch.from_numpy(a).to(torch.bfloat16)   # noqa: E731
    o_ref, Sf_ref = oracle.fwd(bf(q_r), bf(k_r), bf(v_r), torch.from_numpy(b_r).float(), None)
    assert_close("o", o, o_ref, TOL_BF16)
    assert_close("S_final", Sf, Sf_ref, TOL_BF16)


def test_projection_rejects_unsupported_shapes():
    x = torch.empty((1, 100, 64), dtype=torch.bfloat16, device=DEV)
    w = torch.empty((3 * 2 * 128 + 2, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(efla.EflaError, match="L % 128"):
        efla.efla_mixer_proj(x, w, 2)
