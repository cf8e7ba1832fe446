"""fp64 oracle of the token mixer's input projections (TEST INFRASTRUCTURE ONLY: the
test suite and the benchmark's CPU-baseline leg are the only callers; the product
package never imports this module, and this module never imports the product).

The pages report EFLA inside 340M- and 1.3B-parameter language models (gist.science
summary of arXiv 2512.12602, page es, "Resultados Experimentales" item 1) without
printing the layer's equations.  The reading taken is the usual linear-attention layer:
per token x (d_model wide) and head h,
    q_h = (x Wq_h^T) / sqrt(dk),   k_h = x Wk_h^T,   v_h = x Wv_h^T,   beta_h = sigmoid(x wb_h)
with W = [Wq; Wk; Wv; Wb] stacked by output feature (a linear layer's weight).  The
definition is written out directly: one float64 matrix product (a library primitive),
the 1/sqrt(dk) scale, the logistic function, and the head-major reshape.
"""
from __future__ import annotations

import math

import numpy as np


def _f64(t) -> np.ndarray:
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


def mixer_proj(x, w, H: int, dk: int = 128):
    """x [B, L, D], w [3 H dk + H, D] -> q, k, v [B, H, L, dk] and beta [B, H, L] (float64)."""
    x64, w64 = _f64(x), _f64(w)
    B, L, D = x64.shape
    assert w64.shape == (3 * H * dk + H, D), w64.shape
    y = x64.reshape(B * L, D) @ w64.T                     # [B L, 3 H dk + H]

    def heads(cols):                                       # [B L, H dk] -> [B, H, L, dk]
        return cols.reshape(B, L, H, dk).transpose(0, 2, 1, 3).copy()
    q = heads(y[:, :H * dk]) / math.sqrt(dk)
    k = heads(y[:, H * dk:2 * H * dk])
    v = heads(y[:, 2 * H * dk:3 * H * dk])
    logit = y[:, 3 * H * dk:].reshape(B, L, H).transpose(0, 2, 1)
    beta = 1.0 / (1.0 + np.exp(-logit))
    return q, k, v, beta
