"""The gate projections and rotary position embedding that feed the attention
paths (oracle side).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

* Gates ("Gated SA and SWA" section of the Stochastic Attention summary: the
  two paths are mixed through independent sigmoid projections).  The pages
  do not say what is projected; the plain reading is the layer input x of
  each token: a_sa = x W_sa^T + b_sa and a_swa = x W_swa^T + b_swa, one logit
  per (token, query head), the sigmoid applied where the paths merge.
* Rotary position embedding before the gather (the Fibonacci-attention page
  applies RoPE to queries and keys before gathering them; the SA pages are
  silent on positions).  RoPE rotates Q and K by each token's ORIGINAL index
  i, so the score of a pair depends on i - j whatever permutation later
  brings them into one window.  Convention (the pages give none): rotate
  halves -- for k < d/2, theta_k = base^(-2k/d) and the pair
  (x_k, x_{k+d/2}) is rotated by the angle i * theta_k.

All arithmetic is float64.
"""

from __future__ import annotations

import numpy as np


def gate_logits(x, w_sa, w_swa, b_sa=None, b_swa=None):
    """(a_sa, a_swa): logits [B, n, Hq] of the two independent gate
    projections of the layer input x [B, n, D] with weights [Hq, D] and
    optional biases [Hq]."""
    x = np.asarray(x, dtype=np.float64)
    out = []
    for w, b in ((w_sa, b_sa), (w_swa, b_swa)):
        a = np.einsum("bnd,hd->bnh", x, np.asarray(w, dtype=np.float64))
        if b is not None:
            a = a + np.asarray(b, dtype=np.float64)
        out.append(a)
    return out[0], out[1]


def rope_angles(n: int, d: int, base: float = 10000.0) -> np.ndarray:
    """Angles [n, d/2]: position i times theta_k = base^(-2k/d)."""
    if d % 2:
        raise ValueError("head_dim must be even")
    k = np.arange(d // 2, dtype=np.float64)
    theta = base ** (-2.0 * k / d)
    return np.arange(n, dtype=np.float64)[:, None] * theta[None, :]


def rope(x, base: float = 10000.0) -> np.ndarray:
    """x [B, n, H, d] rotated by each token's original index: for k < d/2,
    (x_k, x_{k+d/2}) -> (x_k cos a - x_{k+d/2} sin a, x_{k+d/2} cos a + x_k sin a)
    with a = i * theta_k."""
    x = np.asarray(x, dtype=np.float64)
    n, d = x.shape[1], x.shape[3]
    a = rope_angles(n, d, base)[None, :, None, :]
    c, s = np.cos(a), np.sin(a)
    lo, hi = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)
