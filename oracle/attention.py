"""SA, SWA, gated SA+SWA and full attention in fp64 (oracle side).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Every output row is computed from its definition, one ORIGINAL token i at a
time ("Stochastic Attention" summary, section "Core mechanism"): gather the
neighbour set N(i) (``graph.neighbours_sa`` / ``graph.neighbours_swa``), form
the scores s_j = scale * <Q[i], K[j]> for j in N(i), take a max-subtracted
softmax over them and return sum_j softmax(s)_j V[j].  Going through sigma^{-1}
per token is deliberately a different route from the kernels, which walk the
permuted sequence.

Layouts: Q [B, n, Hq, d]; K, V [B, n, Hkv, d]; sigma [B, n]; gate logits
[B, n, Hq] indexed by original token.  Query head hq reads kv head
hq // (Hq / Hkv) (grouped-query attention; the pages do not discuss GQA, the
standard grouping is used).  scale defaults to 1/sqrt(d) (the pages do not
state one).  All arithmetic is float64.
"""

from __future__ import annotations

import numpy as np

from .graph import neighbours_sa, neighbours_swa
from .prng import inverse_perm


def _as_f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def _head_map(hq: int, hkv: int) -> np.ndarray:
    """Query head hq reads kv head hq // g: the pages do not discuss GQA, and
    the standard grouping is used."""
    if hq % hkv != 0:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    return np.arange(hq) // (hq // hkv)


def _attend(qrow: np.ndarray, kb: np.ndarray, vb: np.ndarray, keys: np.ndarray,
            head_map: np.ndarray, scale: float) -> np.ndarray:
    """Softmax attention of one token's query heads over ``keys``: the
    standard attention that "Core mechanism", step 2 runs inside the window,
    with the maximum subtracted before exponentiating.

    qrow [Hq, d]; kb, vb [n, Hkv, d] (one sequence); returns [Hq, d].
    """
    kh = kb[keys][:, head_map, :]            # [m, Hq, d]
    vh = vb[keys][:, head_map, :]            # [m, Hq, d]
    s = scale * np.einsum("hd,mhd->hm", qrow, kh)
    s = s - s.max(axis=1, keepdims=True)
    e = np.exp(s)
    p = e / e.sum(axis=1, keepdims=True)
    return np.einsum("hm,mhd->hd", p, vh)


def _check(q, k, v):
    if q.ndim != 4 or k.shape != v.shape or k.ndim != 4:
        raise ValueError("expected Q [B,n,Hq,d] and K, V [B,n,Hkv,d]")
    if q.shape[0] != k.shape[0] or q.shape[1] != k.shape[1] or q.shape[3] != k.shape[3]:
        raise ValueError("Q and K/V shapes disagree")


def _rows(b_count: int, n: int, rows):
    if rows is None:
        return [(b, i) for b in range(b_count) for i in range(n)]
    return [(int(b), int(i)) for b, i in rows]


def sa_rows(q, k, v, perm, window: int, causal: bool, scale: float | None = None,
            rows=None) -> np.ndarray:
    """SA output rows Y[b, i] for the (b, i) pairs in ``rows`` -> [R, Hq, d].

    Steps 1-3 of "Core mechanism": permute by sigma, attend within the window
    |p - q| <= floor(w/2) in permuted space, scatter back by sigma^{-1}; the
    causal variant also requires sigma(q) <= sigma(p).
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    _check(q, k, v)
    bsz, n, hq, d = q.shape
    perm = np.asarray(perm, dtype=np.int64).reshape(bsz, n)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    hm = _head_map(hq, k.shape[2])
    invs = {}
    out = []
    for b, i in _rows(bsz, n, rows):
        if b not in invs:
            invs[b] = inverse_perm(perm[b])
        keys = neighbours_sa(perm[b], window, causal, i, invs[b])
        out.append(_attend(q[b, i], k[b], v[b], keys, hm, scale))
    return np.asarray(out).reshape(-1, hq, d)


def swa_rows(q, k, v, window: int, scale: float | None = None, rows=None) -> np.ndarray:
    """SWA output rows over keys [max(0, i-w+1), i] -> [R, Hq, d]
    ("Problem statement": a local window of size w)."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    _check(q, k, v)
    bsz, n, hq, d = q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    hm = _head_map(hq, k.shape[2])
    out = []
    for b, i in _rows(bsz, n, rows):
        keys = neighbours_swa(n, window, i)
        out.append(_attend(q[b, i], k[b], v[b], keys, hm, scale))
    return np.asarray(out).reshape(-1, hq, d)


def sigmoid(x) -> np.ndarray:
    """The gates' sigmoid of the "Gated SA and SWA" equation, in fp64
    (overflow of e^{-x} correctly gives 0)."""
    x = _as_f64(x)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-x))


def gated_rows(q, k, v, perm, gate_sa, gate_swa, window: int, window_swa: int | None = None,
               causal: bool = True, scale: float | None = None, rows=None) -> np.ndarray:
    """Gated dual path ("Gated SA and SWA" section equation):
        Y = g_sa * Y_sa + g_swa * Y_swa,  g = sigmoid(logit),
    with per-token, per-query-head logits broadcast over d -> [R, Hq, d]."""
    q = _as_f64(q)
    bsz, n, hq, _ = q.shape
    w_swa = window if (window_swa is None or window_swa <= 0) else window_swa
    rws = _rows(bsz, n, rows)
    y_sa = sa_rows(q, k, v, perm, window, causal, scale, rws)
    y_swa = swa_rows(q, k, v, w_swa, scale, rws)
    gs = _as_f64(gate_sa).reshape(bsz, n, hq)
    gw = _as_f64(gate_swa).reshape(bsz, n, hq)
    bi = np.asarray(rws, dtype=np.int64).reshape(-1, 2)
    g1 = sigmoid(gs[bi[:, 0], bi[:, 1]])[:, :, None]
    g2 = sigmoid(gw[bi[:, 0], bi[:, 1]])[:, :, None]
    return g1 * y_sa + g2 * y_swa


def _full(rows_fn, q):
    bsz, n, hq, d = np.shape(q)
    return rows_fn().reshape(bsz, n, hq, d)


def sa_forward(q, k, v, perm, window: int, causal: bool, scale: float | None = None) -> np.ndarray:
    """Full SA output [B, n, Hq, d] (all rows; "Core mechanism", steps 1-3)."""
    return _full(lambda: sa_rows(q, k, v, perm, window, causal, scale), q)


def swa_forward(q, k, v, window: int, scale: float | None = None) -> np.ndarray:
    """Full SWA output [B, n, Hq, d] ("Problem statement")."""
    return _full(lambda: swa_rows(q, k, v, window, scale), q)


def gated_forward(q, k, v, perm, gate_sa, gate_swa, window: int, window_swa: int | None = None,
                  causal: bool = True, scale: float | None = None) -> np.ndarray:
    """Full gated SA+SWA output [B, n, Hq, d] ("Gated SA and SWA" equation)."""
    return _full(lambda: gated_rows(q, k, v, perm, gate_sa, gate_swa, window, window_swa,
                                    causal, scale), q)


def masked_attention(q, k, v, mask: np.ndarray, scale: float | None = None) -> np.ndarray:
    """Textbook softmax attention with a boolean mask[i, j] shared by all
    sequences and heads: Y = softmax(scale * Q K^T masked) V.  Every row of
    ``mask`` must allow at least one key."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    _check(q, k, v)
    bsz, n, hq, d = q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    hm = _head_map(hq, k.shape[2])
    mask = np.asarray(mask, dtype=bool)
    if not mask.any(axis=1).all():
        raise ValueError("every query needs at least one key")
    out = np.empty_like(q)
    for b in range(bsz):
        for h in range(hq):
            s = scale * (q[b, :, h, :] @ k[b, :, hm[h], :].T)
            s = np.where(mask, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            e = np.exp(s)
            out[b, :, h, :] = (e / e.sum(axis=1, keepdims=True)) @ v[b, :, hm[h], :]
    return out


def full_attention(q, k, v, causal: bool, scale: float | None = None) -> np.ndarray:
    """Full softmax attention (all keys, or keys j <= i when causal): what SA
    reduces to once the window spans the whole sequence, the reference the
    wide-window pins compare against."""
    n = np.shape(q)[1]
    mask = np.tril(np.ones((n, n), dtype=bool)) if causal else np.ones((n, n), dtype=bool)
    return masked_attention(q, k, v, mask, scale)
