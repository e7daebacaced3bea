"""Gradients of SA, SWA and the gated SA+SWA merge in fp64 (oracle side).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

The pages use SA (gated with SWA) to pretrain a model from scratch ("Stochastic
Attention" summary, "Main contributions" item 3 and the first bullet of
"Results"), which needs the gradient of each path's output with respect to Q,
K, V and the gate logits.  The pages print no gradient; it follows from the
forward definition by the chain rule.  As in ``attention``, the work goes one
ORIGINAL token i at a time over its neighbour set N(i):

    s_j = scale <q_i, k_j>,  p_j = softmax over j in N(i),  y_i = sum_j p_j v_j

and, given the upstream gradient dy_i,

    dv_j  += p_j dy_i
    dp_j   = <dy_i, v_j>
    ds_j   = p_j (dp_j - sum_m p_m dp_m)          (softmax Jacobian)
    dq_i   = scale sum_j ds_j k_j
    dk_j  += scale ds_j q_i

Grouped-query attention: a kv head's gradient sums the contributions of every
query head that reads it.  The gated merge y = g_sa y_sa + g_swa y_swa with
g = sigmoid(a) gives dy_sa = g_sa dy, dy_swa = g_swa dy and
da = g (1 - g) <dy, y_path> per token and query head.  All arithmetic is
float64.
"""

from __future__ import annotations

import numpy as np

from .attention import _as_f64, _check, _head_map, sa_rows, sigmoid, swa_rows
from .graph import neighbours_sa, neighbours_swa
from .prng import inverse_perm


def _row_backward(qrow, kb, vb, keys, head_map, scale, dyrow, dq_out, dk_acc, dv_acc):
    """Chain rule through one token's softmax attention over ``keys``.

    qrow, dyrow [Hq, d]; kb, vb [n, Hkv, d]; writes dq_out [Hq, d] and adds
    into dk_acc, dv_acc [n, Hkv, d]."""
    kh = kb[keys][:, head_map, :]                       # [m, Hq, d]
    vh = vb[keys][:, head_map, :]
    s = scale * np.einsum("hd,mhd->hm", qrow, kh)        # [Hq, m]
    s = s - s.max(axis=1, keepdims=True)
    e = np.exp(s)
    p = e / e.sum(axis=1, keepdims=True)
    dp = np.einsum("hd,mhd->hm", dyrow, vh)              # <dy_i, v_j>
    ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    dq_out[:] = scale * np.einsum("hm,mhd->hd", ds, kh)
    for h in range(qrow.shape[0]):
        kvh = head_map[h]
        np.add.at(dk_acc[:, kvh, :], keys, scale * ds[h][:, None] * qrow[h][None, :])
        np.add.at(dv_acc[:, kvh, :], keys, p[h][:, None] * dyrow[h][None, :])


def _backward(q, k, v, dy, neighbours, scale):
    q, k, v, dy = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dy)
    _check(q, k, v)
    if dy.shape != q.shape:
        raise ValueError("dy must have Q's shape")
    bsz, n, hq, d = q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    hm = _head_map(hq, k.shape[2])
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(bsz):
        for i in range(n):
            _row_backward(q[b, i], k[b], v[b], neighbours(b, i), hm, scale, dy[b, i], dq[b, i],
                          dk[b], dv[b])
    return dq, dk, dv


def sa_backward(q, k, v, perm, dy, window: int, causal: bool, scale: float | None = None):
    """(dQ, dK, dV) of SA ("Core mechanism" steps 1-3; causal rule from
    "Theoretical properties") for the upstream gradient dy [B, n, Hq, d]."""
    perm = np.asarray(perm, dtype=np.int64).reshape(np.shape(q)[0], np.shape(q)[1])
    invs = [inverse_perm(perm[b]) for b in range(perm.shape[0])]
    return _backward(q, k, v, dy,
                     lambda b, i: neighbours_sa(perm[b], window, causal, i, invs[b]), scale)


def sa_dq_rows(q, k, v, perm, dy, window: int, causal: bool, rows, scale: float | None = None):
    """dQ rows [R, Hq, d] of SA for the (b, i) pairs in ``rows`` only: a
    query row's gradient depends on its own window alone, so large cases can
    be checked on a sample (same per-token chain rule as ``sa_backward``)."""
    q, k, v, dy = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dy)
    _check(q, k, v)
    bsz, n, hq, d = q.shape
    perm = np.asarray(perm, dtype=np.int64).reshape(bsz, n)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    hm = _head_map(hq, k.shape[2])
    invs, out = {}, []
    for b, i in rows:
        b, i = int(b), int(i)
        if b not in invs:
            invs[b] = inverse_perm(perm[b])
        keys = neighbours_sa(perm[b], window, causal, i, invs[b])
        dq = np.empty((hq, d))
        dk_sink = np.zeros_like(k[b])
        dv_sink = np.zeros_like(v[b])
        _row_backward(q[b, i], k[b], v[b], keys, hm, scale, dy[b, i], dq, dk_sink, dv_sink)
        out.append(dq)
    return np.asarray(out).reshape(-1, hq, d)


def swa_backward(q, k, v, dy, window: int, scale: float | None = None):
    """(dQ, dK, dV) of SWA over keys [max(0, i-w+1), i] ("Problem statement")."""
    n = np.shape(q)[1]
    return _backward(q, k, v, dy, lambda b, i: neighbours_swa(n, window, i), scale)


def gated_backward(q, k, v, perm, gate_sa, gate_swa, dy, window: int,
                   window_swa: int | None = None, causal: bool = True,
                   scale: float | None = None):
    """(dQ, dK, dV, dA_sa, dA_swa) of the gated dual path ("Gated SA and SWA"
    equation): each path's gradient at its gated upstream gradient, summed,
    and the logit gradients g (1 - g) <dy, y_path> [B, n, Hq]."""
    q, dy = _as_f64(q), _as_f64(dy)
    bsz, n, hq, d = q.shape
    w_swa = window if (window_swa is None or window_swa <= 0) else window_swa
    g_sa = sigmoid(np.reshape(gate_sa, (bsz, n, hq)))
    g_swa = sigmoid(np.reshape(gate_swa, (bsz, n, hq)))
    y_sa = sa_rows(q, k, v, perm, window, causal, scale).reshape(bsz, n, hq, d)
    y_swa = swa_rows(q, k, v, w_swa, scale).reshape(bsz, n, hq, d)
    d1 = sa_backward(q, k, v, perm, g_sa[..., None] * dy, window, causal, scale)
    d2 = swa_backward(q, k, v, g_swa[..., None] * dy, w_swa, scale)
    da_sa = g_sa * (1.0 - g_sa) * np.einsum("bnhd,bnhd->bnh", dy, y_sa)
    da_swa = g_swa * (1.0 - g_swa) * np.einsum("bnhd,bnhd->bnh", dy, y_swa)
    return d1[0] + d2[0], d1[1] + d2[1], d1[2] + d2[2], da_sa, da_swa


def _lse(q, k, neighbours, scale):
    q, k = _as_f64(q), _as_f64(k)
    bsz, n, hq, d = q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    hm = _head_map(hq, k.shape[2])
    out = np.empty((bsz, n, hq))
    for b in range(bsz):
        for i in range(n):
            keys = neighbours(b, i)
            s = scale * np.einsum("hd,mhd->hm", q[b, i], k[b][keys][:, hm, :])
            m = s.max(axis=1)
            out[b, i] = m + np.log(np.exp(s - m[:, None]).sum(axis=1))
    return out


def sa_lse(q, k, perm, window: int, causal: bool, scale: float | None = None):
    """Per-row log-sum-exp log sum_{j in N(i)} exp(scale <q_i, k_j>) of SA,
    [B, n, Hq] by original token: the softmax normaliser a backward pass
    reuses."""
    perm = np.asarray(perm, dtype=np.int64).reshape(np.shape(q)[0], np.shape(q)[1])
    invs = [inverse_perm(perm[b]) for b in range(perm.shape[0])]
    return _lse(q, k, lambda b, i: neighbours_sa(perm[b], window, causal, i, invs[b]), scale)


def swa_lse(q, k, window: int, scale: float | None = None):
    """Per-row log-sum-exp of SWA, [B, n, Hq]."""
    n = np.shape(q)[1]
    return _lse(q, k, lambda b, i: neighbours_swa(n, window, i), scale)
