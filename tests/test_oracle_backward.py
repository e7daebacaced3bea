"""Pins of the oracle's gradients (oracle/backward.py), CPU only.

Nothing here retypes the oracle's formulas.  The gradients are pinned to
things fixed independently of them:
  * central finite differences of the (separately pinned) forward oracle, in
    fp64, for every input: Q, K, V and both gate logits;
  * PyTorch fp64 autograd through a dense restatement of the attention
    (mask built straight from the definition: |sigma^-1(i) - sigma^-1(j)| <= h
    and, when causal, j <= i);
  * exact invariants of softmax attention: the key gradients of one kv head
    sum to zero (shifting every key by the same vector leaves each softmax
    unchanged) and the value gradients sum to the query heads' upstream
    gradients (each row's weights sum to one);
  * the reductions the forward pins also use: sigma = identity turns causal SA
    into SWA with window h + 1, and saturated gates select one path;
  * the log-sum-exp against scipy's logsumexp on the dense scores.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle


def _case(b=2, n=11, hq=4, hkv=2, d=6, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((b, n, hq, d))
    k = rng.standard_normal((b, n, hkv, d))
    v = rng.standard_normal((b, n, hkv, d))
    dy = rng.standard_normal((b, n, hq, d))
    ga = rng.standard_normal((b, n, hq))
    gw = rng.standard_normal((b, n, hq))
    perm = np.stack([oracle.make_perm(seed, 0, i, n) for i in range(b)])
    return q, k, v, dy, ga, gw, perm


def _fd_check(f, x, grad, dy, eps=1e-6, samples=12, seed=1):
    """Central differences of <f(x), dy> at `samples` random entries of x."""
    rng = np.random.default_rng(seed)
    flat = x.reshape(-1)
    for idx in rng.choice(flat.size, size=min(samples, flat.size), replace=False):
        old = flat[idx]
        flat[idx] = old + eps
        fp = float((f() * dy).sum())
        flat[idx] = old - eps
        fm = float((f() * dy).sum())
        flat[idx] = old
        num = (fp - fm) / (2 * eps)
        assert abs(num - grad.reshape(-1)[idx]) <= 1e-6 * max(1.0, abs(num)), (idx, num,
                                                                              grad.reshape(-1)[idx])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("w", [2, 5, 40])
def test_sa_gradients_match_finite_differences(causal, w):
    q, k, v, dy, _, _, perm = _case(seed=w)
    dq, dk, dv = oracle.sa_backward(q, k, v, perm, dy, w, causal)
    f = lambda: oracle.sa_forward(q, k, v, perm, w, causal)
    _fd_check(f, q, dq, dy)
    _fd_check(f, k, dk, dy)
    _fd_check(f, v, dv, dy)


@pytest.mark.parametrize("w", [1, 4, 30])
def test_swa_gradients_match_finite_differences(w):
    q, k, v, dy, _, _, _ = _case(seed=100 + w)
    dq, dk, dv = oracle.swa_backward(q, k, v, dy, w)
    f = lambda: oracle.swa_forward(q, k, v, w)
    _fd_check(f, q, dq, dy)
    _fd_check(f, k, dk, dy)
    _fd_check(f, v, dv, dy)


@pytest.mark.parametrize("w_swa", [0, 3])
def test_gated_gradients_match_finite_differences(w_swa):
    q, k, v, dy, ga, gw, perm = _case(seed=7)
    dq, dk, dv, dga, dgw = oracle.gated_backward(q, k, v, perm, ga, gw, dy, 6, w_swa, True)
    f = lambda: oracle.gated_forward(q, k, v, perm, ga, gw, 6, w_swa, True)
    for x, g in ((q, dq), (k, dk), (v, dv), (ga, dga), (gw, dgw)):
        _fd_check(f, x, g, dy)


def _dense_mask(perm, n, w, causal):
    """The SA mask written straight from the definition, as a dense matrix."""
    inv = np.empty(n, dtype=np.int64)
    inv[perm] = np.arange(n)
    h = w // 2
    m = np.abs(inv[:, None] - inv[None, :]) <= h
    if causal:
        m &= np.tril(np.ones((n, n), dtype=bool))
    return m


def _torch_grads(q, k, v, dy, masks, scale=None):
    """fp64 autograd through dense masked attention (one mask per batch)."""
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    g = q.shape[2] // k.shape[2]
    kk = tk.repeat_interleave(g, dim=2)
    vv = tv.repeat_interleave(g, dim=2)
    sc = 1.0 / np.sqrt(q.shape[3]) if scale is None else scale
    s = torch.einsum("bihd,bjhd->bhij", tq, kk) * sc
    mask = torch.tensor(np.stack(masks))[:, None]
    s = s.masked_fill(~mask, float("-inf"))
    y = torch.einsum("bhij,bjhd->bihd", torch.softmax(s, dim=-1), vv)
    (y * torch.tensor(dy)).sum().backward()
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("hq,hkv", [(4, 2), (3, 3), (8, 1)])
def test_sa_gradients_match_autograd_of_dense_restatement(causal, hq, hkv):
    q, k, v, dy, _, _, perm = _case(b=2, n=17, hq=hq, hkv=hkv, d=5, seed=hq * 10 + hkv)
    w = 6
    want = _torch_grads(q, k, v, dy, [_dense_mask(perm[b], 17, w, causal) for b in range(2)])
    got = oracle.sa_backward(q, k, v, perm, dy, w, causal)
    for g, t in zip(got, want):
        np.testing.assert_allclose(g, t, rtol=1e-10, atol=1e-12)


def test_swa_gradients_match_autograd_of_dense_restatement():
    q, k, v, dy, _, _, _ = _case(b=1, n=15, hq=4, hkv=2, d=4, seed=3)
    w = 5
    i = np.arange(15)
    mask = (i[None, :] <= i[:, None]) & (i[None, :] > i[:, None] - w)
    want = _torch_grads(q, k, v, dy, [mask])
    got = oracle.swa_backward(q, k, v, dy, w)
    for g, t in zip(got, want):
        np.testing.assert_allclose(g, t, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_key_gradients_sum_to_zero_and_value_gradients_to_dy(causal):
    q, k, v, dy, _, _, perm = _case(b=2, n=20, hq=6, hkv=2, d=4, seed=11)
    dq, dk, dv = oracle.sa_backward(q, k, v, perm, dy, 8, causal)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    g = 3
    want = dy.reshape(2, 20, 2, g, 4).sum(axis=(1, 3))
    np.testing.assert_allclose(dv.sum(axis=1), want, rtol=1e-12, atol=1e-12)


def test_sampled_dq_rows_equal_the_full_gradient():
    q, k, v, dy, _, _, perm = _case(b=2, n=16, seed=13)
    dq, _, _ = oracle.sa_backward(q, k, v, perm, dy, 6, True)
    rows = [(0, 0), (1, 15), (1, 3), (0, 9)]
    got = oracle.sa_dq_rows(q, k, v, perm, dy, 6, True, rows)
    for r, (b, i) in enumerate(rows):
        np.testing.assert_array_equal(got[r], dq[b, i])


def test_identity_sigma_causal_sa_gradients_equal_swa():
    q, k, v, dy, _, _, _ = _case(b=1, n=14, seed=5)
    ident = np.arange(14)[None]
    for w in (2, 6, 9):
        a = oracle.sa_backward(q, k, v, ident, dy, w, True)
        b = oracle.swa_backward(q, k, v, dy, w // 2 + 1)
        for x, y in zip(a, b):
            np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-12)


def test_saturated_gates_select_one_path():
    q, k, v, dy, _, _, perm = _case(seed=9)
    big = np.full(q.shape[:3], 40.0)
    dq, dk, dv, dga, dgw = oracle.gated_backward(q, k, v, perm, big, -big, dy, 6, 0, True)
    a = oracle.sa_backward(q, k, v, perm, dy, 6, True)
    for x, y in zip((dq, dk, dv), a):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-12)
    assert np.abs(dga).max() < 1e-15 and np.abs(dgw).max() < 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_lse_matches_scipy_logsumexp_on_dense_scores(causal):
    q, k, _, _, _, _, perm = _case(b=2, n=13, hq=4, hkv=2, d=5, seed=21)
    w = 6
    got = oracle.sa_lse(q, k, perm, w, causal)
    for b in range(2):
        m = _dense_mask(perm[b], 13, w, causal)
        for h in range(4):
            s = (q[b, :, h, :] @ k[b, :, h // 2, :].T) / np.sqrt(5)
            want = logsumexp(np.where(m, s, -np.inf), axis=1)
            np.testing.assert_allclose(got[b, :, h], want, rtol=1e-12, atol=1e-12)
    got_swa = oracle.swa_lse(q, k, 4)
    i = np.arange(13)
    m = (i[None, :] <= i[:, None]) & (i[None, :] > i[:, None] - 4)
    s = (q[0, :, 1, :] @ k[0, :, 0, :].T) / np.sqrt(5)
    np.testing.assert_allclose(got_swa[0, :, 1], logsumexp(np.where(m, s, -np.inf), axis=1),
                               rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ planted mistakes
# Each one-line mistake in oracle/backward.py must fail at least one pin above.

import inspect  # noqa: E402
import types  # noqa: E402

from oracle import backward as _bw  # noqa: E402

BW_MUTANTS = [
    ("softmax-jacobian-drops-mean", "ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))", "ds = p * dp"),
    ("softmax-jacobian-sign", "ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))",
     "ds = p * ((p * dp).sum(axis=1, keepdims=True) - dp)"),
    ("dq-without-scale", 'dq_out[:] = scale * np.einsum("hm,mhd->hd", ds, kh)',
     'dq_out[:] = np.einsum("hm,mhd->hd", ds, kh)'),
    ("dq-uses-v", 'dq_out[:] = scale * np.einsum("hm,mhd->hd", ds, kh)',
     'dq_out[:] = scale * np.einsum("hm,mhd->hd", ds, vh)'),
    ("dk-uses-dy", "scale * ds[h][:, None] * qrow[h][None, :])",
     "scale * ds[h][:, None] * dyrow[h][None, :])"),
    ("dv-uses-ds", "p[h][:, None] * dyrow[h][None, :])", "ds[h][:, None] * dyrow[h][None, :])"),
    ("dp-uses-k", 'dp = np.einsum("hd,mhd->hm", dyrow, vh)', 'dp = np.einsum("hd,mhd->hm", dyrow, kh)'),
    ("kv-head-is-query-head", "        kvh = head_map[h]\n", "        kvh = h % kb.shape[1]\n"),
    ("gate-derivative-missing-factor", 'da_sa = g_sa * (1.0 - g_sa) * np.einsum("bnhd,bnhd->bnh", dy, y_sa)',
     'da_sa = g_sa * np.einsum("bnhd,bnhd->bnh", dy, y_sa)'),
    ("swa-upstream-ungated", "d2 = swa_backward(q, k, v, g_swa[..., None] * dy, w_swa, scale)",
     "d2 = swa_backward(q, k, v, dy, w_swa, scale)"),
    ("lse-drops-max", "out[b, i] = m + np.log(np.exp(s - m[:, None]).sum(axis=1))",
     "out[b, i] = np.log(np.exp(s - m[:, None]).sum(axis=1))"),
]

BW_PINS = [
    (test_sa_gradients_match_finite_differences, (True, 5)),
    (test_swa_gradients_match_finite_differences, (4,)),
    (test_gated_gradients_match_finite_differences, (3,)),
    (test_sa_gradients_match_autograd_of_dense_restatement, (True, 4, 2)),
    (test_lse_matches_scipy_logsumexp_on_dense_scores, (True,)),
]


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("mid,old,new", BW_MUTANTS, ids=[m[0] for m in BW_MUTANTS])
def test_planted_backward_mistake_fails_a_pin(monkeypatch, mid, old, new):
    src = inspect.getsource(_bw)
    assert src.count(old) == 1, old
    mutant = types.ModuleType("oracle.backward_mutant")
    mutant.__package__ = "oracle"
    mutant.__file__ = _bw.__file__
    exec(compile(src.replace(old, new), _bw.__file__, "exec"), mutant.__dict__)
    for name, fn in list(vars(_bw).items()):
        if inspect.isfunction(fn) and fn.__module__ == _bw.__name__:
            for holder in (oracle, _bw):
                if getattr(holder, name, None) is fn:
                    monkeypatch.setattr(holder, name, mutant.__dict__[name])
    caught = False
    for fn, args in BW_PINS:
        try:
            fn(*args)
        except (Exception, pytest.fail.Exception):
            caught = True
            break
    assert caught, f"no pin detects the planted backward mistake {mid!r}"
