"""Pins of the oracle's gate projections and rotary embedding
(oracle/prologue.py), CPU only: special cases that reduce to selection or a
library routine, hand-derived values, and the invariants that define a
rotary embedding (identity at position 0, norm-preserving pair rotations,
scores that depend only on the distance between positions)."""

from __future__ import annotations

import inspect
import types

import numpy as np
import pytest
import torch

import oracle
from oracle import prologue as _pro


def test_gate_logits_select_features_with_unit_weights_and_add_bias():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((2, 5, 6))
    e = np.eye(6)
    a_sa, a_swa = oracle.gate_logits(x, e[[1, 4]], e[[0, 5, 2]], np.array([0.5, -1.0]), None)
    np.testing.assert_array_equal(a_sa, x[..., [1, 4]] + np.array([0.5, -1.0]))
    np.testing.assert_array_equal(a_swa, x[..., [0, 5, 2]])


def test_gate_logits_match_torch_linear_and_are_independent():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 7, 16))
    w1, w2 = rng.standard_normal((4, 16)), rng.standard_normal((4, 16))
    b1, b2 = rng.standard_normal(4), rng.standard_normal(4)
    a1, a2 = oracle.gate_logits(x, w1, w2, b1, b2)
    t = torch.nn.functional.linear
    np.testing.assert_allclose(a1, t(torch.tensor(x), torch.tensor(w1), torch.tensor(b1)).numpy(),
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(a2, t(torch.tensor(x), torch.tensor(w2), torch.tensor(b2)).numpy(),
                               rtol=1e-12, atol=1e-12)
    a1b, _ = oracle.gate_logits(x, w1, w2 * 3.0, b1, b2)
    np.testing.assert_array_equal(a1, a1b)


def test_rope_hand_values_d4():
    """d = 4, base 10000: theta_0 = 1, theta_1 = 1/100; pairs (x0, x2) and
    (x1, x3).  Position 1 turns (1, 0) by 1 rad and by 0.01 rad."""
    x = np.zeros((1, 2, 2, 4))
    x[0, :, 0, 0] = 1.0   # head 0: unit along x0
    x[0, :, 1, 1] = 1.0   # head 1: unit along x1
    y = oracle.rope(x)
    np.testing.assert_allclose(y[0, 0], x[0, 0], atol=0)
    np.testing.assert_allclose(y[0, 1, 0], [np.cos(1.0), 0.0, np.sin(1.0), 0.0], atol=1e-15)
    np.testing.assert_allclose(y[0, 1, 1], [0.0, np.cos(0.01), 0.0, np.sin(0.01)], atol=1e-15)


def test_rope_is_the_complex_rotation_of_half_pairs():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 9, 3, 8))
    y = oracle.rope(x, base=500.0)
    z = (x[..., :4] + 1j * x[..., 4:]) * np.exp(1j * np.arange(9)[None, :, None, None]
                                                * 500.0 ** (-np.arange(4) / 4.0))
    np.testing.assert_allclose(y[..., :4], z.real, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y[..., 4:], z.imag, rtol=1e-12, atol=1e-12)


def test_rope_preserves_pair_norms_and_scores_depend_on_distance_only():
    rng = np.random.default_rng(3)
    d, n = 16, 40
    q = np.broadcast_to(rng.standard_normal(d), (1, n, 1, d)).copy()
    k = np.broadcast_to(rng.standard_normal(d), (1, n, 1, d)).copy()
    rq, rk = oracle.rope(q), oracle.rope(k)
    pn = lambda v: v[..., : d // 2] ** 2 + v[..., d // 2:] ** 2
    np.testing.assert_allclose(pn(rq), pn(q), rtol=1e-12)
    s = np.einsum("id,jd->ij", rq[0, :, 0], rk[0, :, 0])
    for off in (-7, 0, 3, 11):
        diag = np.diagonal(s, offset=off)
        np.testing.assert_allclose(diag, diag[0], rtol=1e-9, atol=1e-9)


MUTANTS = [
    ("sin-sign", "return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)",
     "return np.concatenate([lo * c + hi * s, hi * c - lo * s], axis=-1)"),
    ("theta-exponent", "theta = base ** (-2.0 * k / d)", "theta = base ** (-1.0 * k / d)"),
    ("positions-from-one", "return np.arange(n, dtype=np.float64)[:, None] * theta[None, :]",
     "return np.arange(1, n + 1, dtype=np.float64)[:, None] * theta[None, :]"),
    ("interleaved-pairs", "lo, hi = x[..., : d // 2], x[..., d // 2:]",
     "lo, hi = x[..., 0::2], x[..., 1::2]"),
    ("bias-dropped", "            a = a + np.asarray(b, dtype=np.float64)", "            a = a"),
    ("weights-transposed", 'a = np.einsum("bnd,hd->bnh", x, np.asarray(w, dtype=np.float64))',
     'a = np.einsum("bnd,dh->bnh", x, np.asarray(w, dtype=np.float64).reshape(-1, np.shape(w)[0]))'),
]
PINS = [test_gate_logits_select_features_with_unit_weights_and_add_bias,
        test_gate_logits_match_torch_linear_and_are_independent, test_rope_hand_values_d4,
        test_rope_is_the_complex_rotation_of_half_pairs,
        test_rope_preserves_pair_norms_and_scores_depend_on_distance_only]


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("mid,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_prologue_mistake_fails_a_pin(monkeypatch, mid, old, new):
    src = inspect.getsource(_pro)
    assert src.count(old) == 1, old
    mutant = types.ModuleType("oracle.prologue_mutant")
    mutant.__package__ = "oracle"
    exec(compile(src.replace(old, new), _pro.__file__, "exec"), mutant.__dict__)
    for name in ("gate_logits", "rope", "rope_angles"):
        monkeypatch.setattr(oracle, name, mutant.__dict__[name])
    caught = False
    for fn in PINS:
        try:
            fn()
        except (Exception, pytest.fail.Exception):
            caught = True
            break
    assert caught, mid
