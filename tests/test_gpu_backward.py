"""GPU parity of the backward pass (sa_backward, swa_backward,
sa_swa_gated_backward through the C ABI) against the fp64 oracle gradients
on the same bf16 inputs and upstream gradient.

Tolerance.  The pages state none for gradients.  Each gradient element is a
window sum in which one factor (g p or dS) is rounded once to bf16 (unit
roundoff u = 2^-8) before the tensor-core product, and the result is
rounded to bf16 once more; inputs are identical on both sides.  That gives a
relative-L2 error of a few u / sqrt(3) ~ 0.3%: the forward bar (relative-L2
5e-3) applies unchanged.  Elementwise, a gradient is a signed sum whose
terms can cancel, so the absolute bar scales with the tensor's magnitude:
max-abs <= 2e-2 * max(1, max |reference|).
"""

from __future__ import annotations

import multiprocessing as mp

import numpy as np
import pytest
import torch

import oracle
import stochastic_sliding_window_gb300 as sa
from gpu_helpers import dev_bf16, dev_f32, perms
from sa_synth import make_case, round_bf16

pytestmark = pytest.mark.gpu

REL_L2 = 5e-3
ABS = 2e-2


def compare_grad(got, want, what):
    g = got.float().cpu().numpy().astype(np.float64)
    assert g.shape == want.shape, (what, g.shape, want.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite"
    err = np.abs(g - want)
    scale = max(1.0, float(np.abs(want).max()))
    rel = float(np.linalg.norm(g - want) / max(np.linalg.norm(want), 1e-30))
    assert err.max() <= ABS * scale and rel <= REL_L2, \
        f"{what}: max_abs={err.max():.3e} (bar {ABS * scale:.3e}) rel_l2={rel:.3e}"
    return float(err.max()), rel


class Case:
    def __init__(self, b, n, hq, hkv, d, seed, std=None):
        self.c = make_case(b, n, hq, hkv, d, seed, std=std, gates=True)
        rng = np.random.default_rng(seed + 1000)
        self.dy = round_bf16(rng.standard_normal((b, n, hq, d)).astype(np.float32))
        c = self.c
        self.q, self.k, self.v = dev_bf16(c.q), dev_bf16(c.k), dev_bf16(c.v)
        self.dyd = dev_bf16(self.dy)
        self.ga, self.gw = dev_f32(c.gate_sa), dev_f32(c.gate_swa)


def _err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _check(path, case, perm, perm_d, w, causal, w_swa=0):
    c = case.c
    err = _err()
    if path == "sa":
        got = sa.sa_backward(case.q, case.k, case.v, perm_d, case.dyd, w, causal=causal, err=err)
        want = oracle.sa_backward(c.q, c.k, c.v, perm, case.dy, w, causal)
        names = ("dq", "dk", "dv")
    elif path == "swa":
        got = sa.swa_backward(case.q, case.k, case.v, case.dyd, w, err=err)
        want = oracle.swa_backward(c.q, c.k, c.v, case.dy, w)
        names = ("dq", "dk", "dv")
    else:
        got = sa.sa_swa_gated_backward(case.q, case.k, case.v, perm_d, case.ga, case.gw, case.dyd,
                                       w, window_swa=w_swa, causal=causal, err=err)
        want = oracle.gated_backward(c.q, c.k, c.v, perm, c.gate_sa, c.gate_swa, case.dy, w,
                                     w_swa or None, causal)
        names = ("dq", "dk", "dv", "dgate_sa", "dgate_swa")
    assert sa.check_error(err) == sa.SA_OK
    return {nm: compare_grad(gg, ww, f"{path} w={w} causal={causal} {nm}")
            for nm, gg, ww in zip(names, got, want)}


@pytest.mark.parametrize("path,causal", [("sa", True), ("sa", False), ("swa", True),
                                         ("gated", True), ("gated", False)])
def test_tiny_case_backward(path, causal):
    """B1 n256 H2 d64 w32: every gradient element against the oracle."""
    case = Case(1, 256, 2, 2, 64, seed=0, std=1.0 / 8.0)
    perm, perm_d = perms(0, 0, 1, 256)
    _check(path, case, perm, perm_d, 32, causal)


EDGE = [
    # b, n, hq, hkv, d, w
    (1, 1, 8, 2, 128, 4),
    (2, 7, 8, 2, 128, 1),
    (2, 100, 4, 4, 64, 7),
    (1, 333, 8, 2, 128, 64),
    (1, 300, 32, 8, 128, 128),
    (2, 200, 8, 1, 128, 16),
    (1, 129, 2, 2, 64, 96),
]


@pytest.mark.parametrize("b,n,hq,hkv,d,w", EDGE)
@pytest.mark.parametrize("path,causal", [("sa", True), ("sa", False), ("swa", True),
                                         ("gated", True)])
def test_ragged_and_edge_shapes_backward(b, n, hq, hkv, d, w, path, causal):
    case = Case(b, n, hq, hkv, d, seed=n + w)
    perm, perm_d = perms(7, 2, b, n)
    _check(path, case, perm, perm_d, w, causal)


def test_gated_backward_separate_swa_window():
    case = Case(1, 300, 8, 2, 128, seed=5)
    perm, perm_d = perms(5, 0, 1, 300)
    _check("gated", case, perm, perm_d, 64, True, w_swa=24)


def _oracle_gated_one(args):
    q, k, v, perm, ga, gw, dy, w = args
    return oracle.gated_backward(q, k, v, perm, ga, gw, dy, w, None, True)


def test_pretraining_layer_gated_backward():
    """B4 n2048 16 MHA heads d64 w128 causal gated (the pretraining layer):
    every gradient element; the oracle runs one sequence per process."""
    b, n = 4, 2048
    case = Case(b, n, 16, 16, 64, seed=11, std=1.0 / 8.0)
    perm, perm_d = perms(11, 0, b, n)
    err = _err()
    got = sa.sa_swa_gated_backward(case.q, case.k, case.v, perm_d, case.ga, case.gw, case.dyd, 128,
                                   causal=True, err=err)
    assert sa.check_error(err) == sa.SA_OK
    c = case.c
    jobs = [(c.q[i:i + 1], c.k[i:i + 1], c.v[i:i + 1], perm[i:i + 1], c.gate_sa[i:i + 1],
             c.gate_swa[i:i + 1], case.dy[i:i + 1], 128) for i in range(b)]
    with mp.get_context("spawn").Pool(b) as pool:
        parts = pool.map(_oracle_gated_one, jobs)
    want = [np.concatenate([p[t] for p in parts]) for t in range(5)]
    for nm, gg, ww in zip(("dq", "dk", "dv", "dgate_sa", "dgate_swa"), got, want):
        compare_grad(gg, ww, f"pretraining layer {nm}")


def test_long_prefill_backward_sampled_query_rows():
    """The long-prefill GQA shape (n=32768, 32q/8kv, d128, w=128, causal SA):
    dq rows depend only on their own window, so a seeded sample of them is
    checked against the oracle's per-row gradient; dk and dv are checked
    through their exact sums (each kv head's dk sums to zero, its dv to the
    sum of its query heads' dout)."""
    n, hq, hkv, d, w = 32768, 32, 8, 128, 128
    case = Case(1, n, hq, hkv, d, seed=21)
    perm, perm_d = perms(21, 0, 1, n)
    err = _err()
    dq, dk, dv = sa.sa_backward(case.q, case.k, case.v, perm_d, case.dyd, w, causal=True, err=err)
    assert sa.check_error(err) == sa.SA_OK
    c = case.c
    rng = np.random.default_rng(3)
    rows = sorted({0, n - 1, *rng.integers(0, n, 40).tolist()})
    want = oracle.sa_dq_rows(c.q, c.k, c.v, perm, case.dy, w, True, [(0, i) for i in rows])
    for r, i in enumerate(rows):
        compare_grad(dq[0, i], want[r], f"c3 dq row {i}")
    dks = dk.float().sum(dim=1).cpu().numpy()
    assert np.abs(dks).max() <= 2e-2 * max(1.0, float(dk.float().abs().max()))
    want_v = case.dy.astype(np.float64).reshape(1, n, hkv, hq // hkv, d).sum(axis=(1, 3))
    got_v = dv.double().sum(dim=1).cpu().numpy()
    assert np.linalg.norm(got_v - want_v) <= 5e-3 * np.linalg.norm(want_v)


def test_backward_rejects_too_wide_windows_and_bad_workspace():
    case = Case(1, 64, 4, 4, 64, seed=1)
    _, perm_d = perms(1, 0, 1, 64)
    with pytest.raises(sa.SaError) as ei:
        sa.sa_backward(case.q, case.k, case.v, perm_d, case.dyd, 512)
    assert ei.value.status == sa.SA_ERR_UNSUPPORTED
