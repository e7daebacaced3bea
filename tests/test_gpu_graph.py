"""GPU receptive fields of stacked SA layers (sa_receptive_field through the
C ABI) against the oracle.

Small n: every token's |R_l| for every layer, bit-exact against the oracle's
dense boolean products (oracle.receptive_field_sizes).  Long sequences (the
length-sweep size n = 262144, w = 128): layer 1 and 2 fields of sampled
targets exactly against explicit set unions over the oracle's neighbour sets,
and the properties that hold at any size (fields only grow, never exceed n,
and outgrow sliding-window attention's linear l (w - 1) + 1 from layer 2 on).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import stochastic_sliding_window_gb300 as sa

pytestmark = pytest.mark.gpu


def _perms(seed, layers, n):
    ps = np.stack([oracle.make_perm(seed, l, 0, n) for l in range(layers)])
    lib = np.stack([sa.make_perm(seed, l, 0, n) for l in range(layers)])
    assert np.array_equal(ps, lib.astype(np.int64))
    return ps, torch.from_numpy(lib).cuda()


@pytest.mark.parametrize("n,w,layers", [(64, 2, 6), (64, 9, 4), (257, 16, 5), (512, 32, 4),
                                        (300, 600, 2)])
@pytest.mark.parametrize("causal", [False, True])
def test_all_tokens_bit_exact_against_oracle(n, w, layers, causal):
    ps, pd = _perms(n + w, layers, n)
    targets = torch.arange(n, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = sa.receptive_field(pd, w, targets, causal=causal, err=err).cpu().numpy()
    assert sa.check_error(err) == sa.SA_OK
    want = oracle.receptive_field_sizes([oracle.adjacency_sa(ps[l], w, causal)
                                         for l in range(layers)])
    assert np.array_equal(got, want)


def test_targets_in_any_order_and_repeated():
    n, w, layers = 200, 12, 3
    ps, pd = _perms(9, layers, n)
    want = oracle.receptive_field_sizes([oracle.adjacency_sa(ps[l], w, True) for l in range(layers)])
    t = np.array([199, 0, 5, 5, 77, 199, 123] * 11, dtype=np.int32)  # 77 targets: two groups
    got = sa.receptive_field(pd, w, torch.from_numpy(t).cuda(), causal=True).cpu().numpy()
    assert np.array_equal(got, want[:, t])


def _field(ps, w, causal, i, layers):
    """R_layers(i) by explicit set unions: layer `layers` acts on {i} first."""
    invs = [oracle.inverse_perm(p) for p in ps]
    cur = {int(i)}
    for l in range(layers - 1, -1, -1):
        nxt = set()
        for j in cur:
            nxt.update(oracle.neighbours_sa(ps[l], w, causal, j, invs[l]).tolist())
        cur = nxt
    return len(cur)


@pytest.mark.parametrize("causal", [False, True])
def test_length_sweep_size_fields(causal):
    n, w, layers = 262144, 128, 8
    ps, pd = _perms(41, layers, n)
    rng = np.random.default_rng(5)
    t = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 254)])).astype(np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = sa.receptive_field(pd, w, torch.from_numpy(t).cuda(), causal=causal, err=err).cpu().numpy()
    assert sa.check_error(err) == sa.SA_OK
    for idx in range(0, len(t), 40):  # exact at layers 1 and 2 on sampled targets
        for L in (1, 2):
            assert got[L - 1, idx] == _field(ps, w, causal, t[idx], L), (t[idx], L)
    assert (np.diff(got, axis=0) >= 0).all() and (got <= n).all() and (got >= 1).all()
    swa = np.minimum(t[None, :] + 1, np.arange(1, layers + 1)[:, None] * (w - 1) + 1)
    if not causal:
        assert (got[1:] > swa[1:]).all()
        assert (got[3] == n).mean() > 0.99  # full coverage by ceil(log_w n) + 1 = 4 layers
    else:  # causal fields of later tokens outgrow SWA's from layer 2 on
        late = t > n // 2
        assert got[1, late].mean() > swa[1, late].mean()
        assert (got[2:, late] > swa[2:, late]).all()
