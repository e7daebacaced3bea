"""Pins of the fp64 oracle against things other than itself.

Each test ties one part of the oracle to a published value, a hand
derivation, a closed form, an invariant the pages state, or an independent
library routine (torch's scaled_dot_product_attention in fp64 on the CPU),
chosen so that a plausible mistake (a dropped scale, sigma used where
sigma^-1 belongs, a wrong GQA head map, an off-by-one window) fails one.
"""

from __future__ import annotations

import itertools
import math
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
from oracle import attention, graph, prng
from sa_synth import bf16_bits, make_case, round_bf16

GOLDEN = Path(__file__).parent / "golden"


def _golden_lines(name):
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if line and not line.startswith("#"):
            yield line


def _sets(field: str):
    out = {}
    for item in field.split():
        i, js = item.split(":")
        out[int(i)] = sorted(int(j) for j in js.split(","))
    return out


# ---------------------------------------------------------------- sigma draw

def test_splitmix64_published_vectors():
    for line in _golden_lines("splitmix64.txt"):
        vals = [int(x) for x in line.split()]
        state = vals[0]
        for want in vals[1:]:
            state, got = prng.splitmix64_step(state)
            assert got == want


def test_stream_state_is_one_published_step_from_the_start():
    """The stream of (seed, layer, b) starts from the splitmix64 output for the
    initial state seed + (layer << 32) + b; seeds are chosen so that this
    initial state is one whose first output is published."""
    first = {}
    for line in _golden_lines("splitmix64.txt"):
        vals = [int(x) for x in line.split()]
        first[vals[0]] = vals[1]
    mask = (1 << 64) - 1
    assert prng.stream_state(0, 0, 0) == first[0]
    assert prng.stream_state(1234567, 0, 0) == first[1234567]
    assert prng.stream_state(1234567 - 5, 0, 5) == first[1234567]
    assert prng.stream_state((1234567 - (1 << 32)) & mask, 1, 0) == first[1234567]
    assert prng.stream_state((1234567 - (3 << 32) - 9) & mask, 3, 9) == first[1234567]


def test_make_perm_consumes_successive_stream_outputs():
    """make_perm wires the pinned pieces together: Fisher-Yates (pinned by stub
    draws) fed with successive splitmix64 outputs (pinned by the published
    vectors) from the stream state (pinned above)."""
    for seed, layer, b, n in ((0, 0, 0, 8), (7, 2, 1, 33), (2**63 + 5, 1, 3, 100)):
        state = prng.stream_state(seed, layer, b)
        draws = []
        for _ in range(max(n - 1, 0)):
            state, out = prng.splitmix64_step(state)
            draws.append(out)
        it = iter(draws)
        assert prng.make_perm(seed, layer, b, n).tolist() == \
            prng.fisher_yates(n, lambda: next(it)).tolist()


def test_fisher_yates_index_mapping_with_stub_draws():
    # x = 0 maps every draw to j = 0; Durstenfeld's loop then rotates the
    # identity left by one: sigma[p] = (p + 1) mod n.
    for n in (1, 2, 3, 7, 16):
        got = prng.fisher_yates(n, lambda: 0)
        assert got.tolist() == [(p + 1) % n for p in range(n)]
    # x = 2^64 - 1 maps to j = i (the largest index allowed): no swap at all.
    top = (1 << 64) - 1
    assert prng.fisher_yates(9, lambda: top).tolist() == list(range(9))
    # x = 2^63 maps to j = floor((i + 1) / 2); check against a by-hand list
    # swap for n = 4: i=3 -> j=2, i=2 -> j=1, i=1 -> j=1.
    s = [0, 1, 2, 3]
    for i, j in ((3, 2), (2, 1), (1, 1)):
        s[i], s[j] = s[j], s[i]
    assert prng.fisher_yates(4, lambda: 1 << 63).tolist() == s


def test_perm_draw_is_uniform_over_s4():
    counts = {}
    seeds = 4800
    for seed in range(seeds):
        key = tuple(prng.make_perm(seed, 0, 0, 4).tolist())
        counts[key] = counts.get(key, 0) + 1
    assert len(counts) == 24
    exp = seeds / 24
    chi2 = sum((c - exp) ** 2 / exp for c in counts.values())
    from scipy.stats import chi2 as chi2_dist
    assert chi2_dist.sf(chi2, 23) > 1e-4


def test_streams_differ_by_layer_and_batch():
    n = 64
    base = prng.make_perm(7, 0, 0, n)
    assert not np.array_equal(base, prng.make_perm(7, 1, 0, n))
    assert not np.array_equal(base, prng.make_perm(7, 0, 1, n))
    assert not np.array_equal(base, prng.make_perm(8, 0, 0, n))
    assert np.array_equal(base, prng.make_perm(7, 0, 0, n))
    assert sorted(base.tolist()) == list(range(n))


def test_inverse_perm():
    for seed in range(5):
        p = prng.make_perm(seed, 2, 1, 100)
        inv = prng.inverse_perm(p)
        assert np.array_equal(inv[p], np.arange(100))
        assert np.array_equal(p[inv], np.arange(100))
    with pytest.raises(ValueError):
        prng.inverse_perm(np.array([0, 0, 1]))
    with pytest.raises(ValueError):
        prng.inverse_perm(np.array([0, 3, 1]))


# ---------------------------------------------------------------- neighbour sets

@pytest.mark.parametrize("golden", ["sa_hand_n6.txt", "sa_hand_n6_w5.txt"])
def test_hand_worked_neighbour_sets(golden):
    rec = {}
    for line in _golden_lines(golden):
        key, rest = line.split(None, 1)
        rec[key] = rest
    sigma = np.array([int(x) for x in rec["sigma"].split()])
    w = int(rec["window"])
    assert prng.inverse_perm(sigma).tolist() == [int(x) for x in rec["inverse"].split()]
    for field, causal in (("noncausal", False), ("causal", True)):
        want = _sets(rec[field])
        for i in range(6):
            assert graph.neighbours_sa(sigma, w, causal, i).tolist() == want[i]
    want = _sets(rec["swa"])
    for i in range(6):
        assert graph.neighbours_swa(6, w, i).tolist() == want[i]
    # The attention itself: Q = K = 0 makes the softmax uniform, and V = I
    # exposes the support, so row i must be 1/|N(i)| on N(i).
    q = np.zeros((1, 6, 1, 6))
    v = np.eye(6).reshape(1, 6, 1, 6)
    for field, causal in (("noncausal", False), ("causal", True)):
        y = attention.sa_forward(q, q, v, sigma[None], w, causal)[0, :, 0, :]
        for i, js in _sets(rec[field]).items():
            expect = np.zeros(6)
            expect[js] = 1.0 / len(js)
            np.testing.assert_allclose(y[i], expect, atol=1e-15)


@pytest.mark.parametrize("n,w", [(6, 2), (17, 4), (64, 9), (64, 200), (33, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_attended_pair_count_closed_form(n, w, causal):
    for seed in range(4):
        a = graph.adjacency_sa(prng.make_perm(seed, 0, 0, n), w, causal)
        assert a.sum() == graph.attended_pairs_closed_form(n, w, "sa", causal)
        assert a.diagonal().all()
        if causal:
            assert not np.triu(a, 1).any()
    a = graph.adjacency_swa(n, w)
    assert a.sum() == graph.attended_pairs_closed_form(n, w, "swa")


def test_expected_degree_closed_form():
    n, w = 256, 32
    want = graph.expected_degree_closed_form(n, w)
    assert abs(want - 31.9375) < 1e-12  # 1 + (2*16*256 - 16*17)/256 = 1 + 7920/256
    for seed in range(3):
        a = graph.adjacency_sa(prng.make_perm(seed, 0, 0, n), w, False)
        assert abs(a.sum(axis=1).mean() - want) < 1e-12


def test_closed_forms_at_full_windows():
    """With w >= 2n - 2 every token reaches every other: pair probability 1,
    expected degree n, n^2 non-causal and n(n+1)/2 causal pairs; the brute
    force agrees."""
    for n in (2, 5, 16, 40):
        for w in (2 * n - 2, 2 * n, 5 * n + 1):
            if w < 1:
                continue
            assert graph.pair_probability_closed_form(n, w) == 1.0
            assert graph.expected_degree_closed_form(n, w) == n
            assert graph.attended_pairs_closed_form(n, w, "sa", False) == n * n
            assert graph.attended_pairs_closed_form(n, w, "sa", True) == n * (n + 1) // 2
            perm = prng.make_perm(n, w, 0, n)
            assert graph.adjacency_sa(perm, w, False).all()
            assert np.array_equal(graph.adjacency_sa(perm, w, True),
                                  np.tril(np.ones((n, n), dtype=bool)))


def test_pair_probability_matches_closed_form_and_w_over_n():
    n, w, seeds = 16, 4, 1500
    p_exact = graph.pair_probability_closed_form(n, w)
    # the pages: "about w/n"
    assert abs(p_exact - w / n) < (w / n) * (w / n) + 1.0 / n
    assert abs(graph.pair_probability_closed_form(256, 32) - 0.12132352941176471) < 1e-15
    freq = np.zeros((n, n))
    for seed in range(seeds):
        freq += graph.adjacency_sa(prng.make_perm(seed, 3, 0, n), w, False)
    freq /= seeds
    off = ~np.eye(n, dtype=bool)
    sd = math.sqrt(p_exact * (1 - p_exact) / seeds)
    assert np.all(np.abs(freq[off] - p_exact) < 5 * sd)
    # causal: the same probability below the diagonal, zero above it
    freq_c = np.zeros((n, n))
    for seed in range(seeds):
        freq_c += graph.adjacency_sa(prng.make_perm(seed, 4, 0, n), w, True)
    freq_c /= seeds
    low = np.tril(np.ones((n, n), dtype=bool), -1)
    assert np.all(np.abs(freq_c[low] - p_exact) < 5 * sd)
    assert freq_c[np.triu(np.ones((n, n), dtype=bool), 1)].max() == 0.0


def test_receptive_field_swa_is_linear():
    n, w, layers = 64, 8, 6
    sizes = graph.receptive_field_sizes([graph.adjacency_swa(n, w)] * layers)
    for l in range(1, layers + 1):
        assert sizes[l - 1].tolist() == [min(i + 1, l * (w - 1) + 1) for i in range(n)]


def test_receptive_field_matches_set_unions_over_layers():
    """R_l(i) by explicit set unions over each layer's neighbour sets, layer 1
    first ("Theoretical properties", receptive-field bullet), on tiny inputs
    with a different sigma per layer so that the layer order matters."""
    n, w = 9, 2
    sigmas = [prng.make_perm(11, l, 0, n) for l in range(3)]
    for causal in (False, True):
        reach = [{i} for i in range(n)]
        want = []
        for sigma in sigmas:
            nb = [set(graph.neighbours_sa(sigma, w, causal, i).tolist()) for i in range(n)]
            reach = [set().union(*(reach[j] for j in nb[i])) for i in range(n)]
            want.append([len(r) for r in reach])
        adj = [graph.adjacency_sa(s, w, causal) for s in sigmas]
        assert graph.receptive_field_sizes(adj).tolist() == want


def test_receptive_field_sa_grows_far_faster_than_swa():
    n, w, seeds = 256, 32, 12
    sa_cov = np.zeros(4)
    for seed in range(seeds):
        adj = [graph.adjacency_sa(prng.make_perm(seed, l, 0, n), w, False) for l in range(4)]
        sa_cov += graph.receptive_field_sizes(adj).mean(axis=1) / n
    sa_cov /= seeds
    swa = graph.receptive_field_sizes([graph.adjacency_swa(n, w)] * 4)
    swa_cov = (swa / np.arange(1, n + 1)).mean(axis=1)
    # full coverage by ceil(log_w n) + 1 = 3 layers, ahead of SWA from layer 2
    assert sa_cov[2] > 0.999 and sa_cov[3] == 1.0
    assert sa_cov[1] > swa_cov[1] + 0.2
    # causal SA with n >> w: depth-3 reach far beyond SWA's l*w
    n, w = 1024, 16
    adj = [graph.adjacency_sa(prng.make_perm(5, l, 0, n), w, True) for l in range(3)]
    sizes = graph.receptive_field_sizes(adj)
    late = sizes[2, n // 2:].mean()
    assert late > 4 * (3 * (w - 1) + 1)


# ---------------------------------------------------------------- attention values

def _sdpa(q, k, v, mask=None, causal=False, scale=None):
    """torch SDPA in fp64, BSHD in and out, GQA through enable_gqa."""
    tq = torch.from_numpy(np.asarray(q, np.float64)).permute(0, 2, 1, 3)
    tk = torch.from_numpy(np.asarray(k, np.float64)).permute(0, 2, 1, 3)
    tv = torch.from_numpy(np.asarray(v, np.float64)).permute(0, 2, 1, 3)
    am = None if mask is None else torch.from_numpy(np.asarray(mask, bool))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=am, is_causal=causal, scale=scale,
        enable_gqa=tq.shape[1] != tk.shape[1])
    return out.permute(0, 2, 1, 3).numpy()


def _case(b=2, n=40, hq=4, hkv=2, d=16, seed=0):
    c = make_case(b, n, hq, hkv, d, seed, std=0.7, gates=True, bf16=False)
    return c


@pytest.mark.parametrize("causal", [False, True])
def test_full_attention_matches_sdpa(causal):
    c = _case()
    got = attention.full_attention(c.q, c.k, c.v, causal)
    np.testing.assert_allclose(got, _sdpa(c.q, c.k, c.v, causal=causal), atol=1e-12)


def test_softmax_is_stable_at_large_scores():
    """Scores of several hundred (exp overflows fp64 past ~709) must still give
    the softmax: SA with a full window against torch SDPA in fp64."""
    c = _case(b=1, n=24, hq=2, hkv=2, d=16)
    q = np.asarray(c.q) * 40.0
    k = np.asarray(c.k) * 40.0
    s_max = np.abs(np.einsum("bihd,bjhd->bhij", q, k)).max() / 4.0
    assert s_max > 800.0
    perm = prng.make_perm(6, 0, 0, 24)[None]
    for causal in (False, True):
        want = _sdpa(q, k, c.v, causal=causal)
        got = attention.sa_forward(q, k, c.v, perm, 48, causal)
        assert np.isfinite(got).all()
        np.testing.assert_allclose(got, want, atol=1e-10)
        got = attention.full_attention(q, k, c.v, causal)
        assert np.isfinite(got).all()
        np.testing.assert_allclose(got, want, atol=1e-10)


def test_argument_checks():
    """Empty and impossible inputs: an empty shuffle is empty; a window below 1,
    a negative length or a query with no key is rejected."""
    assert prng.fisher_yates(0, lambda: 0).tolist() == []
    with pytest.raises(ValueError):
        prng.fisher_yates(-1, lambda: 0)
    with pytest.raises(ValueError):
        graph.half_width(0)
    with pytest.raises(ValueError):
        graph.neighbours_swa(5, 0, 2)
    c = _case(b=1, n=4, hq=1, hkv=1, d=8)
    mask = np.ones((4, 4), dtype=bool)
    attention.masked_attention(c.q, c.k, c.v, mask)
    mask[2] = False
    with pytest.raises(ValueError):
        attention.masked_attention(c.q, c.k, c.v, mask)


def test_identity_perm_is_banded_attention():
    c = _case(n=37)
    n = 37
    ident = np.tile(np.arange(n), (2, 1))
    for w in (1, 2, 7, 10):
        h = w // 2
        i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
        band = np.abs(i - j) <= h
        got = attention.sa_forward(c.q, c.k, c.v, ident, w, causal=False)
        np.testing.assert_allclose(got, _sdpa(c.q, c.k, c.v, mask=band), atol=1e-12)
        # causal SA with sigma = id is SWA over the h+1 trailing keys
        got_c = attention.sa_forward(c.q, c.k, c.v, ident, w, causal=True)
        np.testing.assert_allclose(got_c, attention.swa_forward(c.q, c.k, c.v, h + 1), atol=1e-12)
        trail = (j <= i) & (j >= i - h)
        np.testing.assert_allclose(got_c, _sdpa(c.q, c.k, c.v, mask=trail), atol=1e-12)


def test_swa_matches_masked_sdpa():
    c = _case(n=50)
    i, j = np.meshgrid(np.arange(50), np.arange(50), indexing="ij")
    for w in (1, 5, 16, 80):
        mask = (j <= i) & (j >= i - w + 1)
        np.testing.assert_allclose(attention.swa_forward(c.q, c.k, c.v, w),
                                   _sdpa(c.q, c.k, c.v, mask=mask), atol=1e-12)


def test_wide_window_is_full_attention():
    c = _case(n=24)
    perm = np.stack([prng.make_perm(1, 0, b, 24) for b in range(2)])
    full_w = 2 * 24
    np.testing.assert_allclose(attention.sa_forward(c.q, c.k, c.v, perm, full_w, False),
                               _sdpa(c.q, c.k, c.v), atol=1e-12)
    np.testing.assert_allclose(attention.sa_forward(c.q, c.k, c.v, perm, full_w, True),
                               _sdpa(c.q, c.k, c.v, causal=True), atol=1e-12)
    # w = n is NOT enough under |p - q| <= w/2: some pairs stay apart
    diff = np.abs(attention.sa_forward(c.q, c.k, c.v, perm, 24, False) - _sdpa(c.q, c.k, c.v))
    assert diff.max() > 1e-6


@pytest.mark.parametrize("causal", [False, True])
def test_permuted_space_route_agrees(causal):
    """Steps 1-3 literally (permute, banded attention in permuted space with
    the causal rule sigma(q) <= sigma(p), scatter back by sigma) must agree
    with the oracle's per-token neighbour-set route."""
    c = _case(n=45)
    n, w = 45, 8
    h = w // 2
    out = np.empty_like(c.q, dtype=np.float64)
    perm = np.stack([prng.make_perm(9, 2, b, n) for b in range(2)])
    for b in range(2):
        s = perm[b]
        pq, pk, pv = c.q[b:b + 1, s], c.k[b:b + 1, s], c.v[b:b + 1, s]
        p, qq = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
        mask = np.abs(p - qq) <= h
        if causal:
            mask &= s[qq] <= s[p]
        yp = _sdpa(pq, pk, pv, mask=mask)
        out[b, s] = yp[0]
    np.testing.assert_allclose(attention.sa_forward(c.q, c.k, c.v, perm, w, causal), out,
                               atol=1e-12)


def test_relabelling_equivariance_noncausal():
    c = _case(b=1, n=30)
    n, w = 30, 6
    sigma = prng.make_perm(3, 0, 0, n)
    pi = prng.make_perm(4, 0, 0, n)
    pi_inv = prng.inverse_perm(pi)
    y = attention.sa_forward(c.q, c.k, c.v, sigma[None], w, False)
    sigma_t = pi_inv[sigma]
    y_t = attention.sa_forward(c.q[:, pi], c.k[:, pi], c.v[:, pi], sigma_t[None], w, False)
    np.testing.assert_allclose(y_t, y[:, pi], atol=1e-13)


def test_gate_limits_reduce_to_single_paths():
    c = _case(n=20)
    perm = np.stack([prng.make_perm(0, 0, b, 20) for b in range(2)])
    w = 6
    y_sa = attention.sa_forward(c.q, c.k, c.v, perm, w, True)
    y_swa = attention.swa_forward(c.q, c.k, c.v, w)
    big = np.full(c.gate_sa.shape, 40.0)
    got = attention.gated_forward(c.q, c.k, c.v, perm, big, -big, w)
    np.testing.assert_allclose(got, y_sa, atol=1e-15)
    got = attention.gated_forward(c.q, c.k, c.v, perm, -big, big, w)
    np.testing.assert_allclose(got, y_swa, atol=1e-15)
    got = attention.gated_forward(c.q, c.k, c.v, perm, big, big, w)
    np.testing.assert_allclose(got, y_sa + y_swa, atol=1e-15)
    zero = np.zeros_like(big)
    got = attention.gated_forward(c.q, c.k, c.v, perm, zero, zero, w)
    np.testing.assert_allclose(got, 0.5 * (y_sa + y_swa), atol=1e-15)
    assert attention.sigmoid(np.array([-1000.0]))[0] == 0.0


def test_gated_merge_with_arbitrary_logits_uses_the_logistic_function():
    """Y = sigmoid(a_sa) Y_sa + sigmoid(a_swa) Y_swa ("Gated SA and SWA"
    equation) at ordinary logit values, with the logistic function taken from
    scipy rather than the oracle."""
    special = pytest.importorskip("scipy.special")
    c = _case(n=20)
    perm = np.stack([prng.make_perm(0, 2, b, 20) for b in range(2)])
    w = 6
    a_sa = 1.5 * np.asarray(c.gate_sa, dtype=np.float64)
    a_swa = 1.5 * np.asarray(c.gate_swa, dtype=np.float64)
    got = attention.gated_forward(c.q, c.k, c.v, perm, a_sa, a_swa, w)
    want = (special.expit(a_sa)[..., None] * attention.sa_forward(c.q, c.k, c.v, perm, w, True)
            + special.expit(a_swa)[..., None] * attention.swa_forward(c.q, c.k, c.v, w))
    np.testing.assert_allclose(got, want, atol=1e-14)


def test_gated_swa_window_is_its_own():
    """With window_swa set, the SWA branch of the gated sum uses it, not w."""
    c = _case(n=20)
    perm = np.stack([prng.make_perm(0, 1, b, 20) for b in range(2)])
    big = np.full(c.gate_sa.shape, 40.0)
    got = attention.gated_forward(c.q, c.k, c.v, perm, -big, big, 8, 3)
    np.testing.assert_allclose(got, attention.swa_forward(c.q, c.k, c.v, 3), atol=1e-15)
    assert np.abs(got - attention.swa_forward(c.q, c.k, c.v, 8)).max() > 1e-3
    got = attention.gated_forward(c.q, c.k, c.v, perm, big, -big, 8, 3)
    np.testing.assert_allclose(got, attention.sa_forward(c.q, c.k, c.v, perm, 8, True), atol=1e-15)
    # window_swa <= 0 means "the same window as SA"
    got = attention.gated_forward(c.q, c.k, c.v, perm, -big, big, 8, 0)
    np.testing.assert_allclose(got, attention.swa_forward(c.q, c.k, c.v, 8), atol=1e-15)


def test_gqa_head_map_and_scale_pinned_by_sdpa():
    c = _case(b=1, n=12, hq=6, hkv=3, d=8)
    perm = np.arange(12)[None]
    got = attention.sa_forward(c.q, c.k, c.v, perm, 100, False, scale=0.3)
    np.testing.assert_allclose(got, _sdpa(c.q, c.k, c.v, scale=0.3), atol=1e-12)


def test_rows_subset_matches_full():
    c = _case(n=30)
    perm = np.stack([prng.make_perm(2, 0, b, 30) for b in range(2)])
    full = attention.gated_forward(c.q, c.k, c.v, perm, c.gate_sa, c.gate_swa, 8, 5)
    rows = [(1, 3), (0, 29), (1, 0)]
    sub = attention.gated_rows(c.q, c.k, c.v, perm, c.gate_sa, c.gate_swa, 8, 5, rows=rows)
    for r, (b, i) in enumerate(rows):
        np.testing.assert_array_equal(sub[r], full[b, i])


# ---------------------------------------------------------------- shared inputs

def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32) * 3
    x[:4] = [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -0.0, 65504.0]   # ties and specials
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16_bits(x), want)
    assert np.array_equal(round_bf16(x), torch.from_numpy(x).to(torch.bfloat16).float().numpy())
