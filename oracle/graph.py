"""Neighbour sets and connectivity statistics of SA and SWA (oracle side).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Definitions ("Stochastic Attention" summary, section "Core mechanism"):

* SA, non-causal: token i sits at permuted position p = sigma^{-1}(i) and
  attends to the tokens at permuted positions q with |q - p| <= h,
  h = floor(w / 2), truncated at the sequence ends (no wrap-around):
      N(i) = { sigma[q] : |q - p| <= h, 0 <= q < n }.
* SA, causal ("Theoretical properties", causal-constraint bullet): the mask is
  applied in permuted space and a token only sees tokens that precede it in
  the ORIGINAL order:  N_c(i) = { j in N(i) : j <= i }.  i is in both sets.
* SWA ("Problem statement"; keys of the previous w tokens including i):
      N_swa(i) = [max(0, i - w + 1), i].
"""

from __future__ import annotations

import numpy as np

from .prng import inverse_perm


def half_width(window: int) -> int:
    """SA half-width h = floor(w / 2): the window |p - q| <= w/2 of "Core
    mechanism", step 2; the pages leave odd w open and floor is taken."""
    if window < 1:
        raise ValueError("window must be >= 1")
    return window // 2


def neighbours_sa(perm: np.ndarray, window: int, causal: bool, i: int,
                  inv: np.ndarray | None = None) -> np.ndarray:
    """Sorted original-token indices that token i attends to under SA.

    "Core mechanism", steps 1-3: token i sits at permuted position
    p = sigma^-1(i) and attends to the tokens at permuted positions within
    distance h of p, truncated at the sequence ends.  Causal ("Theoretical
    properties", causal-constraint bullet): only keys whose original index
    does not exceed i."""
    perm = np.asarray(perm)
    n = perm.shape[0]
    if inv is None:
        inv = inverse_perm(perm)
    h = half_width(window)
    p = int(inv[i])
    lo, hi = max(0, p - h), min(n - 1, p + h)
    keys = [int(perm[q]) for q in range(lo, hi + 1)]
    if causal:
        keys = [j for j in keys if j <= i]
    return np.asarray(sorted(keys), dtype=np.int64)


def neighbours_swa(n: int, window: int, i: int) -> np.ndarray:
    """Original-token indices that token i attends to under SWA: the local
    window of size w ending at i ("Problem statement"), clipped at 0."""
    if window < 1:
        raise ValueError("window must be >= 1")
    return np.arange(max(0, i - window + 1), i + 1, dtype=np.int64)


def adjacency_sa(perm: np.ndarray, window: int, causal: bool) -> np.ndarray:
    """Boolean A[i, j] = (j in N(i)) for one sequence, built token by token:
    the random neighbourhood graph of "Core mechanism", closing paragraph."""
    perm = np.asarray(perm)
    n = perm.shape[0]
    inv = inverse_perm(perm)
    a = np.zeros((n, n), dtype=bool)
    for i in range(n):
        a[i, neighbours_sa(perm, window, causal, i, inv)] = True
    return a


def adjacency_swa(n: int, window: int) -> np.ndarray:
    """Boolean A[i, j] = (j in N_swa(i)): SWA's banded graph ("Problem
    statement")."""
    a = np.zeros((n, n), dtype=bool)
    for i in range(n):
        a[i, neighbours_swa(n, window, i)] = True
    return a


def attended_pairs_closed_form(n: int, window: int, path: str, causal: bool = True) -> int:
    """Exact number of (query, key) pairs attended in one sequence: the
    linear O(n w) work of "Theoretical properties" and "Results / Efficiency".

    Independent of sigma: the window covers the same set of permuted position
    pairs for every sigma.  Non-causal SA counts every ordered pair at
    permuted distance <= h; causal SA keeps, of each unordered pair at
    distance 1..h, exactly the one edge from the later token to the earlier;
    SWA counts min(i + 1, w) keys for token i.
    """
    if path == "sa":
        h = min(half_width(window), n - 1) if n > 0 else 0
        far = sum(n - d for d in range(1, h + 1))
        return n + (far if causal else 2 * far)
    if path == "swa":
        w = min(window, n)
        return w * (w + 1) // 2 + (n - w) * w
    raise ValueError(path)


def pair_probability_closed_form(n: int, window: int) -> float:
    """P(j in N(i)) for a fixed pair i != j (j < i when causal), sigma uniform.

    Under a uniform sigma the permuted positions of i and j are a uniformly
    random ordered pair of distinct positions; of the n(n-1) such pairs,
    2 * sum_{d=1..h} (n - d) = 2hn - h(h+1) lie within distance h.  The pages
    state this probability is about w/n ("Core mechanism", last paragraph).
    """
    h = min(half_width(window), n - 1)
    return (2 * h * n - h * (h + 1)) / (n * (n - 1))


def expected_degree_closed_form(n: int, window: int) -> float:
    """E|N(i)| for non-causal SA averaged over tokens: 1 + (2hn - h(h+1))/n.
    The pages give the neighbourhood's expected size as about w ("Core
    mechanism", closing paragraph)."""
    h = min(half_width(window), n - 1)
    return 1.0 + (2 * h * n - h * (h + 1)) / n


def receptive_field_sizes(adjacencies: list[np.ndarray]) -> np.ndarray:
    """Receptive fields over stacked layers ("Theoretical properties",
    receptive-field bullet): |R_l(i)| for l = 1..L, where R_0(i) = {i} and
    R_l(i) = union over j in N_l(i) of R_{l-1}(j)  (layer 1 acts first).

    ``adjacencies[l-1]`` is layer l's boolean A[i, j] = (j in N_l(i)).
    Returns int64 [L, n].
    """
    n = adjacencies[0].shape[0]
    reach = np.eye(n, dtype=bool)
    sizes = []
    for a in adjacencies:
        reach = (a.astype(np.int64) @ reach.astype(np.int64)) > 0
        sizes.append(reach.sum(axis=1))
    return np.asarray(sizes, dtype=np.int64)
