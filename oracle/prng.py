"""Seeded draw of the per-layer permutation sigma (oracle side).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

The pages say only that each layer draws sigma ~ Uniform(S_n) independently
("Stochastic Attention" summary, section "Core mechanism", step 1).  They fix
no generator, so one is fixed here that both the oracle and the library
implement separately from its published definition:

* splitmix64 (S. Vigna's public-domain generator): state += 0x9E3779B97F4A7C15,
  then the output is the state passed through two xor-shift-multiply rounds
  and a final xor-shift, all modulo 2**64.
* Stream seeding: the stream for (seed, layer, batch_index) starts from the
  OUTPUT of one splitmix64 step applied to seed + (layer << 32) + batch_index,
  so distinct (layer, batch) pairs do not give shifted copies of one stream.
* Fisher-Yates (Durstenfeld's in-place form): start from the identity; for
  i = n-1 down to 1 draw x and swap positions i and j = floor(x * (i+1) / 2**64)
  (Lemire's multiply-high range reduction, no rejection step).

Convention for applying sigma (the permuted sequence): X'[p] = X[sigma[p]].

Python integers are used for all 64-bit arithmetic, so nothing here depends on
NumPy's overflow behaviour.
"""

from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB


def splitmix64_step(state: int) -> tuple[int, int]:
    """One splitmix64 step: returns (new_state, output).

    S. Vigna's public-domain generator.  The pages ask only for
    sigma ~ Uniform(S_n) ("Core mechanism", step 1) and name no generator; this
    one is the convention fixed for both the oracle and the library."""
    state = (state + GOLDEN_GAMMA) & MASK64
    z = state
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    z ^= z >> 31
    return state, z


def stream_state(seed: int, layer: int, batch_index: int) -> int:
    """Initial splitmix64 state of the sigma stream for (seed, layer, batch).

    One stream per layer and sequence: "Core mechanism", step 1 draws an
    independent permutation for every layer."""
    if layer < 0 or batch_index < 0:
        raise ValueError("layer and batch_index must be non-negative")
    start = (seed + (layer << 32) + batch_index) & MASK64
    _, out = splitmix64_step(start)
    return out


def fisher_yates(n: int, draw) -> np.ndarray:
    """Durstenfeld shuffle of [0, n) driven by ``draw()`` -> uint64 Python int.

    With uniform draws it yields sigma ~ Uniform(S_n) ("Core mechanism",
    step 1); index j for position i is the high word of x * (i + 1).

    ``draw`` is a parameter so that tests can drive the index mapping with
    stub generators.
    """
    if n < 0:
        raise ValueError("n must be non-negative")
    sigma = list(range(n))
    for i in range(n - 1, 0, -1):
        x = draw()
        j = (x * (i + 1)) >> 64
        sigma[i], sigma[j] = sigma[j], sigma[i]
    return np.asarray(sigma, dtype=np.int64)


def make_perm(seed: int, layer: int, batch_index: int, n: int) -> np.ndarray:
    """sigma for (seed, layer, batch_index) over n tokens, as int64[n]
    ("Core mechanism", step 1: X'[p] = X[sigma[p]])."""
    state = stream_state(seed, layer, batch_index)

    def draw():
        nonlocal state
        state, out = splitmix64_step(state)
        return out

    return fisher_yates(n, draw)


def inverse_perm(perm: np.ndarray) -> np.ndarray:
    """sigma^{-1} with inv[sigma[p]] = p ("Core mechanism", step 3).

    Works on [n] or batched [B, n] arrays.  Raises ValueError if a row is not
    a permutation of [0, n).
    """
    perm = np.asarray(perm)
    squeeze = perm.ndim == 1
    rows = perm[None, :] if squeeze else perm
    inv = np.full(rows.shape, -1, dtype=np.int64)
    n = rows.shape[1]
    for b in range(rows.shape[0]):
        for p in range(n):
            i = int(rows[b, p])
            if i < 0 or i >= n or inv[b, i] != -1:
                raise ValueError("not a permutation")
            inv[b, i] = p
    return inv[0] if squeeze else inv
