"""Shared helpers of the GPU parity tests (inputs, comparison, tolerances)."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import stochastic_sliding_window_gb300 as sa
from sa_synth import make_case

# bf16 kernels against the fp64 oracle: max-abs and relative-L2 bounds.
MAX_ABS = 2e-2
REL_L2 = 5e-3

KERNELS = [sa.KERNEL_SIMT, sa.KERNEL_TCGEN05_GATHER, sa.KERNEL_TCGEN05_RING,
           sa.KERNEL_TCGEN05_CHUNK]
KERNEL_IDS = ["simt", "gather", "ring", "chunk"]


def span(path: str, g: int, w: int) -> int:
    """Keys of one tile's window: Bt = 128/g positions plus the halo."""
    bt = 128 // g
    return bt + 2 * (w // 2) if path == "sa" else bt + w - 1


def _ring_fits(sp: int, g: int, d: int) -> bool:
    """The ring kernel's resources: 2 Q stages, K and V rings of span + 2 Bt
    rows, the doubled sigma ring, two new-token lists, four buffers of mask
    words and 31 barriers in 227 KB of shared memory; spans of at most 256
    keys; two TMEM stages in 512 columns."""
    rnd = lambda x, m: -(-x // m) * m
    pad = rnd(sp, 32)
    bt = 128 // g
    r = rnd(pad + 2 * bt, 16)
    off_sig = 2 * 128 * d * 2 + 2 * r * d * 2
    off_vtok = rnd(off_sig + 2 * r * 4, 16)
    off_bits = rnd(off_vtok + 2 * pad * 4, 16)
    off_bar = rnd(off_bits + 4 * bt * (pad // 32) * 4, 64)
    smem = off_bar + 8 * 31 + 32 + 1024
    cols = rnd(max(pad, pad // 2 + d), 32)
    return pad <= 256 and smem <= 232448 and 2 * cols <= 512


def must_support(kernel: int, path: str, g: int, w: int, w_swa: int = 0, d: int = 128) -> bool:
    """Shapes each tcgen05 variant is required to accept (the ring kernel
    exactly; the chunk kernel any window; the gather kernel at least up to
    256-key windows)."""
    if kernel == sa.KERNEL_SIMT:
        return True
    if 128 % g:
        return False
    if kernel == sa.KERNEL_TCGEN05_CHUNK:
        return d in (64, 128) and g <= 32
    paths = [("sa", w), ("swa", w_swa or w)] if path == "gated" else [(path, w)]
    if kernel == sa.KERNEL_TCGEN05_RING:
        return (128 // g) % 16 == 0 and all(_ring_fits(span(pp, g, ww), g, d) for pp, ww in paths)
    return all(span(pp, g, ww) <= 256 for pp, ww in paths)


def kernel_ran(requested: int) -> bool:
    got = sa.last_kernel()
    if requested == sa.KERNEL_TCGEN05:
        return got in (sa.KERNEL_TCGEN05_GATHER, sa.KERNEL_TCGEN05_RING, sa.KERNEL_TCGEN05_CHUNK)
    return got == requested


def dev_bf16(x: np.ndarray) -> torch.Tensor:
    """Upload fp32 values that are already bf16-exact (conversion is exact)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to("cuda").to(torch.bfloat16)


def dev_f32(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to("cuda")


def perms(seed: int, layer: int, batch: int, n: int) -> tuple[np.ndarray, torch.Tensor]:
    """sigma from the oracle's generator and the library's; they must agree."""
    ora = np.stack([oracle.make_perm(seed, layer, b, n) for b in range(batch)])
    lib = sa.make_perms(seed, layer, batch, n)
    assert np.array_equal(ora, lib.astype(np.int64))
    return ora, torch.from_numpy(lib).to("cuda")


class Inputs:
    def __init__(self, batch, n, hq, hkv, d, seed=0, std=None, gates=True):
        self.case = make_case(batch, n, hq, hkv, d, seed, std=std, gates=gates)
        c = self.case
        self.q, self.k, self.v = dev_bf16(c.q), dev_bf16(c.k), dev_bf16(c.v)
        if gates:
            self.ga, self.gw = dev_f32(c.gate_sa), dev_f32(c.gate_swa)
        self.shape = (batch, n, hq, hkv, d)


def compare(got: torch.Tensor, want: np.ndarray, what: str = ""):
    g = got.float().cpu().numpy().astype(np.float64)
    assert g.shape == want.shape, (g.shape, want.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - want)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(g - want)) / denom if denom > 0 else float(np.linalg.norm(g))
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    return max_abs, rel


def sample_rows(batch: int, n: int, count: int, seed: int = 0) -> list[tuple[int, int]]:
    """Seeded sample of (b, i) rows that always includes both sequence ends."""
    rng = np.random.default_rng(seed)
    rows = {(0, 0), (0, n - 1), (batch - 1, 0), (batch - 1, n - 1), (0, min(1, n - 1))}
    while len(rows) < min(count, batch * n):
        rows.add((int(rng.integers(batch)), int(rng.integers(n))))
    return sorted(rows)


def gather_rows(y: torch.Tensor, rows) -> torch.Tensor:
    b = torch.tensor([r[0] for r in rows], device=y.device)
    i = torch.tensor([r[1] for r in rows], device=y.device)
    return y[b, i]
