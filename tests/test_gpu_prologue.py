"""GPU parity of the gate projection GEMM and of RoPE by original token index
(sa_gate_projection, sa_rope through the C ABI) against the fp64 oracle, and
of each feeding the attention paths end to end.

Tolerances: the gate logits are fp32 sums of exact bf16 x bf16 products, so
they match the fp64 oracle to relative-L2 1e-5.  RoPE rounds each rotated
value to bf16 once (unit roundoff 2^-8): max-abs 1e-2 * max(1, max|ref|),
relative-L2 5e-3.  End-to-end outputs keep the attention bar (max-abs 2e-2,
relative-L2 5e-3)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import stochastic_sliding_window_gb300 as sa
from gpu_helpers import compare, dev_bf16, dev_f32, perms
from sa_synth import make_case, round_bf16

pytestmark = pytest.mark.gpu


def _rel(g, w):
    return float(np.linalg.norm(g - w) / max(np.linalg.norm(w), 1e-30))


@pytest.mark.parametrize("b,n,dm,hq,bias", [(4, 2048, 1024, 16, True), (1, 300, 64, 3, False),
                                            (2, 129, 512, 32, True), (1, 1, 128, 128, True),
                                            (3, 77, 192, 8, False)])
def test_gate_projection_matches_oracle(b, n, dm, hq, bias):
    rng = np.random.default_rng(dm + hq)
    x = round_bf16(rng.standard_normal((b, n, dm)).astype(np.float32))
    w1 = round_bf16((rng.standard_normal((hq, dm)) / np.sqrt(dm)).astype(np.float32))
    w2 = round_bf16((rng.standard_normal((hq, dm)) / np.sqrt(dm)).astype(np.float32))
    b1 = rng.standard_normal(hq).astype(np.float32) if bias else None
    b2 = rng.standard_normal(hq).astype(np.float32) if bias else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    a1, a2 = sa.gate_projection(dev_bf16(x), dev_bf16(w1), dev_bf16(w2),
                                dev_f32(b1) if bias else None, dev_f32(b2) if bias else None,
                                err=err)
    assert sa.check_error(err) == sa.SA_OK
    want1, want2 = oracle.gate_logits(x, w1, w2, b1, b2)
    for got, want in ((a1, want1), (a2, want2)):
        g = got.cpu().numpy().astype(np.float64)
        assert g.shape == want.shape
        assert _rel(g, want) <= 1e-5 and np.abs(g - want).max() <= 1e-4 * max(1, np.abs(want).max())


def test_gate_projection_feeds_the_gated_forward():
    """Pretraining-layer shape: logits from the projection drive the gated
    SA + SWA forward; the oracle composes its own projection and merge."""
    b, n, hq, d, dm, w = 2, 2048, 16, 64, 1024, 128
    c = make_case(b, n, hq, hq, d, 11, std=1.0 / 8.0, gates=False)
    rng = np.random.default_rng(4)
    x = round_bf16(rng.standard_normal((b, n, dm)).astype(np.float32))
    w1 = round_bf16((rng.standard_normal((hq, dm)) / np.sqrt(dm)).astype(np.float32))
    w2 = round_bf16((rng.standard_normal((hq, dm)) / np.sqrt(dm)).astype(np.float32))
    perm, perm_d = perms(11, 0, b, n)
    a1, a2 = sa.gate_projection(dev_bf16(x), dev_bf16(w1), dev_bf16(w2))
    y = sa.sa_swa_gated_forward(dev_bf16(c.q), dev_bf16(c.k), dev_bf16(c.v), perm_d, a1, a2, w)
    g1, g2 = oracle.gate_logits(x, w1, w2)
    rows = [(bb, i) for bb in range(b) for i in np.random.default_rng(1).integers(0, n, 150)]
    want = oracle.gated_rows(c.q, c.k, c.v, perm, g1, g2, w, None, True, rows=rows)
    got = y[torch.tensor([r[0] for r in rows]), torch.tensor([r[1] for r in rows])]
    compare(got, want, "projection -> gated forward")


@pytest.mark.parametrize("b,n,h,d,base", [(2, 333, 4, 128, 10000.0), (1, 262144, 2, 128, 10000.0),
                                          (3, 50, 8, 64, 500000.0), (1, 7, 1, 2, 10.0),
                                          (1, 100, 48, 128, 10000.0),  # 3 items per thread
                                          (2, 61, 3, 12, 10000.0),     # 4-byte accesses
                                          (1, 9, 5, 16, 10000.0)])     # partial last block
def test_rope_matches_oracle(b, n, h, d, base):
    rng = np.random.default_rng(n + d)
    x = round_bf16(rng.standard_normal((b, n, h, d)).astype(np.float32))
    xd = dev_bf16(x)
    sa.rope_(xd, base)
    g = xd.float().cpu().numpy().astype(np.float64)
    want = oracle.rope(x, base)
    assert np.abs(g - want).max() <= 1e-2 * max(1.0, np.abs(want).max())
    assert _rel(g, want) <= 5e-3


def test_rope_unaligned_rows_use_narrow_accesses():
    """A tensor whose data starts 4 bytes past a 16-byte boundary takes the
    4-byte path and gives the same result."""
    rng = np.random.default_rng(5)
    x = round_bf16(rng.standard_normal((2, 40, 4, 64)).astype(np.float32))
    buf = torch.empty(x.size + 2, dtype=torch.bfloat16, device="cuda")
    xd = buf[2:].view(x.shape)
    xd.copy_(dev_bf16(x))
    assert xd.data_ptr() % 16 == 4
    sa.rope_(xd, 10000.0)
    g = xd.float().cpu().numpy().astype(np.float64)
    want = oracle.rope(x, 10000.0)
    assert np.abs(g - want).max() <= 1e-2 * max(1.0, np.abs(want).max())
    assert _rel(g, want) <= 5e-3


def test_rope_odd_element_offset_uses_2byte_accesses():
    """Data starting 2 bytes past a 4-byte boundary takes the 2-byte path."""
    rng = np.random.default_rng(6)
    x = round_bf16(rng.standard_normal((1, 30, 3, 32)).astype(np.float32))
    buf = torch.empty(x.size + 1, dtype=torch.bfloat16, device="cuda")
    xd = buf[1:].view(x.shape)
    xd.copy_(dev_bf16(x))
    assert xd.data_ptr() % 4 == 2
    sa.rope_(xd, 10000.0)
    g = xd.float().cpu().numpy().astype(np.float64)
    want = oracle.rope(x, 10000.0)
    assert np.abs(g - want).max() <= 1e-2 * max(1.0, np.abs(want).max())
    assert _rel(g, want) <= 5e-3


def test_rope_then_causal_sa():
    """RoPE on Q and K by original index, then causal SA over the permuted
    order (long-prefill GQA heads, n = 4096): the oracle rotates in fp64,
    stores bf16 like the library, then attends."""
    b, n, hq, hkv, d, w = 1, 4096, 32, 8, 128, 128
    c = make_case(b, n, hq, hkv, d, 23, gates=False)
    perm, perm_d = perms(23, 0, b, n)
    q, k = dev_bf16(c.q), dev_bf16(c.k)
    sa.rope_(q)
    sa.rope_(k)
    y = sa.sa_forward(q, k, dev_bf16(c.v), perm_d, w, causal=True)
    rq, rk = round_bf16(oracle.rope(c.q).astype(np.float32)), round_bf16(oracle.rope(c.k).astype(np.float32))
    rows = [(0, int(i)) for i in np.random.default_rng(2).integers(0, n, 200)]
    want = oracle.sa_rows(rq, rk, c.v, perm, w, True, rows=rows)
    got = y[0, torch.tensor([r[1] for r in rows])]
    compare(got, want, "rope -> causal SA")
