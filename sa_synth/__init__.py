"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds NO attention arithmetic: it draws seeded normal arrays,
rounds them to bfloat16 (round-to-nearest-even on the fp32 bit pattern) and
names the workload shapes.  It is the only module that both the oracle tests
and the library tests import, so that both sides read identical values.

The permutation sigma is NOT drawn here: the oracle and the library each
implement the seeded splitmix64 / Fisher-Yates generator on their own.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bfloat16 bit patterns (uint16), round-to-nearest-even.

    Inputs are finite (seeded normals); NaN handling is not needed."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((bits >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((bits + rounding) >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact fp32 values."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 values rounded to the nearest bfloat16, returned as fp32."""
    return bf16_to_f32(bf16_bits(x))


@dataclass
class Case:
    """One seeded input set.  q/k/v are fp32 arrays holding bf16-exact values
    (the kernels read the same numbers as bf16); gates are fp32."""
    batch: int
    seqlen: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    seed: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    gate_sa: np.ndarray | None = None
    gate_swa: np.ndarray | None = None
    meta: dict = field(default_factory=dict)


def make_case(batch: int, seqlen: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
              seed: int, std: float | None = None, gates: bool = False,
              bf16: bool = True) -> Case:
    """Q [B,n,Hq,d], K/V [B,n,Hkv,d] ~ N(0, std^2) (std defaults to 1/sqrt(d)),
    drawn in the order Q, K, V, gate_sa, gate_swa from PCG64(seed); gate logits
    [B,n,Hq] ~ N(0, 1)."""
    std = (1.0 / np.sqrt(head_dim)) if std is None else std
    rng = np.random.Generator(np.random.PCG64(seed))

    def draw(shape, s):
        x = (rng.standard_normal(shape, dtype=np.float32) * np.float32(s)).astype(np.float32)
        return round_bf16(x) if bf16 else x

    q = draw((batch, seqlen, num_q_heads, head_dim), std)
    k = draw((batch, seqlen, num_kv_heads, head_dim), std)
    v = draw((batch, seqlen, num_kv_heads, head_dim), std)
    ga = gw = None
    if gates:
        ga = rng.standard_normal((batch, seqlen, num_q_heads), dtype=np.float32)
        gw = rng.standard_normal((batch, seqlen, num_q_heads), dtype=np.float32)
    return Case(batch, seqlen, num_q_heads, num_kv_heads, head_dim, seed, q, k, v, ga, gw)


# Workload shapes of the method's published use: the tiny oracle case, a
# pretraining-layer shape, the long-prefill GQA sweep, very long context and
# the length sweep.  (name -> dict of shape fields)
WORKLOADS = {
    "tiny": dict(batch=1, seqlen=256, num_q_heads=2, num_kv_heads=2, head_dim=64,
                 windows=(32,), std=1.0 / 8.0, paths=("sa", "sa_causal", "swa", "gated")),
    "pretrain_layer": dict(batch=4, seqlen=2048, num_q_heads=16, num_kv_heads=16, head_dim=64,
                           windows=(128,), std=1.0 / 8.0, paths=("gated",)),
    "long_prefill_gqa": dict(batch=1, seqlen=32768, num_q_heads=32, num_kv_heads=8, head_dim=128,
                             windows=(32, 64, 128, 256), std=None, paths=("sa_causal",)),
    "very_long_context": dict(batch=1, seqlen=131072, num_q_heads=32, num_kv_heads=4,
                              head_dim=128, windows=(1024, 2048), std=None, paths=("gated",)),
    "length_sweep": dict(batch=1, seqlens=(2048, 8192, 32768, 131072, 262144), num_q_heads=16,
                         num_kv_heads=16, head_dim=128, windows=(128,), std=None, layers=8,
                         paths=("sa_causal",)),
}
