"""The Python binding rejects malformed arguments before anything reaches the
C ABI (which trusts the sizes it is given), and the wait-bound hook round-trips.

CPU only: shape, dtype and rank checks run before the device checks, so
wrong-shaped CPU tensors are enough to reach them; correctly shaped CPU
tensors are then refused for not being on a CUDA device.  Nothing launches.
"""

from __future__ import annotations

import pytest
import torch

import stochastic_sliding_window_gb300 as sa

B, N, HQ, HKV, D = 2, 64, 8, 2, 64


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def _good():
    return dict(q=_t(B, N, HQ, D), k=_t(B, N, HKV, D), v=_t(B, N, HKV, D),
                perm=_t(B, N, dtype=torch.int32), out=_t(B, N, HQ, D),
                ga=_t(B, N, HQ, dtype=torch.float32), gw=_t(B, N, HQ, dtype=torch.float32),
                err=_t(1, dtype=torch.int32))


def _sa(a):
    return sa.sa_forward(a["q"], a["k"], a["v"], a["perm"], 16, out=a["out"], err=a["err"])


def _gated(a):
    return sa.sa_swa_gated_forward(a["q"], a["k"], a["v"], a["perm"], a["ga"], a["gw"], 16,
                                   out=a["out"], err=a["err"])


def _swa(a):
    return sa.swa_forward(a["q"], a["k"], a["v"], 16, out=a["out"], err=a["err"])


BAD = [
    ("out", _t(B, N, HQ, D // 2), "out"),
    ("out", _t(B, N - 1, HQ, D), "out"),
    ("out", _t(B, N, HKV, D), "out"),
    ("perm", _t(1, N, dtype=torch.int32), "perm"),
    ("perm", _t(B, N + 1, dtype=torch.int32), "perm"),
    ("ga", _t(B, N, HKV, dtype=torch.float32), "gate_sa"),
    ("gw", _t(B, N - 3, HQ, dtype=torch.float32), "gate_swa"),
    ("v", _t(B, N, HKV + 1, D), "v"),
    ("k", _t(B, N // 2, HKV, D), "k"),
]


@pytest.mark.parametrize("field,bad,name", BAD, ids=[f"{b[0]}{tuple(b[1].shape)}" for b in BAD])
@pytest.mark.parametrize("call", [_sa, _gated, _swa], ids=["sa", "gated", "swa"])
def test_wrong_shapes_raise_before_launch(call, field, bad, name):
    a = _good()
    a[field] = bad
    if call is _swa and field in ("perm", "ga", "gw"):
        pytest.skip("argument not taken by swa_forward")
    if call is _sa and field in ("ga", "gw"):
        pytest.skip("argument not taken by sa_forward")
    with pytest.raises(ValueError, match=name):
        call(a)


@pytest.mark.parametrize("field,bad", [
    ("q", _t(B, N, HQ, D, dtype=torch.float16)),
    ("perm", _t(B, N, dtype=torch.int64)),
    ("ga", _t(B, N, HQ, dtype=torch.float64)),
    ("err", _t(1, dtype=torch.int64)),
    ("err", _t(0, dtype=torch.int32)),
])
def test_wrong_dtypes_raise_before_launch(field, bad):
    a = _good()
    a[field] = bad
    with pytest.raises(TypeError):
        _gated(a)


def test_non_contiguous_raises():
    a = _good()
    a["q"] = _t(B, HQ, N, D).transpose(1, 2)
    with pytest.raises(ValueError, match="contiguous"):
        _sa(a)


@pytest.mark.parametrize("call", [_sa, _gated, _swa], ids=["sa", "gated", "swa"])
def test_well_formed_cpu_tensors_are_refused(call):
    with pytest.raises(ValueError, match="CUDA"):
        call(_good())


def test_inverse_perm_checks_shapes():
    perm = _t(B, N, dtype=torch.int32)
    with pytest.raises(ValueError, match="inv"):
        sa.sa_inverse_perm(perm, inv=_t(B, N - 1, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA"):
        sa.sa_inverse_perm(perm)


def test_wait_limit_hook_round_trips():
    default = sa.get_wait_limit()
    assert default == 4_000_000_000
    try:
        sa.set_wait_limit(1234)
        assert sa.get_wait_limit() == 1234
        sa.set_wait_limit(0)
        assert sa.get_wait_limit() == default
        sa.set_wait_limit(-5)
        assert sa.get_wait_limit() == default
    finally:
        sa.set_wait_limit(0)
