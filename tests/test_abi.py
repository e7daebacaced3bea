"""The C-ABI library builds, loads and exports what include/libsa.h declares.

CPU only: nothing here launches a kernel.  The host-side sigma generator is
checked bit-exactly against the oracle's own implementation, and argument
validation is checked on calls that are rejected before any CUDA call.
"""

from __future__ import annotations

import ctypes
import re
from pathlib import Path

import numpy as np
import pytest

import oracle
import stochastic_sliding_window_gb300 as sa

HEADER = Path(__file__).resolve().parents[1] / "include" / "libsa.h"


def _declared_functions() -> set[str]:
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                           text, flags=re.M))
    return {n for n in names if n.startswith("sa_") or n.startswith("swa_")}


def test_library_exports_every_declared_symbol():
    lib = sa.load()
    declared = _declared_functions()
    assert {"sa_forward", "swa_forward", "sa_swa_gated_forward", "sa_inverse_perm",
            "sa_make_perm"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
        assert name in sa.SIGNATURES, name
    assert set(sa.SIGNATURES) == declared


def test_status_strings():
    lib = sa.load()
    for st in range(7):
        s = lib.sa_status_string(st).decode()
        assert s.startswith("SA_")
    assert "unknown" in lib.sa_status_string(99).decode()


@pytest.mark.parametrize("seed,layer,b,n", [
    (0, 0, 0, 1), (0, 0, 0, 2), (1, 0, 0, 257), (123456789, 7, 3, 1000),
    ((1 << 64) - 1, 2, 1, 333), (42, 1000, 0, 4096), (2 ** 40 + 5, 0, 12, 65),
])
def test_host_perm_generator_is_bit_exact_with_oracle(seed, layer, b, n):
    got = sa.make_perm(seed, layer, b, n)
    want = oracle.make_perm(seed, layer, b, n)
    assert got.dtype == np.int32
    assert np.array_equal(got.astype(np.int64), want)


def test_host_perm_generator_rejects_bad_args():
    lib = sa.load()
    buf = (ctypes.c_int32 * 4)()
    assert lib.sa_make_perm(0, -1, 0, 4, buf) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_make_perm(0, 0, -1, 4, buf) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_make_perm(0, 0, 0, 0, buf) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_make_perm(0, 0, 0, 4, None) == sa.SA_ERR_INVALID_ARG
    assert "layer" in lib.sa_last_error_message().decode() or \
        "NULL" in lib.sa_last_error_message().decode()


def _params(**kw):
    base = dict(batch=1, seqlen=16, num_q_heads=4, num_kv_heads=2, head_dim=64, window=4,
                window_swa=0, causal=1, softmax_scale=0.0, kernel=0, err=None)
    base.update(kw)
    return sa.SaParams(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(batch=0), 1), (dict(seqlen=0), 1), (dict(num_q_heads=3), 1), (dict(head_dim=96), 2),
    (dict(window=0), 1), (dict(kernel=7), 1), (dict(kernel=-1), 1),
    # sizes whose token or row index would not fit 32 bits
    (dict(batch=65536, seqlen=65536), 2),
    (dict(batch=1, seqlen=1 << 27, num_q_heads=16, num_kv_heads=2), 2),
])
def test_forward_argument_validation_without_gpu(kw, status):
    lib = sa.load()
    prm = _params(**kw)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    st = lib.sa_forward(ctypes.byref(prm), fake, fake, fake, fake, ctypes.c_void_p(0x20000), None)
    assert st == status
    assert lib.sa_last_error_message().decode() != ""


def test_null_and_misaligned_pointers_rejected():
    lib = sa.load()
    prm = _params()
    good = ctypes.c_void_p(0x10000)
    assert lib.sa_forward(None, good, good, good, good, good, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_forward(ctypes.byref(prm), None, good, good, good,
                          ctypes.c_void_p(0x20000), None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_forward(ctypes.byref(prm), ctypes.c_void_p(0x10008), good, good, good,
                          ctypes.c_void_p(0x20000), None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_forward(ctypes.byref(prm), good, good, good, None,
                          ctypes.c_void_p(0x20000), None) == sa.SA_ERR_INVALID_ARG
    # out aliasing an input
    assert lib.sa_forward(ctypes.byref(prm), good, ctypes.c_void_p(0x30000),
                          ctypes.c_void_p(0x40000), good, good, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_swa_gated_forward(ctypes.byref(prm), good, ctypes.c_void_p(0x30000),
                                    ctypes.c_void_p(0x40000), good, None, good,
                                    ctypes.c_void_p(0x50000), None, 0, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_inverse_perm(good, good, 1, 16, None, None) == sa.SA_ERR_INVALID_ARG  # overlap
    assert lib.sa_inverse_perm(good, ctypes.c_void_p(0x30000), 0, 16, None, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_gated_workspace_size(ctypes.byref(prm)) == 0


def test_params_struct_layout_matches_header():
    # sa_params_t: ten 4-byte fields then one pointer (8-byte aligned).
    assert ctypes.sizeof(sa.SaParams) == 48
    assert sa.SaParams.err.offset == 40
    assert sa.SaParams.softmax_scale.offset == 32


def test_binding_constants_match_the_header():
    """Status codes, kernel selectors and error bits of the Python binding are
    the values include/libsa.h declares."""
    text = (Path(__file__).resolve().parents[1] / "include" / "libsa.h").read_text()
    enum = dict((m.group(1), int(m.group(2)))
                for m in re.finditer(r"\b(SA_(?:OK|ERR_\w+|KERNEL_\w+))\s*=\s*(\d+)", text))
    defines = dict((m.group(1), int(m.group(2)))
                   for m in re.finditer(r"#define\s+(SA_ERRBIT_\w+)\s+(\d+)", text))
    assert len(enum) == 13 and len(defines) == 4
    for name, value in enum.items():
        py = name if name.startswith("SA_OK") or name.startswith("SA_ERR_") else name[3:]
        assert getattr(sa, py) == value, name
    for name, value in defines.items():
        assert getattr(sa, name[3:]) == value, name
