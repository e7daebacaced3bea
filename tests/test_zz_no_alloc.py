"""sa_backward_noalloc: the backward pass for callers that cannot allocate
device memory where they run it (a loop whose device memory is reserved at
start-up, a framework that owns every allocation, a C caller without an
allocator).  Its scratch is a fixed array inside the library instead of a
caller workspace.  The GPU test calls it through the C ABI twice in a row, on
two different problems, and checks each result against sa_backward's on the
same inputs (the bars of the backward parity tests).  This file is collected
last so that a run stopping at its first failure has run everything else.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import stochastic_sliding_window_gb300 as sa

REL_L2 = 5e-3
ABS = 2e-2
MAX_ROWS = 1 << 20  # batch * seqlen * num_q_heads the library's scratch holds


def _params(b, n, hq, hkv, d, w, causal, err=None):
    return sa.SaParams(b, n, hq, hkv, d, w, 0, int(causal), 0.0, sa.KERNEL_AUTO,
                       ctypes.c_void_p(err.data_ptr() if err is not None else None))


def _close(got, want, what):
    g, r = got.double(), want.double()
    err = (g - r).abs().max().item()
    rel = ((g - r).norm() / r.norm().clamp_min(1e-30)).item()
    bar = ABS * max(1.0, r.abs().max().item())
    assert torch.isfinite(g).all(), what
    assert err <= bar and rel <= REL_L2, f"{what}: max_abs={err:.3e} (bar {bar:.3e}) rel_l2={rel:.3e}"


def test_rejects_problems_beyond_its_scratch_without_touching_the_gpu():
    lib = sa.load()
    prm = _params(1, MAX_ROWS // 16 + 1, 16, 16, 64, 32, True)
    st = lib.sa_backward_noalloc(ctypes.byref(prm), None, None, None, None, None, None, None,
                                 None, None)
    assert st == sa.SA_ERR_UNSUPPORTED
    assert "static scratch" in lib.sa_last_error_message().decode()


@pytest.mark.gpu
def test_noalloc_backward_matches_sa_backward_on_two_calls_in_a_row():
    lib = sa.load()
    rng = np.random.default_rng(123)
    cases = [(2, 1000, 8, 2, 128, 64, True), (1, 2048, 16, 16, 64, 128, False)]
    for b, n, hq, hkv, d, w, causal in cases:
        def bf16(*shape, s=1.0):
            return (torch.from_numpy(rng.standard_normal(shape).astype(np.float32)) * s) \
                .to("cuda").to(torch.bfloat16)
        q, k, v = bf16(b, n, hq, d, s=d ** -0.5), bf16(b, n, hkv, d, s=d ** -0.5), bf16(b, n, hkv, d)
        dout = bf16(b, n, hq, d)
        perm = torch.from_numpy(sa.make_perms(int(rng.integers(1 << 30)), 0, b, n)).to("cuda")
        want = sa.sa_backward(q, k, v, perm, dout, w, causal=causal)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(k)
        prm = _params(b, n, hq, hkv, d, w, causal, err)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        st = lib.sa_backward_noalloc(ctypes.byref(prm), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                     perm.data_ptr(), dout.data_ptr(), dq.data_ptr(),
                                     dk.data_ptr(), dv.data_ptr(), stream)
        assert st == sa.SA_OK, lib.sa_last_error_message().decode()
        assert sa.check_error(err) == sa.SA_OK
        for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), want):
            _close(got, ref, f"n={n} {name}")
