"""GPU checks of what the method's definition fixes exactly: neighbour sets,
sigma = identity, full windows, relabelling, sigma^-1, and error reporting."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import stochastic_sliding_window_gb300 as sa
from gpu_helpers import (KERNEL_IDS, KERNELS, Inputs, compare, dev_bf16, gather_rows,
                         must_support, perms, sample_rows)

pytestmark = pytest.mark.gpu


def _err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("kernel", KERNELS, ids=KERNEL_IDS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("w", [2, 9, 16])
def test_neighbour_sets_probe(kernel, causal, w):
    """Q = K = 0 makes every window weight equal and V = I exposes the
    support: row i must be 1/|N(i)| exactly on the oracle's N(i)."""
    n, d = 64, 64
    z = np.zeros((1, n, 1, d), np.float32)
    eye = np.eye(n, d, dtype=np.float32).reshape(1, n, 1, d)
    perm, perm_d = perms(77, w, 1, n)
    err = _err()
    y = sa.sa_forward(dev_bf16(z), dev_bf16(z), dev_bf16(eye), perm_d, w, causal=causal,
                      kernel=kernel, err=err)
    assert sa.check_error(err) == sa.SA_OK
    y = y.float().cpu().numpy()[0, :, 0, :]
    for i in range(n):
        nb = oracle.neighbours_sa(perm[0], w, causal, i)
        support = np.nonzero(y[i])[0]
        assert support.tolist() == nb.tolist(), (i, support, nb)
        assert np.allclose(y[i, nb], 1.0 / len(nb), rtol=2 ** -7)


@pytest.mark.parametrize("kernel", KERNELS, ids=KERNEL_IDS)
def test_identity_perm_reduces_to_windows(kernel):
    n = 400
    inp = Inputs(2, n, 8, 2, 128, seed=5, gates=False)
    ident = torch.arange(n, dtype=torch.int32, device="cuda").repeat(2, 1).contiguous()
    for w in (8, 30, 64):
        h = w // 2
        y_sa = sa.sa_forward(inp.q, inp.k, inp.v, ident, w, causal=True, kernel=kernel)
        y_swa = sa.swa_forward(inp.q, inp.k, inp.v, h + 1, kernel=kernel)
        d = (y_sa.float() - y_swa.float()).abs().max().item()
        assert d <= 2e-2
        want = oracle.swa_forward(inp.case.q, inp.case.k, inp.case.v, h + 1)
        compare(y_sa, want, f"sigma=id causal w={w}")


@pytest.mark.parametrize("kernel", KERNELS, ids=KERNEL_IDS)
def test_full_window_is_full_attention(kernel):
    n = 90
    inp = Inputs(1, n, 4, 2, 64, seed=8, gates=False)
    perm, perm_d = perms(8, 0, 1, n)
    for causal in (False, True):
        try:
            y = sa.sa_forward(inp.q, inp.k, inp.v, perm_d, 2 * n, causal=causal, kernel=kernel)
        except sa.SaError as e:
            assert e.status == sa.SA_ERR_UNSUPPORTED and not must_support(kernel, "sa", 2, 2 * n, d=64)
            continue
        want = oracle.full_attention(inp.case.q, inp.case.k, inp.case.v, causal)
        compare(y, want, f"full window causal={causal}")


@pytest.mark.parametrize("kernel", KERNELS, ids=KERNEL_IDS)
def test_relabelling_equivariance_is_bitwise(kernel):
    """SA(X o pi; pi^-1 o sigma) = SA(X; sigma) o pi: the permuted-space
    computation is identical, so the outputs agree bit for bit."""
    n = 1000
    inp = Inputs(1, n, 8, 2, 128, seed=13, gates=False)
    sigma = oracle.make_perm(1, 0, 0, n)
    pi = oracle.make_perm(2, 0, 0, n)
    sigma_t = oracle.inverse_perm(pi)[sigma]
    pi_d = torch.from_numpy(pi).to("cuda")
    s_d = torch.from_numpy(sigma.astype(np.int32))[None].to("cuda")
    st_d = torch.from_numpy(sigma_t.astype(np.int32))[None].to("cuda")
    y = sa.sa_forward(inp.q, inp.k, inp.v, s_d, 64, causal=False, kernel=kernel)
    qt, kt, vt = (x[:, pi_d].contiguous() for x in (inp.q, inp.k, inp.v))
    yt = sa.sa_forward(qt, kt, vt, st_d, 64, causal=False, kernel=kernel)
    assert torch.equal(yt, y[:, pi_d])


def test_tensor_core_and_simt_kernels_agree():
    n = 4096
    inp = Inputs(1, n, 32, 8, 128, seed=17, gates=True)
    perm, perm_d = perms(17, 0, 1, n)
    for w in (32, 64, 128):
        # ring and gather run the same MMAs; their softmax references differ
        # (span maximum against attended maximum), which changes only how p
        # rounds to bf16
        a = sa.sa_forward(inp.q, inp.k, inp.v, perm_d, w, causal=True, kernel=sa.KERNEL_TCGEN05_RING)
        b = sa.sa_forward(inp.q, inp.k, inp.v, perm_d, w, causal=True,
                          kernel=sa.KERNEL_TCGEN05_GATHER)
        assert (a.float() - b.float()).abs().max().item() <= 2e-2
    for w in (32, 128):
        # the chunk kernel streams the same windows in chunks (online softmax)
        a = sa.sa_forward(inp.q, inp.k, inp.v, perm_d, w, causal=True, kernel=sa.KERNEL_TCGEN05_RING)
        b = sa.sa_forward(inp.q, inp.k, inp.v, perm_d, w, causal=True,
                          kernel=sa.KERNEL_TCGEN05_CHUNK)
        assert (a.float() - b.float()).abs().max().item() <= 2e-2
    for w in (32, 128, 256):
        a = sa.sa_forward(inp.q, inp.k, inp.v, perm_d, w, causal=True, kernel=sa.KERNEL_TCGEN05)
        b = sa.sa_forward(inp.q, inp.k, inp.v, perm_d, w, causal=True, kernel=sa.KERNEL_SIMT)
        assert (a.float() - b.float()).abs().max().item() <= 2e-2
        a = sa.sa_swa_gated_forward(inp.q, inp.k, inp.v, perm_d, inp.ga, inp.gw, w,
                                    kernel=sa.KERNEL_TCGEN05)
        assert sa.last_launch_count() == 2
        b = sa.sa_swa_gated_forward(inp.q, inp.k, inp.v, perm_d, inp.ga, inp.gw, w,
                                    kernel=sa.KERNEL_SIMT)
        assert (a.float() - b.float()).abs().max().item() <= 2e-2


def test_auto_kernel_choice():
    inp = Inputs(1, 2048, 32, 8, 128, seed=1, gates=False)
    _, perm_d = perms(1, 0, 1, 2048)
    sa.sa_forward(inp.q, inp.k, inp.v, perm_d, 128)
    assert sa.last_kernel() == sa.KERNEL_TCGEN05_RING and sa.last_launch_count() == 1
    sa.sa_forward(inp.q, inp.k, inp.v, perm_d, 256)
    assert sa.last_kernel() == sa.KERNEL_TCGEN05_CHUNK
    sa.sa_forward(inp.q, inp.k, inp.v, perm_d, 2048)
    assert sa.last_kernel() == sa.KERNEL_TCGEN05_CHUNK
    sa.sa_forward(inp.q, inp.k, inp.v, perm_d, 2048, kernel=sa.KERNEL_TCGEN05)
    assert sa.last_kernel() == sa.KERNEL_TCGEN05_CHUNK
    sa.sa_forward(inp.q, inp.k, inp.v, perm_d, 256, kernel=sa.KERNEL_TCGEN05_GATHER)
    assert sa.last_kernel() == sa.KERNEL_TCGEN05_GATHER
    for k in (sa.KERNEL_TCGEN05_GATHER, sa.KERNEL_TCGEN05_RING):
        with pytest.raises(sa.SaError) as ei:
            sa.sa_forward(inp.q, inp.k, inp.v, perm_d, 2048, kernel=k)
        assert ei.value.status == sa.SA_ERR_UNSUPPORTED
    with pytest.raises(sa.SaError) as ei:
        sa.sa_forward(inp.q, inp.k, inp.v, perm_d, 256, kernel=sa.KERNEL_TCGEN05_RING)
    assert ei.value.status == sa.SA_ERR_UNSUPPORTED


# ------------------------------------------------------------ sigma^-1

@pytest.mark.parametrize("batch,n", [(1, 1), (3, 1000), (2, 32768), (1, 262144)])
def test_inverse_perm_bit_exact(batch, n):
    perm, perm_d = perms(99, 3, batch, n)
    err = _err()
    inv = sa.sa_inverse_perm(perm_d, err=err)
    assert sa.check_error(err) == sa.SA_OK
    want = np.stack([oracle.inverse_perm(perm[b]) for b in range(batch)])
    assert np.array_equal(inv.cpu().numpy().astype(np.int64), want)


def test_inverse_perm_reports_bad_permutations():
    n = 500
    perm, _ = perms(4, 0, 2, n)
    dup = perm.copy()
    dup[1, 10] = dup[1, 11]
    err = _err()
    sa.sa_inverse_perm(torch.from_numpy(dup.astype(np.int32)).cuda(), err=err)
    assert sa.check_error(err) == sa.SA_ERR_BAD_PERM
    assert int(err.item()) & sa.ERRBIT_DUP
    bad = perm.copy()
    bad[0, 3] = n
    err = _err()
    sa.sa_inverse_perm(torch.from_numpy(bad.astype(np.int32)).cuda(), err=err)
    assert sa.check_error(err) == sa.SA_ERR_BAD_PERM
    assert int(err.item()) & sa.ERRBIT_RANGE
    sa.clear_error(err)
    assert sa.check_error(err) == sa.SA_OK


@pytest.mark.parametrize("kernel", KERNELS, ids=KERNEL_IDS)
def test_forward_reports_out_of_range_perm_without_fault(kernel):
    n = 300
    inp = Inputs(1, n, 8, 2, 128, seed=2, gates=False)
    perm, _ = perms(2, 0, 1, n)
    bad = perm.copy()
    bad[0, 17] = n + 5
    bad[0, 200] = -3
    err = _err()
    sa.sa_forward(inp.q, inp.k, inp.v, torch.from_numpy(bad.astype(np.int32)).cuda(), 16,
                  kernel=kernel, err=err)
    assert sa.check_error(err) == sa.SA_ERR_BAD_PERM
    # the context stays usable
    _, good = perms(2, 0, 1, n)
    err2 = _err()
    sa.sa_forward(inp.q, inp.k, inp.v, good, 16, kernel=kernel, err=err2)
    assert sa.check_error(err2) == sa.SA_OK


@pytest.mark.parametrize("kernel", KERNELS, ids=KERNEL_IDS)
@pytest.mark.parametrize("path", ["sa", "swa", "gated"])
def test_writes_stay_inside_out(kernel, path):
    """Canary-padded output: the out tensor sits inside a NaN-filled buffer
    with 8 KB on each side.  Every row of out must be written (finite) and
    the padding must keep its NaNs (no scatter row outside out)."""
    b, n, hq, hkv, d, w = 2, 333, 8, 2, 128, 64
    if not must_support(kernel, path, hq // hkv, w, d=d):
        pytest.skip("shape outside this kernel's required range")
    inp = Inputs(b, n, hq, hkv, d, seed=11)
    _, perm_d = perms(3, 0, b, n)
    numel, pad = b * n * hq * d, 4096  # pad: bf16 elements, a multiple of 16 bytes
    buf = torch.full((pad + numel + pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[pad:pad + numel].view(b, n, hq, d)
    err = _err()
    if path == "sa":
        sa.sa_forward(inp.q, inp.k, inp.v, perm_d, w, causal=True, out=out, kernel=kernel, err=err)
    elif path == "swa":
        sa.swa_forward(inp.q, inp.k, inp.v, w, out=out, kernel=kernel, err=err)
    else:
        sa.sa_swa_gated_forward(inp.q, inp.k, inp.v, perm_d, inp.ga, inp.gw, w, causal=True,
                                out=out, kernel=kernel, err=err)
    assert sa.check_error(err) == sa.SA_OK
    assert torch.isnan(buf[:pad]).all() and torch.isnan(buf[pad + numel:]).all()
    assert torch.isfinite(out.float()).all()


# ------------------------------------------------------------ bounded waits

TC_KERNELS = [sa.KERNEL_TCGEN05_RING, sa.KERNEL_TCGEN05_CHUNK, sa.KERNEL_TCGEN05_GATHER]


@pytest.mark.parametrize("kernel", TC_KERNELS, ids=["ring", "chunk", "gather"])
@pytest.mark.parametrize("path", ["sa", "gated"])
def test_short_wait_bound_gives_up_cleanly(kernel, path):
    """A 200-cycle bound on every pipeline wait is far shorter than the first
    wait for data from memory, so the call must give up: the kernel returns,
    the error word reports SA_ERR_TIMEOUT, and the next call on the same
    context (default bound) is correct."""
    n, w = 2048, 64
    inp = Inputs(1, n, 32, 8, 128, seed=19, gates=True)
    perm, perm_d = perms(19, 0, 1, n)

    def run(err):
        if path == "sa":
            return sa.sa_forward(inp.q, inp.k, inp.v, perm_d, w, causal=True, kernel=kernel,
                                 err=err)
        return sa.sa_swa_gated_forward(inp.q, inp.k, inp.v, perm_d, inp.ga, inp.gw, w,
                                       causal=True, kernel=kernel, err=err)

    for attempt in range(2):
        err = _err()
        try:
            sa.set_wait_limit(200)
            run(err)
            status = sa.check_error(err)  # synchronises: every CTA has returned
        finally:
            sa.set_wait_limit(0)
        assert status == sa.SA_ERR_TIMEOUT, (attempt, status)
        assert int(err.item()) & sa.ERRBIT_TIMEOUT
        assert not int(err.item()) & sa.ERRBIT_INTERNAL
        err2 = _err()
        y = run(err2)
        assert sa.check_error(err2) == sa.SA_OK
        rows = sample_rows(1, n, 96, seed=attempt)
        want = (oracle.sa_rows(inp.case.q, inp.case.k, inp.case.v, perm, w, True, rows=rows)
                if path == "sa" else
                oracle.gated_rows(inp.case.q, inp.case.k, inp.case.v, perm, inp.case.gate_sa,
                                  inp.case.gate_swa, w, None, True, rows=rows))
        compare(gather_rows(y, rows), want, f"after timeout, {path}")
