"""ctypes binding of libsa (include/libsa.h).

Argument marshalling only: shapes and dtypes are checked, pointers, sizes and
the current CUDA stream are handed to the C entry points, and status codes
become exceptions.  Every step of the attention runs in libsa's kernels; if
the library is missing and cannot be built, calls raise -- there is no
fallback implementation.
"""

from __future__ import annotations

import ctypes
from ctypes import (POINTER, byref, c_char_p, c_double, c_float, c_int32, c_int64, c_size_t,
                    c_uint64, c_void_p)
from pathlib import Path

import numpy as np

LIB_PATH = Path(__file__).resolve().with_name("libsa.so")

SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED, SA_ERR_CUDA, SA_ERR_BAD_PERM, SA_ERR_TIMEOUT, \
    SA_ERR_INTERNAL = range(7)
KERNEL_AUTO, KERNEL_SIMT, KERNEL_TCGEN05, KERNEL_TCGEN05_GATHER, KERNEL_TCGEN05_RING = 0, 1, 2, 3, 4
KERNEL_TCGEN05_CHUNK = 5
ERRBIT_RANGE, ERRBIT_DUP, ERRBIT_TIMEOUT, ERRBIT_INTERNAL = 1, 2, 4, 8

# Every function the header declares, with (restype, argtypes).
SIGNATURES = {
    "sa_forward": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "swa_forward": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "sa_swa_gated_forward": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "sa_gated_workspace_size": (c_size_t, [c_void_p]),
    "sa_backward": (c_int32, [c_void_p] * 10 + [c_size_t, c_void_p]),
    "swa_backward": (c_int32, [c_void_p] * 9 + [c_size_t, c_void_p]),
    "sa_backward_workspace_size": (c_size_t, [c_void_p]),
    "sa_backward_noalloc": (c_int32, [c_void_p] * 10),
    "sa_swa_gated_backward": (c_int32, [c_void_p] * 14 + [c_size_t, c_void_p]),
    "sa_swa_gated_backward_workspace_size": (c_size_t, [c_void_p]),
    "sa_inverse_perm": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_void_p]),
    "sa_gate_projection": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "sa_rope": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_int32, c_double, c_void_p]),
    "sa_receptive_field_workspace_size": (c_size_t, [c_int32]),
    "sa_receptive_field": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_int32, c_void_p,
                                     c_int32, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]),
    "sa_make_perm": (c_int32, [c_uint64, c_int32, c_int32, c_int32, POINTER(c_int32)]),
    "sa_shard_span": (c_int32, [c_int32, c_int32, c_int32, c_int32]),
    "sa_shard_plan": (c_int32, [POINTER(c_int32), c_int32, c_int32, c_int32, c_int32,
                                POINTER(c_int32), POINTER(c_int32), c_int32, POINTER(c_int32),
                                POINTER(c_int32), POINTER(c_int32)]),
    "sa_check_error": (c_int32, [c_void_p, c_void_p]),
    "sa_clear_error": (c_int32, [c_void_p, c_void_p]),
    "sa_set_wait_limit": (c_int32, [c_int64]),
    "sa_get_wait_limit": (c_int64, []),
    "sa_status_string": (c_char_p, [c_int32]),
    "sa_last_error_message": (c_char_p, []),
    "sa_last_kernel": (c_int32, []),
    "sa_last_launch_count": (c_int32, []),
}


class SaParams(ctypes.Structure):
    """Mirror of sa_params_t."""
    _fields_ = [
        ("batch", c_int32),
        ("seqlen", c_int32),
        ("num_q_heads", c_int32),
        ("num_kv_heads", c_int32),
        ("head_dim", c_int32),
        ("window", c_int32),
        ("window_swa", c_int32),
        ("causal", c_int32),
        ("softmax_scale", c_float),
        ("kernel", c_int32),
        ("err", c_void_p),
    ]


class SaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


_lib = None


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libsa.so (building it first if it is absent or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        from .build import build
        build()
    if not LIB_PATH.exists():
        raise RuntimeError(f"libsa is not built ({LIB_PATH} missing)")
    lib = ctypes.CDLL(str(LIB_PATH))
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _raise(st: int):
    lib = load()
    msg = lib.sa_last_error_message().decode() or lib.sa_status_string(st).decode()
    raise SaError(st, msg)


def _check(st: int):
    if st != SA_OK:
        _raise(st)


def _stream(t, stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, name, dtype, ndim):
    """Type, dtype, rank and contiguity of one tensor argument."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor")


def _shape(t, name, want):
    if tuple(t.shape) != tuple(want):
        raise ValueError(f"{name} must have shape {tuple(want)}, got {tuple(t.shape)}")


def _on_device(first, name0, named):
    """Every tensor on the first one's CUDA device (the library works on the
    current device, which each call sets to that one)."""
    if not first.is_cuda:
        raise ValueError(f"{name0} must be a CUDA tensor")
    for name, t in named:
        if t is not None and t.device != first.device:
            raise ValueError(f"{name} must be on {first.device}, got {t.device}")


def _check_err(err):
    import torch
    if err is None:
        return
    if not isinstance(err, torch.Tensor) or err.dtype != torch.int32 or err.numel() < 1:
        raise TypeError("err must be an int32 tensor with at least one element")


def _params(q, k, window, window_swa, causal, softmax_scale, kernel, err) -> SaParams:
    b, n, hq, d = q.shape
    return SaParams(b, n, hq, k.shape[2], d, int(window), int(window_swa), int(bool(causal)),
                    float(softmax_scale), int(kernel), c_void_p(err.data_ptr() if err is not None else None))


def _validate(q, k, v, out, perm=None, gates=(), err=None):
    """Every check the C ABI cannot make, since it trusts the sizes it is
    given: dtypes, ranks, contiguity, shapes against q's, one device.  Raises
    before anything is launched."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _need(t, name, torch.bfloat16, 4)
    b, n, hq, d = q.shape
    if k.shape[0] != b or k.shape[1] != n or k.shape[3] != d:
        raise ValueError(f"k must be [B={b}, n={n}, Hkv, d={d}], got {tuple(k.shape)}")
    _shape(v, "v", k.shape)
    _shape(out, "out", q.shape)
    if perm is not None:
        _need(perm, "perm", torch.int32, 2)
        _shape(perm, "perm", (b, n))
    for name, g in gates:
        _need(g, name, torch.float32, 3)
        _shape(g, name, (b, n, hq))
    _check_err(err)
    _on_device(q, "q", [("k", k), ("v", v), ("out", out), ("perm", perm), ("err", err)]
               + list(gates))


def sa_forward(q, k, v, perm, window: int, causal: bool = True, softmax_scale: float = 0.0,
               out=None, kernel: int = KERNEL_AUTO, err=None, stream=None):
    """Stochastic Attention forward; returns out (bf16 [B, n, Hq, d])."""
    import torch
    out = torch.empty_like(q) if out is None else out
    _validate(q, k, v, out, perm=perm, err=err)
    prm = _params(q, k, window, 0, causal, softmax_scale, kernel, err)
    with torch.cuda.device(q.device):
        _check(load().sa_forward(byref(prm), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                 perm.data_ptr(), out.data_ptr(), _stream(q, stream)))
    return out


def swa_forward(q, k, v, window: int, softmax_scale: float = 0.0, out=None,
                kernel: int = KERNEL_AUTO, err=None, stream=None):
    """Sliding-window attention over the original order."""
    import torch
    out = torch.empty_like(q) if out is None else out
    _validate(q, k, v, out, err=err)
    prm = _params(q, k, window, 0, True, softmax_scale, kernel, err)
    with torch.cuda.device(q.device):
        _check(load().swa_forward(byref(prm), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                  out.data_ptr(), _stream(q, stream)))
    return out


def sa_swa_gated_forward(q, k, v, perm, gate_sa, gate_swa, window: int, window_swa: int = 0,
                         causal: bool = True, softmax_scale: float = 0.0, out=None,
                         kernel: int = KERNEL_AUTO, err=None, stream=None):
    """sigmoid(gate_sa) * SA + sigmoid(gate_swa) * SWA."""
    import torch
    out = torch.empty_like(q) if out is None else out
    _validate(q, k, v, out, perm=perm, gates=(("gate_sa", gate_sa), ("gate_swa", gate_swa)),
              err=err)
    prm = _params(q, k, window, window_swa, causal, softmax_scale, kernel, err)
    lib = load()
    with torch.cuda.device(q.device):
        ws = lib.sa_gated_workspace_size(byref(prm))
        work = torch.empty(ws, dtype=torch.uint8, device=q.device) if ws else None
        _check(lib.sa_swa_gated_forward(byref(prm), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                        perm.data_ptr(), gate_sa.data_ptr(), gate_swa.data_ptr(),
                                        out.data_ptr(),
                                        work.data_ptr() if work is not None else None, ws,
                                        _stream(q, stream)))
    return out


def _grads(q, k, dq, dk, dv):
    import torch
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(k) if dv is None else dv
    for name, t, like in (("dq", dq, q), ("dk", dk, k), ("dv", dv, k)):
        _need(t, name, torch.bfloat16, 4)
        _shape(t, name, like.shape)
    return dq, dk, dv


def _workspace(nbytes, device):
    import torch
    # 256-byte aligned: torch's caching allocator returns at least 512-byte
    # aligned blocks
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def sa_backward(q, k, v, perm, dout, window: int, causal: bool = True, softmax_scale: float = 0.0,
                dq=None, dk=None, dv=None, err=None, stream=None):
    """Gradients (dq, dk, dv) of sa_forward for the upstream gradient dout."""
    import torch
    _validate(q, k, v, dout, perm=perm, err=err)
    dq, dk, dv = _grads(q, k, dq, dk, dv)
    _on_device(q, "q", [("dq", dq), ("dk", dk), ("dv", dv)])
    prm = _params(q, k, window, 0, causal, softmax_scale, KERNEL_AUTO, err)
    lib = load()
    with torch.cuda.device(q.device):
        ws = lib.sa_backward_workspace_size(byref(prm))
        work = _workspace(ws, q.device)
        _check(lib.sa_backward(byref(prm), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                               perm.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                               dv.data_ptr(), work.data_ptr(), ws, _stream(q, stream)))
    return dq, dk, dv


def swa_backward(q, k, v, dout, window: int, softmax_scale: float = 0.0, dq=None, dk=None,
                 dv=None, err=None, stream=None):
    """Gradients (dq, dk, dv) of swa_forward for the upstream gradient dout."""
    import torch
    _validate(q, k, v, dout, err=err)
    dq, dk, dv = _grads(q, k, dq, dk, dv)
    _on_device(q, "q", [("dq", dq), ("dk", dk), ("dv", dv)])
    prm = _params(q, k, window, 0, True, softmax_scale, KERNEL_AUTO, err)
    lib = load()
    with torch.cuda.device(q.device):
        ws = lib.sa_backward_workspace_size(byref(prm))
        work = _workspace(ws, q.device)
        _check(lib.swa_backward(byref(prm), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                work.data_ptr(), ws, _stream(q, stream)))
    return dq, dk, dv


def sa_swa_gated_backward(q, k, v, perm, gate_sa, gate_swa, dout, window: int,
                          window_swa: int = 0, causal: bool = True, softmax_scale: float = 0.0,
                          dq=None, dk=None, dv=None, dgate_sa=None, dgate_swa=None, err=None,
                          stream=None):
    """Gradients (dq, dk, dv, dgate_sa, dgate_swa) of sa_swa_gated_forward."""
    import torch
    _validate(q, k, v, dout, perm=perm, gates=(("gate_sa", gate_sa), ("gate_swa", gate_swa)),
              err=err)
    dq, dk, dv = _grads(q, k, dq, dk, dv)
    dgate_sa = torch.empty_like(gate_sa) if dgate_sa is None else dgate_sa
    dgate_swa = torch.empty_like(gate_swa) if dgate_swa is None else dgate_swa
    for name, t in (("dgate_sa", dgate_sa), ("dgate_swa", dgate_swa)):
        _need(t, name, torch.float32, 3)
        _shape(t, name, gate_sa.shape)
    _on_device(q, "q", [("dq", dq), ("dk", dk), ("dv", dv), ("dgate_sa", dgate_sa),
                        ("dgate_swa", dgate_swa)])
    prm = _params(q, k, window, window_swa, causal, softmax_scale, KERNEL_AUTO, err)
    lib = load()
    with torch.cuda.device(q.device):
        ws = lib.sa_swa_gated_backward_workspace_size(byref(prm))
        work = _workspace(ws, q.device)
        _check(lib.sa_swa_gated_backward(
            byref(prm), q.data_ptr(), k.data_ptr(), v.data_ptr(), perm.data_ptr(),
            gate_sa.data_ptr(), gate_swa.data_ptr(), dout.data_ptr(), dq.data_ptr(),
            dk.data_ptr(), dv.data_ptr(), dgate_sa.data_ptr(), dgate_swa.data_ptr(),
            work.data_ptr(), ws, _stream(q, stream)))
    return dq, dk, dv, dgate_sa, dgate_swa


def sa_inverse_perm(perm, inv=None, err=None, stream=None):
    """sigma^{-1} on the device; check the verdict with check_error(err)."""
    import torch
    _need(perm, "perm", torch.int32, 2)
    inv = torch.empty_like(perm) if inv is None else inv
    _need(inv, "inv", torch.int32, 2)
    _shape(inv, "inv", perm.shape)
    _check_err(err)
    _on_device(perm, "perm", [("inv", inv), ("err", err)])
    b, n = perm.shape
    with torch.cuda.device(perm.device):
        _check(load().sa_inverse_perm(perm.data_ptr(), inv.data_ptr(), b, n,
                                      err.data_ptr() if err is not None else None,
                                      _stream(perm, stream)))
    return inv


def gate_projection(x, w_sa, w_swa, b_sa=None, b_swa=None, gate_sa=None, gate_swa=None, err=None,
                    stream=None):
    """Both gate logits of the layer input x (bf16 [B, n, d_model]) with
    weights [Hq, d_model] (bf16) and optional biases [Hq] (fp32): fp32
    [B, n, Hq] each, in one GEMM."""
    import torch
    _need(x, "x", torch.bfloat16, 3)
    _need(w_sa, "w_sa", torch.bfloat16, 2)
    _need(w_swa, "w_swa", torch.bfloat16, 2)
    b, n, dm = x.shape
    hq = w_sa.shape[0]
    _shape(w_sa, "w_sa", (hq, dm))
    _shape(w_swa, "w_swa", (hq, dm))
    for name, t in (("b_sa", b_sa), ("b_swa", b_swa)):
        if t is not None:
            _need(t, name, torch.float32, 1)
            _shape(t, name, (hq,))
    gate_sa = torch.empty((b, n, hq), dtype=torch.float32, device=x.device) if gate_sa is None else gate_sa
    gate_swa = torch.empty((b, n, hq), dtype=torch.float32, device=x.device) if gate_swa is None else gate_swa
    for name, t in (("gate_sa", gate_sa), ("gate_swa", gate_swa)):
        _need(t, name, torch.float32, 3)
        _shape(t, name, (b, n, hq))
    _check_err(err)
    _on_device(x, "x", [("w_sa", w_sa), ("w_swa", w_swa), ("b_sa", b_sa), ("b_swa", b_swa),
                        ("gate_sa", gate_sa), ("gate_swa", gate_swa), ("err", err)])
    ptr = lambda t: t.data_ptr() if t is not None else None
    with torch.cuda.device(x.device):
        _check(load().sa_gate_projection(x.data_ptr(), b * n, dm, hq, w_sa.data_ptr(),
                                         w_swa.data_ptr(), ptr(b_sa), ptr(b_swa),
                                         gate_sa.data_ptr(), gate_swa.data_ptr(), ptr(err),
                                         _stream(x, stream)))
    return gate_sa, gate_swa


def rope_(x, base: float = 10000.0, stream=None):
    """Rotate x (bf16 [B, n, H, d], in place) by each token's original index."""
    import torch
    _need(x, "x", torch.bfloat16, 4)
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    b, n, h, d = x.shape
    with torch.cuda.device(x.device):
        _check(load().sa_rope(x.data_ptr(), b, n, h, d, float(base), _stream(x, stream)))
    return x


def receptive_field(perms, window: int, targets, causal: bool = False, sizes=None, err=None,
                    stream=None):
    """|R_l(t)| for l = 1..L of stacked SA layers with sigma perms[l-1]
    (device int32 [L, n]) for each target token (device int32 [T]): int64
    [L, T] on the device."""
    import torch
    _need(perms, "perms", torch.int32, 2)
    _need(targets, "targets", torch.int32, 1)
    layers, n = perms.shape
    sizes = torch.empty((layers, targets.numel()), dtype=torch.int64, device=perms.device) \
        if sizes is None else sizes
    _need(sizes, "sizes", torch.int64, 2)
    _shape(sizes, "sizes", (layers, targets.numel()))
    _check_err(err)
    _on_device(perms, "perms", [("targets", targets), ("sizes", sizes), ("err", err)])
    lib = load()
    with torch.cuda.device(perms.device):
        ws = lib.sa_receptive_field_workspace_size(n)
        work = torch.empty(ws, dtype=torch.uint8, device=perms.device)
        _check(lib.sa_receptive_field(perms.data_ptr(), layers, n, int(window), int(bool(causal)),
                                      targets.data_ptr(), targets.numel(), sizes.data_ptr(),
                                      work.data_ptr(), ws,
                                      err.data_ptr() if err is not None else None,
                                      _stream(perms, stream)))
    return sizes


def check_error(err=None, stream=None) -> int:
    """Synchronise and map the device error word to a status (0 = fine)."""
    import torch
    _check_err(err)
    dev = err.device if err is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        s = _stream(torch.empty(0, device=dev), stream)
        return int(load().sa_check_error(err.data_ptr() if err is not None else None, s))


def clear_error(err=None, stream=None):
    import torch
    _check_err(err)
    dev = err.device if err is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        _check(load().sa_clear_error(err.data_ptr() if err is not None else None,
                                     _stream(torch.empty(0, device=dev), stream)))


def set_wait_limit(cycles: int) -> None:
    """Bound every pipeline wait of later tcgen05 launches to `cycles` SM
    cycles (<= 0: the default).  A tiny bound makes a call give up on
    purpose: the timeout path's test."""
    _check(load().sa_set_wait_limit(int(cycles)))


def get_wait_limit() -> int:
    return int(load().sa_get_wait_limit())


def make_perm(seed: int, layer: int, batch_index: int, n: int) -> np.ndarray:
    """sigma for (seed, layer, batch_index) from the library's host generator."""
    buf = (c_int32 * n)()
    _check(load().sa_make_perm(c_uint64(seed & ((1 << 64) - 1)), int(layer), int(batch_index),
                               int(n), buf))
    return np.frombuffer(buf, dtype=np.int32).copy()


def make_perms(seed: int, layer: int, batch: int, n: int) -> np.ndarray:
    """[batch, n] int32: one sigma per sequence."""
    return np.stack([make_perm(seed, layer, b, n) for b in range(batch)])


def last_kernel() -> int:
    return int(load().sa_last_kernel())


def last_launch_count() -> int:
    return int(load().sa_last_launch_count())
