"""Stochastic Attention (SA) forward hot path for GB300 (sm_103a).

Python face of the ``libsa`` C-ABI library (include/libsa.h): SA over a
seeded random permutation of the tokens, sliding-window attention, the
sigmoid-gated SA+SWA merge and the device inverse permutation, each running
in hand-written CUDA kernels.  PyTorch supplies device memory and streams.
"""

from ._libsa import (
    ERRBIT_DUP,
    ERRBIT_INTERNAL,
    ERRBIT_RANGE,
    ERRBIT_TIMEOUT,
    KERNEL_AUTO,
    KERNEL_SIMT,
    KERNEL_TCGEN05,
    KERNEL_TCGEN05_GATHER,
    KERNEL_TCGEN05_RING,
    KERNEL_TCGEN05_CHUNK,
    SA_ERR_BAD_PERM,
    SA_ERR_CUDA,
    SA_ERR_INTERNAL,
    SA_ERR_INVALID_ARG,
    SA_ERR_TIMEOUT,
    SA_ERR_UNSUPPORTED,
    SA_OK,
    SIGNATURES,
    SaError,
    SaParams,
    check_error,
    clear_error,
    get_wait_limit,
    last_kernel,
    last_launch_count,
    load,
    make_perm,
    make_perms,
    gate_projection,
    receptive_field,
    rope_,
    sa_backward,
    sa_forward,
    sa_inverse_perm,
    sa_swa_gated_backward,
    sa_swa_gated_forward,
    set_wait_limit,
    swa_backward,
    swa_forward,
)

__all__ = [
    "ERRBIT_DUP", "ERRBIT_INTERNAL", "ERRBIT_RANGE", "ERRBIT_TIMEOUT", "KERNEL_AUTO", "KERNEL_SIMT", "KERNEL_TCGEN05", "KERNEL_TCGEN05_GATHER", "KERNEL_TCGEN05_RING", "KERNEL_TCGEN05_CHUNK",
    "SA_ERR_BAD_PERM", "SA_ERR_CUDA", "SA_ERR_INTERNAL", "SA_ERR_INVALID_ARG", "SA_ERR_TIMEOUT", "SA_ERR_UNSUPPORTED",
    "SA_OK", "SIGNATURES", "SaError", "SaParams", "check_error", "clear_error", "last_kernel",
    "last_launch_count", "load", "make_perm", "make_perms", "sa_forward", "sa_inverse_perm",
    "sa_swa_gated_forward", "set_wait_limit", "get_wait_limit", "swa_forward",
    "sa_backward", "swa_backward", "sa_swa_gated_backward", "receptive_field",
    "gate_projection", "rope_",
]
