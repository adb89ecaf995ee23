"""GB300 (sm_103a) dynamic short convolution.

    y[t,d] = x[t,d] + sum_{k<W} w^(t)[g(d), k] * x[t-k, d]

(notes on "Dynamic Short Convolutions Improve Transformers", eq. 2 with the
residual of eq. 3), forward and backward, with materialised, head-wise and
low-rank fused filters (the low-rank generator's first projection on chip
too), over packed documents; the static short convolution
(eq. 1) on the same machinery; a single-token decode step against a
per-sequence history ring; and the projection that produces the convolution's
input and filter with the convolution applied in its epilogue.  The compute lives in
``libdsc.so`` (hand-written CUDA kernels behind a C ABI, ``include/dsc.h``);
this package is a thin ctypes binding with the same function names, plus the
build step and the seeded input generators used by tests and benchmarks.

Importing the package does not load the library; the first call does, and
raises if it has not been built.
"""
from ._abi import (  # noqa: F401
    DSC_BF16,
    DSC_ERR_CUDA,
    DSC_ERR_INVALID_ARG,
    DSC_ERR_TIMEOUT,
    DSC_ERR_UNSUPPORTED,
    DSC_F32,
    DSC_OK,
    DscError,
    dsc_bwd,
    dsc_decode_step,
    dsc_fwd,
    dsc_launch_count,
    dsc_lowrank_bwd,
    dsc_lowrank_bwd_noalloc,
    dsc_lowrank_bwd_workspace_bytes,
    dsc_lowrank_fwd,
    dsc_lowrank_zproj_fwd,
    dsc_proj_fwd,
    dsc_static_bwd,
    dsc_static_fwd,
    dsc_sync_status,
    dsc_test_wait_timeout,
    dsc_validate_cu_seqlens,
    dsc_version,
    lib,
    status_string,
)
