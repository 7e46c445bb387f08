"""GB300 (sm_103a) hot path of DP-SGD with randomized clipping (DP-SGD-RC).

The compute lives in libdprc.so (C ABI: include/dprc.h): tensor-core
Hutchinson and Hutch++ per-sample gradient-norm estimation, the exact norm
(direct and ghost-clipping forms), clip factors and Philox Gaussian noise.
This package is its ctypes binding plus the seeded synthetic workloads used by
the tests and the benchmark.
"""

from .binding import (  # noqa: F401
    DPRC_BF16,
    DPRC_EXACT_AUTO,
    DPRC_EXACT_DIRECT,
    DPRC_EXACT_GHOST,
    DPRC_EXACT_GHOST_N128,
    DPRC_EXACT_GHOST_N256,
    DPRC_F32,
    DPRC_OP_EXACT,
    DPRC_OP_HUTCH,
    DPRC_OP_HUTCH_HOST,
    DPRC_OP_HUTCH_LAYERS,
    DPRC_OP_HUTCH_PM1,
    DPRC_OP_HUTCHPP,
    EXPORTED,
    DprcError,
    dprc_abi_version,
    dprc_add_noise,
    dprc_add_noise_at,
    dprc_clip_factors,
    dprc_device_error,
    dprc_exact_norm,
    dprc_exact_norm_plan,
    dprc_norm_hutch,
    dprc_norm_hutch_clip,
    dprc_norm_hutch_clip_host,
    dprc_norm_hutch_launches,
    dprc_norm_hutch_layers,
    dprc_norm_hutch_pm1,
    dprc_norm_hutch_noalloc,
    dprc_norm_hutchpp,
    dprc_norm_hutchpp_launches,
    dprc_philox_words,
    dprc_set_phase_events,
    dprc_test_hutch_fault,
    dprc_workspace_bytes,
    host_stage,
    lib,
    workspace,
)
from .step import RandomizedClippingStep  # noqa: F401,E402
