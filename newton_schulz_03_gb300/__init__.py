"""One-GPU Muon optimiser step for GB300 (sm_103a).

The compute runs in hand-written CUDA kernels behind the C ABI of
``include/muon.h``; this package is the ctypes binding (same function
names) plus the synthetic workload definitions used by tests and the
benchmark.
"""

from ._native import (  # noqa: F401
    EXPORTED, KERNEL_NAMES, LIB_PATH, Handle, MuonError, load_library, muon_adamw_step,
    muon_apply_update,
    muon_create, muon_destroy, muon_kernel_stats, muon_last_device_error,
    muon_last_error_message, muon_momentum_cast, muon_newton_schulz_bf16, muon_newton_schulz_bf16_static,
    host_empty, muon_host_alloc, muon_host_free, muon_norm_from_sumsq, muon_partition,
    muon_plan_describe, muon_shard_apply, muon_shard_momentum_cast, muon_transpose_bf16, muon_selftest_bounded_wait,
    muon_reset_kernel_stats, muon_set_kernel_timing, muon_status_string, muon_step,
    muon_step_ex, muon_step_host, muon_version, SCALE_NONE, SCALE_SQRT_ASPECT, SCALE_RMS_MATCH,
)

__all__ = [
    "EXPORTED", "KERNEL_NAMES", "LIB_PATH", "Handle", "MuonError", "load_library",
    "muon_adamw_step",
    "muon_apply_update", "muon_create", "muon_destroy", "muon_kernel_stats",
    "muon_last_device_error", "muon_last_error_message", "muon_momentum_cast",
    "muon_newton_schulz_bf16", "muon_newton_schulz_bf16_static", "muon_partition",
    "muon_host_alloc", "muon_host_free", "host_empty", "muon_shard_momentum_cast",
    "muon_norm_from_sumsq", "muon_transpose_bf16", "muon_shard_apply",
    "muon_plan_describe",
    "muon_selftest_bounded_wait", "muon_reset_kernel_stats",
    "muon_set_kernel_timing", "muon_status_string", "muon_step", "muon_step_ex", "muon_step_host",
    "SCALE_NONE", "SCALE_SQRT_ASPECT", "SCALE_RMS_MATCH",
    "muon_version",
]
