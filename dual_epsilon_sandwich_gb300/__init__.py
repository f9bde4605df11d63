"""GB300-native RMSNorm, post-norm-then-add and dual-epsilon sandwich tail.

The computation runs in ``libmrn.so`` (hand-written sm_103a CUDA kernels behind
the C ABI in ``include/mrn.h``); :mod:`dual_epsilon_sandwich_gb300.mrn` is its
Python binding.  :mod:`dual_epsilon_sandwich_gb300.workloads` holds the seeded
synthetic inputs used by the tests and the benchmark.
"""
from .mrn import (  # noqa: F401
    MRN_BF16, MRN_F32, MRN_LAUNCH_PDL, MrnError, add_rmsnorm, mrn_add_rmsnorm,
    mrn_force_geometry, mrn_last_cuda_error, mrn_launch_count, mrn_launch_options,
    mrn_norm_residual_norm, mrn_query_geometry, mrn_rmsnorm, mrn_rmsnorm_q8_1,
    mrn_rmsnorm_then_add, mrn_rmsnorm_then_add_scale, mrn_set_launch_options,
    mrn_status_string, mrn_wait_timeouts, norm_residual_norm, rmsnorm, rmsnorm_q8_1,
    rmsnorm_then_add, rmsnorm_then_add_scale)
