"""Batched speculative-decoding verification on GB300 (sm_103a).

The work happens in libspecdec.so (include/specdec.h); this package is its ctypes
binding, device marshalling, the seeded synthetic workloads and the acceptance metrics.
"""
from ._native import (  # noqa: F401
    SPECDEC_BF16,
    SPECDEC_F32,
    SPECDEC_KMAX,
    SpecdecError,
    launch_config,
    load,
    specdec_verify,
    specdec_wait,
    status_string,
)
from .metrics import acceptance_rates, mean_acceptance_length  # noqa: F401
