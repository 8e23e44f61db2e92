"""GB300 all-pairs softened gravity: a C-ABI CUDA library and its binding.

The compute path lives in ``libnbody.so`` (hand-written sm_103a CUDA, see
``include/nbody.h``); this package only marshals torch tensors into it.
``workloads`` draws the seeded synthetic bodies the tests and the benchmark
use.
"""
from ._binding import (EXPORTS, LIB_PATH, NBODY_NOALLOC_MAX_N, NBODY_PATH_AUTO,
                       NBODY_PATH_CLUSTER, NBODY_PATH_SYMMETRIC, NBODY_PATH_TILED,
                       NBODY_PRECISION_COMPENSATED,
                       NBODY_PRECISION_DEFAULT, NbodyError, load_library,
                       nbody_euler_step, nbody_forces, nbody_forces_ex, nbody_forces_noalloc,
                       nbody_forces_ts,
                       nbody_last_cuda_error, nbody_plan_forces, nbody_simulate,
                       nbody_status_string)

__all__ = ["EXPORTS", "LIB_PATH", "NBODY_NOALLOC_MAX_N", "NBODY_PATH_AUTO", "NBODY_PATH_CLUSTER",
           "NBODY_PATH_SYMMETRIC", "NBODY_PATH_TILED", "NBODY_PRECISION_COMPENSATED", "NBODY_PRECISION_DEFAULT", "NbodyError", "load_library", "nbody_euler_step", "nbody_forces",
           "nbody_forces_ex", "nbody_forces_noalloc", "nbody_forces_ts", "nbody_last_cuda_error",
           "nbody_plan_forces", "nbody_simulate", "nbody_status_string"]
