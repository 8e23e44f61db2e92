"""GB300 all-pairs softened gravity: a C-ABI CUDA library and its binding.

The compute path lives in ``libnbody.so`` (hand-written sm_103a CUDA, see
``include/nbody.h``); this package only marshals torch tensors into it.
``workloads`` draws the seeded synthetic bodies the tests and the benchmark
use.
"""
from ._binding import (EXPORTS, LIB_PATH, NBODY_DEFAULT_WORKSPACE_BYTES, NBODY_MIN_EPS2,
                       NBODY_NOALLOC_MAX_N,
                       NBODY_PATH_AUTO, NBODY_PATH_CLUSTER, NBODY_PATH_ROWS, NBODY_PATH_SYMMETRIC,
                       NBODY_PATH_TILED, NBODY_POOL_KEEP_BYTES, NBODY_PRECISION_COMPENSATED,
                       NBODY_PRECISION_DEFAULT, NBODY_QUANTITIES_ACC, NBODY_QUANTITIES_ACC_POT,
                       NbodyError, load_library, nbody_euler_step, nbody_forces, nbody_forces_acc,
                       nbody_forces_ex, nbody_forces_noalloc, nbody_forces_ts,
                       nbody_forces_ts_ws, nbody_forces_workspace_bytes, nbody_forces_ws,
                       nbody_last_cuda_error, nbody_plan_forces, nbody_plan_forces_ts,
                       nbody_release_cached,
                       nbody_simulate, nbody_simulate_workspace_bytes, nbody_simulate_ws,
                       nbody_status_string)

__all__ = ["EXPORTS", "LIB_PATH", "NBODY_DEFAULT_WORKSPACE_BYTES", "NBODY_MIN_EPS2", "NBODY_NOALLOC_MAX_N",
           "NBODY_PATH_AUTO", "NBODY_PATH_CLUSTER", "NBODY_PATH_ROWS", "NBODY_PATH_SYMMETRIC", "NBODY_PATH_TILED",
           "NBODY_POOL_KEEP_BYTES", "NBODY_PRECISION_COMPENSATED", "NBODY_PRECISION_DEFAULT",
           "NBODY_QUANTITIES_ACC", "NBODY_QUANTITIES_ACC_POT", "NbodyError", "load_library",
           "nbody_euler_step", "nbody_forces", "nbody_forces_acc", "nbody_forces_ex",
           "nbody_forces_noalloc", "nbody_forces_ts", "nbody_forces_ts_ws",
           "nbody_forces_workspace_bytes", "nbody_forces_ws", "nbody_last_cuda_error", "nbody_plan_forces_ts",
           "nbody_plan_forces", "nbody_release_cached", "nbody_simulate",
           "nbody_simulate_workspace_bytes", "nbody_simulate_ws", "nbody_status_string"]
