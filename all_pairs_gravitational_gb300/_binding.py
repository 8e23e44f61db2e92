"""ctypes binding of libnbody.so: argument marshalling only.

Every function has the name of the C entry point it calls (include/nbody.h).
Tensors must be CUDA float32 [n, 4], contiguous; the call runs on the
tensor's device and on the current torch stream of that device unless a
stream is given.  There is no fallback: without the built library every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libnbody.so")

NBODY_PATH_AUTO = 0
NBODY_PATH_TILED = 1
NBODY_PATH_CLUSTER = 2
NBODY_PATH_SYMMETRIC = 3
NBODY_PRECISION_DEFAULT = 0
NBODY_PRECISION_COMPENSATED = 1

STATUS_NAMES = {
    0: "NBODY_OK", 1: "NBODY_ERR_INVALID_ARG", 2: "NBODY_ERR_MISALIGNED", 3: "NBODY_ERR_ALIAS",
    4: "NBODY_ERR_CUDA", 5: "NBODY_ERR_TIMEOUT", 6: "NBODY_ERR_DEVICE", 7: "NBODY_ERR_TOO_LARGE",
}

NBODY_NOALLOC_MAX_N = 4194304

# Every symbol include/nbody.h declares (checked by the tests).
EXPORTS = ["nbody_forces", "nbody_euler_step", "nbody_status_string", "nbody_last_cuda_error",
           "nbody_plan_forces", "nbody_forces_ex", "nbody_forces_noalloc", "nbody_forces_ts",
           "nbody_simulate"]


class nbody_forces_opts(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("splits", ctypes.c_int32), ("precision", ctypes.c_int32)]


class nbody_plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("i_per_thread", ctypes.c_int32), ("threads", ctypes.c_int32),
                ("tile", ctypes.c_int32), ("num_iblocks", ctypes.c_int32),
                ("splits", ctypes.c_int32), ("tiles_per_split", ctypes.c_int32),
                ("cluster", ctypes.c_int32), ("warps_j", ctypes.c_int32),
                ("grid", ctypes.c_int64), ("scratch_bytes", ctypes.c_int64),
                ("fill", ctypes.c_double)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class NbodyError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = nbody_status_string(status)
        if status == 4:
            msg += f" (cudaError {nbody_last_cuda_error()})"
        super().__init__(f"{what}: {msg}" if what else msg)


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_SIGS = {
    "nbody_forces": ([_P, ctypes.c_int64, ctypes.c_float, _P, _P], ctypes.c_int),
    "nbody_forces_ex": ([_P, ctypes.c_int64, ctypes.c_float, _P, _P, _P], ctypes.c_int),
    "nbody_euler_step": ([_P, _P, _P, ctypes.c_int64, ctypes.c_float, _P], ctypes.c_int),
    "nbody_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "nbody_last_cuda_error": ([], ctypes.c_int),
    "nbody_plan_forces": ([ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P], ctypes.c_int),
    "nbody_forces_noalloc": ([_P, ctypes.c_int64, ctypes.c_float, _P, _P], ctypes.c_int),
    "nbody_forces_ts": ([_P, ctypes.c_int64, _P, ctypes.c_int64, ctypes.c_float, _P, _P],
                        ctypes.c_int),
    "nbody_simulate": ([_P, _P, _P, ctypes.c_int64, ctypes.c_float, ctypes.c_float,
                        ctypes.c_int64, _P], ctypes.c_int),
}


def load_library():
    """Load libnbody.so (built by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() "
                                   "(the CUDA library has no fallback)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGS.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def nbody_status_string(status: int) -> str:
    return load_library().nbody_status_string(int(status)).decode()


def nbody_last_cuda_error() -> int:
    return int(load_library().nbody_last_cuda_error())


def _ptr(t) -> int:
    return int(t.data_ptr())


def _bodies(t, name, n=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.float32 or t.dim() != 2 or t.shape[1] != 4:
        raise ValueError(f"{name} must be float32 of shape [n, 4], got {t.dtype} {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if n is not None and t.shape[0] != n:
        raise ValueError(f"{name} has {t.shape[0]} rows, expected {n}")
    return t


def _stream_handle(device, stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(int(stream.cuda_stream))


def _opts(path=NBODY_PATH_AUTO, variant=-1, splits=0, precision=NBODY_PRECISION_DEFAULT):
    return nbody_forces_opts(int(path), int(variant), int(splits), int(precision))


def nbody_forces(pos_mass, eps2, acc_pot=None, stream=None):
    """(ax, ay, az, p) of every body, as a new or the given [n, 4] tensor."""
    return nbody_forces_ex(pos_mass, eps2, acc_pot, stream=stream)


def nbody_forces_ex(pos_mass, eps2, acc_pot=None, path=NBODY_PATH_AUTO, variant=-1, splits=0,
                    precision=NBODY_PRECISION_DEFAULT, stream=None):
    import torch
    lib = load_library()
    _bodies(pos_mass, "pos_mass")
    n = pos_mass.shape[0]
    if acc_pot is None:
        acc_pot = torch.empty_like(pos_mass)
    _bodies(acc_pot, "acc_pot", n)
    if acc_pot.device != pos_mass.device:
        raise ValueError("pos_mass and acc_pot must be on the same device")
    opts = _opts(path, variant, splits, precision)
    with torch.cuda.device(pos_mass.device):
        st = lib.nbody_forces_ex(_ptr(pos_mass), n, ctypes.c_float(float(eps2)), _ptr(acc_pot),
                                 ctypes.byref(opts), _stream_handle(pos_mass.device, stream))
    if st != 0:
        raise NbodyError(st, "nbody_forces")
    return acc_pot


def nbody_forces_ts(targets, sources, eps2, out=None, stream=None):
    """(ax, ay, az, p) at each target from every source, as a new or the given
    [nt, 4] tensor."""
    import torch
    lib = load_library()
    _bodies(targets, "targets")
    _bodies(sources, "sources")
    nt, ns = targets.shape[0], sources.shape[0]
    if out is None:
        out = torch.empty_like(targets)
    _bodies(out, "out", nt)
    if not (targets.device == sources.device == out.device):
        raise ValueError("targets, sources and out must be on the same device")
    with torch.cuda.device(targets.device):
        st = lib.nbody_forces_ts(_ptr(targets), nt, _ptr(sources), ns, ctypes.c_float(float(eps2)),
                                 _ptr(out), _stream_handle(targets.device, stream))
    if st != 0:
        raise NbodyError(st, "nbody_forces_ts")
    return out


def nbody_forces_noalloc(pos_mass, eps2, acc_pot, stream=None):
    """nbody_forces computed with the library's fixed scratch: the C call
    allocates nothing, so acc_pot must be given (n <= NBODY_NOALLOC_MAX_N)."""
    import torch
    lib = load_library()
    _bodies(pos_mass, "pos_mass")
    n = pos_mass.shape[0]
    _bodies(acc_pot, "acc_pot", n)
    if acc_pot.device != pos_mass.device:
        raise ValueError("pos_mass and acc_pot must be on the same device")
    with torch.cuda.device(pos_mass.device):
        st = lib.nbody_forces_noalloc(_ptr(pos_mass), n, ctypes.c_float(float(eps2)),
                                      _ptr(acc_pot), _stream_handle(pos_mass.device, stream))
    if st != 0:
        raise NbodyError(st, "nbody_forces_noalloc")
    return acc_pot


def nbody_euler_step(pos_mass, vel, acc_pot, dt, stream=None):
    """In-place Euler step: positions with the old velocities, then velocities."""
    import torch
    lib = load_library()
    _bodies(pos_mass, "pos_mass")
    n = pos_mass.shape[0]
    _bodies(vel, "vel", n)
    _bodies(acc_pot, "acc_pot", n)
    if not (pos_mass.device == vel.device == acc_pot.device):
        raise ValueError("pos_mass, vel and acc_pot must be on the same device")
    with torch.cuda.device(pos_mass.device):
        st = lib.nbody_euler_step(_ptr(pos_mass), _ptr(vel), _ptr(acc_pot), n,
                                  ctypes.c_float(float(dt)),
                                  _stream_handle(pos_mass.device, stream))
    if st != 0:
        raise NbodyError(st, "nbody_euler_step")


def nbody_simulate(pos_mass, vel, acc_pot, eps2, dt, steps, stream=None):
    """`steps` device-resident force + Euler steps, in place (CUDA-graph replay)."""
    import torch
    lib = load_library()
    _bodies(pos_mass, "pos_mass")
    n = pos_mass.shape[0]
    _bodies(vel, "vel", n)
    _bodies(acc_pot, "acc_pot", n)
    if not (pos_mass.device == vel.device == acc_pot.device):
        raise ValueError("pos_mass, vel and acc_pot must be on the same device")
    with torch.cuda.device(pos_mass.device):
        st = lib.nbody_simulate(_ptr(pos_mass), _ptr(vel), _ptr(acc_pot), n,
                                ctypes.c_float(float(eps2)), ctypes.c_float(float(dt)), int(steps),
                                _stream_handle(pos_mass.device, stream))
    if st != 0:
        raise NbodyError(st, "nbody_simulate")


def nbody_plan_forces(n, sm_count, ctas_per_sm=0, path=NBODY_PATH_AUTO, variant=-1, splits=0,
                      precision=NBODY_PRECISION_DEFAULT):
    """Host-only: the decomposition nbody_forces would launch (a dict)."""
    lib = load_library()
    plan = nbody_plan()
    opts = _opts(path, variant, splits, precision)
    st = lib.nbody_plan_forces(int(n), int(sm_count), int(ctas_per_sm), ctypes.byref(opts),
                               ctypes.byref(plan))
    if st != 0:
        raise NbodyError(st, "nbody_plan_forces")
    return plan.as_dict()
