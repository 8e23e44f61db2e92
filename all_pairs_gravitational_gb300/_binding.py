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
NBODY_PATH_ROWS = 4
NBODY_PRECISION_DEFAULT = 0
NBODY_PRECISION_COMPENSATED = 1
NBODY_QUANTITIES_ACC_POT = 0
NBODY_QUANTITIES_ACC = 1
NBODY_DEFAULT_WORKSPACE_BYTES = 1000000000
NBODY_POOL_KEEP_BYTES = 64 << 20
NBODY_MIN_EPS2 = 1.0e-25      # smallest accepted eps^2 (as the header's)

STATUS_NAMES = {
    0: "NBODY_OK", 1: "NBODY_ERR_INVALID_ARG", 2: "NBODY_ERR_MISALIGNED", 3: "NBODY_ERR_ALIAS",
    4: "NBODY_ERR_CUDA", 5: "NBODY_ERR_TIMEOUT", 6: "NBODY_ERR_DEVICE", 7: "NBODY_ERR_TOO_LARGE",
    8: "NBODY_ERR_WORKSPACE",
}

NBODY_NOALLOC_MAX_N = 4194304

# Every symbol include/nbody.h declares (checked by the tests).
EXPORTS = ["nbody_forces", "nbody_forces_acc", "nbody_euler_step", "nbody_status_string",
           "nbody_last_cuda_error", "nbody_release_cached", "nbody_plan_forces",
           "nbody_plan_forces_ws", "nbody_plan_forces_ts", "nbody_forces_ex", "nbody_forces_ws", "nbody_forces_ts_ws",
           "nbody_simulate_ws", "nbody_forces_noalloc", "nbody_forces_ts", "nbody_simulate"]


class nbody_forces_opts(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("splits", ctypes.c_int32), ("precision", ctypes.c_int32),
                ("quantities", ctypes.c_int32), ("dists", ctypes.c_int32)]


class nbody_plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("i_per_thread", ctypes.c_int32), ("threads", ctypes.c_int32),
                ("tile", ctypes.c_int32), ("num_iblocks", ctypes.c_int32),
                ("splits", ctypes.c_int32), ("tiles_per_split", ctypes.c_int32),
                ("cluster", ctypes.c_int32), ("warps_j", ctypes.c_int32),
                ("dists", ctypes.c_int32), ("groups", ctypes.c_int32),
                ("groups_per_pass", ctypes.c_int32), ("passes", ctypes.c_int32),
                ("grid", ctypes.c_int64), ("scratch_bytes", ctypes.c_int64),
                ("scratch_min_bytes", ctypes.c_int64), ("fill", ctypes.c_double)]

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
_SZ = ctypes.POINTER(ctypes.c_size_t)
_SIGS = {
    "nbody_forces": ([_P, ctypes.c_int64, ctypes.c_float, _P, _P], ctypes.c_int),
    "nbody_forces_acc": ([_P, ctypes.c_int64, ctypes.c_float, _P, _P], ctypes.c_int),
    "nbody_forces_ws": ([_P, ctypes.c_int64, ctypes.c_float, _P, _P, _P, _SZ, _P], ctypes.c_int),
    "nbody_forces_ts_ws": ([_P, ctypes.c_int64, _P, ctypes.c_int64, ctypes.c_float, _P, _P, _P,
                            _SZ, _P], ctypes.c_int),
    "nbody_simulate_ws": ([_P, _P, _P, ctypes.c_int64, ctypes.c_float, ctypes.c_float,
                           ctypes.c_int64, _P, _SZ, _P], ctypes.c_int),
    "nbody_release_cached": ([], ctypes.c_int),
    "nbody_plan_forces_ws": ([ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, ctypes.c_int64,
                              _P], ctypes.c_int),
    "nbody_forces_ex": ([_P, ctypes.c_int64, ctypes.c_float, _P, _P, _P], ctypes.c_int),
    "nbody_euler_step": ([_P, _P, _P, ctypes.c_int64, ctypes.c_float, _P], ctypes.c_int),
    "nbody_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "nbody_last_cuda_error": ([], ctypes.c_int),
    "nbody_plan_forces": ([ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P], ctypes.c_int),
    "nbody_plan_forces_ts": ([ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P,
                              ctypes.c_int64, _P], ctypes.c_int),
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


def _opts(path=NBODY_PATH_AUTO, variant=-1, splits=0, precision=NBODY_PRECISION_DEFAULT,
          quantities=NBODY_QUANTITIES_ACC_POT, dists=0):
    return nbody_forces_opts(int(path), int(variant), int(splits), int(precision),
                             int(quantities), int(dists))


def _workspace(ws, device, standin):
    """(pointer, byte count) of a workspace tensor on `device`.  An empty one
    (or None) is passed as a workspace of 0 bytes at `standin`, a non-null
    pointer the call never touches (a null pointer asks for the size)."""
    import torch
    if ws is None:
        return standin, 0
    if not isinstance(ws, torch.Tensor) or not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if ws.device != device:
        raise ValueError("workspace must be on the bodies' device")
    nbytes = ws.numel() * ws.element_size()
    return (_ptr(ws), nbytes) if nbytes > 0 else (standin, 0)


def _out_for(pos_mass, acc_pot, name="acc_pot"):
    import torch
    n = pos_mass.shape[0]
    if acc_pot is None:
        acc_pot = torch.empty_like(pos_mass)
    _bodies(acc_pot, name, n)
    if acc_pot.device != pos_mass.device:
        raise ValueError(f"pos_mass and {name} must be on the same device")
    return acc_pot


def nbody_forces(pos_mass, eps2, acc_pot=None, stream=None):
    """(ax, ay, az, p) of every body, as a new or the given [n, 4] tensor."""
    import torch
    lib = load_library()
    _bodies(pos_mass, "pos_mass")
    acc_pot = _out_for(pos_mass, acc_pot)
    with torch.cuda.device(pos_mass.device):
        st = lib.nbody_forces(_ptr(pos_mass), pos_mass.shape[0], ctypes.c_float(float(eps2)),
                              _ptr(acc_pot), _stream_handle(pos_mass.device, stream))
    if st != 0:
        raise NbodyError(st, "nbody_forces")
    return acc_pot


def nbody_forces_acc(pos_mass, eps2, acc_pot=None, stream=None):
    """(ax, ay, az, 0) of every body: the acceleration without the potential."""
    import torch
    lib = load_library()
    _bodies(pos_mass, "pos_mass")
    acc_pot = _out_for(pos_mass, acc_pot)
    with torch.cuda.device(pos_mass.device):
        st = lib.nbody_forces_acc(_ptr(pos_mass), pos_mass.shape[0], ctypes.c_float(float(eps2)),
                                  _ptr(acc_pot), _stream_handle(pos_mass.device, stream))
    if st != 0:
        raise NbodyError(st, "nbody_forces_acc")
    return acc_pot


def nbody_forces_ex(pos_mass, eps2, acc_pot=None, path=NBODY_PATH_AUTO, variant=-1, splits=0,
                    precision=NBODY_PRECISION_DEFAULT, quantities=NBODY_QUANTITIES_ACC_POT,
                    dists=0, stream=None):
    import torch
    lib = load_library()
    _bodies(pos_mass, "pos_mass")
    acc_pot = _out_for(pos_mass, acc_pot)
    opts = _opts(path, variant, splits, precision, quantities, dists)
    with torch.cuda.device(pos_mass.device):
        st = lib.nbody_forces_ex(_ptr(pos_mass), pos_mass.shape[0], ctypes.c_float(float(eps2)),
                                 _ptr(acc_pot), ctypes.byref(opts),
                                 _stream_handle(pos_mass.device, stream))
    if st != 0:
        raise NbodyError(st, "nbody_forces_ex")
    return acc_pot


def nbody_forces_ws(pos_mass, eps2, acc_pot=None, workspace=None, path=NBODY_PATH_AUTO,
                    variant=-1, splits=0, precision=NBODY_PRECISION_DEFAULT,
                    quantities=NBODY_QUANTITIES_ACC_POT, dists=0, stream=None):
    """nbody_forces_ex within a caller-owned workspace (any CUDA tensor; its
    bytes are the budget).  The library allocates nothing."""
    import torch
    lib = load_library()
    _bodies(pos_mass, "pos_mass")
    acc_pot = _out_for(pos_mass, acc_pot)
    ptr, nbytes = _workspace(workspace, pos_mass.device, _ptr(acc_pot))
    size = ctypes.c_size_t(nbytes)
    opts = _opts(path, variant, splits, precision, quantities, dists)
    with torch.cuda.device(pos_mass.device):
        st = lib.nbody_forces_ws(_ptr(pos_mass), pos_mass.shape[0], ctypes.c_float(float(eps2)),
                                 _ptr(acc_pot), ctypes.byref(opts), ctypes.c_void_p(ptr),
                                 ctypes.byref(size), _stream_handle(pos_mass.device, stream))
    if st != 0:
        raise NbodyError(st, "nbody_forces_ws")
    return acc_pot


def nbody_forces_workspace_bytes(n, eps2=1e-4, path=NBODY_PATH_AUTO, variant=-1, splits=0,
                                 precision=NBODY_PRECISION_DEFAULT,
                                 quantities=NBODY_QUANTITIES_ACC_POT, dists=0, device=None):
    """Bytes nbody_forces_ws would use by default for n bodies on the current
    (or given) CUDA device: its size query."""
    import torch
    lib = load_library()
    size = ctypes.c_size_t(0)
    opts = _opts(path, variant, splits, precision, quantities, dists)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = lib.nbody_forces_ws(None, int(n), ctypes.c_float(float(eps2)), None,
                                 ctypes.byref(opts), None, ctypes.byref(size), None)
    if st != 0:
        raise NbodyError(st, "nbody_forces_ws (size query)")
    return int(size.value)


def nbody_forces_ts_ws(targets, sources, eps2, out=None, workspace=None, path=NBODY_PATH_AUTO,
                       quantities=NBODY_QUANTITIES_ACC_POT, stream=None, variant=-1, splits=0):
    """nbody_forces_ts within a caller-owned workspace tensor (launch options
    as nbody_forces_ex)."""
    import torch
    lib = load_library()
    _bodies(targets, "targets")
    _bodies(sources, "sources")
    nt, ns = targets.shape[0], sources.shape[0]
    out = _out_for(targets, out, "out")
    if sources.device != targets.device:
        raise ValueError("targets, sources and out must be on the same device")
    ptr, nbytes = _workspace(workspace, targets.device, _ptr(out))
    size = ctypes.c_size_t(nbytes)
    opts = _opts(path=path, variant=variant, splits=splits, quantities=quantities)
    with torch.cuda.device(targets.device):
        st = lib.nbody_forces_ts_ws(_ptr(targets), nt, _ptr(sources), ns,
                                    ctypes.c_float(float(eps2)), _ptr(out), ctypes.byref(opts),
                                    ctypes.c_void_p(ptr), ctypes.byref(size),
                                    _stream_handle(targets.device, stream))
    if st != 0:
        raise NbodyError(st, "nbody_forces_ts_ws")
    return out


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


def nbody_simulate_ws(pos_mass, vel, acc_pot, eps2, dt, steps, workspace, stream=None):
    """nbody_simulate with a caller-owned workspace tensor, which the cached
    graph keeps using until a call with other arguments or
    nbody_release_cached: keep it alive and untouched until then."""
    import torch
    lib = load_library()
    _bodies(pos_mass, "pos_mass")
    n = pos_mass.shape[0]
    _bodies(vel, "vel", n)
    _bodies(acc_pot, "acc_pot", n)
    if not (pos_mass.device == vel.device == acc_pot.device):
        raise ValueError("pos_mass, vel and acc_pot must be on the same device")
    ptr, nbytes = _workspace(workspace, pos_mass.device, _ptr(acc_pot))
    size = ctypes.c_size_t(nbytes)
    with torch.cuda.device(pos_mass.device):
        st = lib.nbody_simulate_ws(_ptr(pos_mass), _ptr(vel), _ptr(acc_pot), n,
                                   ctypes.c_float(float(eps2)), ctypes.c_float(float(dt)),
                                   int(steps), ctypes.c_void_p(ptr), ctypes.byref(size),
                                   _stream_handle(pos_mass.device, stream))
    if st != 0:
        raise NbodyError(st, "nbody_simulate_ws")


def nbody_simulate_workspace_bytes(n, eps2=1e-4, dt=1e-3, device=None):
    """Bytes nbody_simulate_ws would use by default (its size query)."""
    import torch
    lib = load_library()
    size = ctypes.c_size_t(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = lib.nbody_simulate_ws(None, None, None, int(n), ctypes.c_float(float(eps2)),
                                   ctypes.c_float(float(dt)), 1, None, ctypes.byref(size), None)
    if st != 0:
        raise NbodyError(st, "nbody_simulate_ws (size query)")
    return int(size.value)


def nbody_release_cached(device=None):
    """Return the library's device memory on the current (or given) device;
    blocks until that device is idle."""
    import torch
    lib = load_library()
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = lib.nbody_release_cached()
    if st != 0:
        raise NbodyError(st, "nbody_release_cached")


def nbody_plan_forces(n, sm_count, ctas_per_sm=0, path=NBODY_PATH_AUTO, variant=-1, splits=0,
                      precision=NBODY_PRECISION_DEFAULT, quantities=NBODY_QUANTITIES_ACC_POT,
                      dists=0, workspace_bytes=None):
    """Host-only: the decomposition nbody_forces would launch (a dict), within
    the default budget or `workspace_bytes`."""
    lib = load_library()
    plan = nbody_plan()
    opts = _opts(path, variant, splits, precision, quantities, dists)
    if workspace_bytes is None:
        st = lib.nbody_plan_forces(int(n), int(sm_count), int(ctas_per_sm), ctypes.byref(opts),
                                   ctypes.byref(plan))
    else:
        st = lib.nbody_plan_forces_ws(int(n), int(sm_count), int(ctas_per_sm), ctypes.byref(opts),
                                      int(workspace_bytes), ctypes.byref(plan))
    if st != 0:
        raise NbodyError(st, "nbody_plan_forces")
    return plan.as_dict()


def nbody_plan_forces_ts(nt, ns, sm_count, ctas_per_sm=0, path=NBODY_PATH_AUTO, variant=-1,
                         splits=0, quantities=NBODY_QUANTITIES_ACC_POT, workspace_bytes=None):
    """Host-only: the decomposition nbody_forces_ts would launch for nt targets
    and ns sources in separate arrays (a dict)."""
    lib = load_library()
    plan = nbody_plan()
    opts = _opts(path, variant, splits, NBODY_PRECISION_DEFAULT, quantities, 0)
    st = lib.nbody_plan_forces_ts(int(nt), int(ns), int(sm_count), int(ctas_per_sm),
                                  ctypes.byref(opts),
                                  -1 if workspace_bytes is None else int(workspace_bytes),
                                  ctypes.byref(plan))
    if st != 0:
        raise NbodyError(st, "nbody_plan_forces_ts")
    return plan.as_dict()
