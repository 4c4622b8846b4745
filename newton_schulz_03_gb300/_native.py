"""ctypes binding of the C ABI in include/muon.h (argument marshalling only).

Every function here has the name of the C entry point it calls.  Tensors
are PyTorch tensors (device memory and streams come from PyTorch); the
work itself runs in the library's CUDA kernels.  There is no fallback: if
the shared library is missing or the device is not sm_103, calls raise.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple, Union

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmuon_gb300.so")

MUON_OK = 0
STATUS_NAMES = {
    0: "MUON_OK", 1: "MUON_ERR_INVALID_ARG", 2: "MUON_ERR_NOMEM", 3: "MUON_ERR_CUDA",
    4: "MUON_ERR_UNSUPPORTED_ARCH", 5: "MUON_ERR_TIMEOUT", 6: "MUON_ERR_NONFINITE",
    7: "MUON_ERR_NO_DEVICE",
}
KERNEL_NAMES = ("momentum_cast", "norm", "ns_gram", "ns_poly", "ns_update", "apply", "scale",
                "adamw", "transpose")
N_KERNELS = len(KERNEL_NAMES)

# Symbols the header declares (checked by the CPU test-suite).
EXPORTED = (
    "muon_status_string", "muon_last_error_message", "muon_version", "muon_create",
    "muon_destroy", "muon_plan_describe", "muon_step", "muon_step_host", "muon_momentum_cast",
    "muon_newton_schulz_bf16", "muon_apply_update", "muon_last_device_error",
    "muon_set_kernel_timing", "muon_kernel_stats", "muon_reset_kernel_stats",
    "muon_newton_schulz_bf16_static", "muon_selftest_bounded_wait", "muon_step_ex",
    "muon_adamw_step", "muon_partition", "muon_host_alloc", "muon_host_free",
    "muon_shard_momentum_cast", "muon_norm_from_sumsq", "muon_transpose_bf16", "muon_shard_apply",
)
SCALE_NONE, SCALE_SQRT_ASPECT, SCALE_RMS_MATCH = 0, 1, 2


class MuonError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS_NAMES.get(status, f"status {status}")
        super().__init__(f"{self.status_name}: {message}")


class _Group(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int32), ("cols", ctypes.c_int32),
                ("count", ctypes.c_int32), ("update_scale", ctypes.c_float)]


class _Stats(ctypes.Structure):
    _fields_ = [("total_ms", ctypes.c_double * N_KERNELS),
                ("launches", ctypes.c_int64 * N_KERNELS),
                ("total_launches", ctypes.c_int64)]


class _Options(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("wd", ctypes.c_float), ("mu", ctypes.c_float),
                ("ns_steps", ctypes.c_int32), ("nesterov", ctypes.c_int32),
                ("coeffs", ctypes.POINTER(ctypes.c_float)), ("scale_rule", ctypes.c_int32),
                ("rms_target", ctypes.c_float)]


class _AdamwOptions(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("wd", ctypes.c_float), ("step", ctypes.c_int32)]


class _PlanInfo(ctypes.Structure):
    _fields_ = [("n_batches", ctypes.c_int32), ("n_chunks", ctypes.c_int32),
                ("max_chunk_matrices", ctypes.c_int32), ("matrices", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_size_t), ("ns_algorithmic_flops", ctypes.c_double),
                ("launches_per_step", ctypes.c_int64)]


_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (once) the in-tree shared library (or the one MUON_LIB_PATH
    names); raise if it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or os.environ.get("MUON_LIB_PATH") or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing: build it with `python -m newton_schulz_03_gb300.build_lib`")
    lib = ctypes.CDLL(p)
    c_int, c_i32, c_f, c_vp, c_sz = ctypes.c_int, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "muon_status_string": (ctypes.c_char_p, [c_int]),
        "muon_last_error_message": (ctypes.c_char_p, []),
        "muon_version": (ctypes.c_char_p, []),
        "muon_create": (c_int, [P(c_vp), c_i32, c_sz]),
        "muon_destroy": (c_int, [c_vp]),
        "muon_plan_describe": (c_int, [P(_Group), c_i32, c_i32, c_sz, P(_PlanInfo)]),
        "muon_shard_momentum_cast": (c_int, [c_vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                             c_vp, c_vp, c_f, c_vp, c_vp, c_vp]),
        "muon_norm_from_sumsq": (c_int, [c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp,
                                         c_vp]),
        "muon_transpose_bf16": (c_int, [c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp]),
        "muon_shard_apply": (c_int, [c_vp, ctypes.c_int64, c_vp, c_vp, c_f, c_f, c_f, c_vp]),
        "muon_host_alloc": (c_int, [c_sz, P(c_vp)]),
        "muon_host_free": (c_int, [c_vp]),
        "muon_partition": (c_int, [P(_Group), c_i32, c_i32, c_i32, P(ctypes.c_int64), P(c_i32),
                                   P(ctypes.c_double)]),
        "muon_step": (c_int, [c_vp, P(_Group), c_i32, P(c_vp), P(c_vp), P(c_vp), c_f, c_f, c_f,
                              c_i32, c_vp]),
        "muon_step_host": (c_int, [c_vp, P(_Group), c_i32, P(c_vp), P(c_vp), P(c_vp), c_f, c_f,
                                   c_f, c_i32, c_vp]),
        "muon_step_ex": (c_int, [c_vp, P(_Group), c_i32, P(c_vp), P(c_vp), P(c_vp), P(_Options),
                                 c_vp]),
        "muon_momentum_cast": (c_int, [c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_f, c_vp, c_vp,
                                       c_vp]),
        "muon_newton_schulz_bf16": (c_int, [c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_i32,
                                            P(c_f), c_vp]),
        "muon_apply_update": (c_int, [c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_f, c_f, c_f,
                                      c_vp]),
        "muon_newton_schulz_bf16_static": (c_int, [c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_i32,
                                                   P(c_f), c_vp, c_vp]),
        "muon_last_device_error": (c_int, [c_vp, c_vp]),
        "muon_selftest_bounded_wait": (c_int, [c_vp, c_i32, c_vp]),
        "muon_adamw_step": (c_int, [c_vp, c_i32, P(ctypes.c_int64), P(c_vp), P(c_vp), P(c_vp),
                                    P(c_vp), P(_AdamwOptions), c_vp]),
        "muon_set_kernel_timing": (c_int, [c_vp, c_i32]),
        "muon_kernel_stats": (c_int, [c_vp, P(_Stats)]),
        "muon_reset_kernel_stats": (c_int, [c_vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != MUON_OK:
        msg = load_library().muon_last_error_message().decode(errors="replace")
        raise MuonError(status, msg)


def _ptr(x) -> int:
    """Address of a tensor / array / raw integer pointer."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_contiguous():
            raise ValueError("tensors passed to the library must be contiguous")
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)!r}")


def _stream(stream) -> int:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return 0
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


GroupLike = Union[Tuple[int, int, int], Tuple[int, int, int, float]]


def _groups(groups: Sequence[GroupLike]):
    arr = (_Group * max(len(groups), 1))()
    for i, g in enumerate(groups):
        rows, cols, count = int(g[0]), int(g[1]), int(g[2])
        scale = float(g[3]) if len(g) > 3 else 1.0
        arr[i] = _Group(rows, cols, count, scale)
    return arr


def _ptr_array(xs: Sequence) -> ctypes.Array:
    arr = (ctypes.c_void_p * max(len(xs), 1))()
    for i, x in enumerate(xs):
        arr[i] = _ptr(x)
    return arr


# ---------------------------------------------------------------- entry points
def muon_status_string(status: int) -> str:
    return load_library().muon_status_string(status).decode()


def muon_last_error_message() -> str:
    return load_library().muon_last_error_message().decode(errors="replace")


def muon_version() -> str:
    return load_library().muon_version().decode()


def muon_create(device: int = -1, workspace_bytes_max: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(load_library().muon_create(ctypes.byref(h), device, workspace_bytes_max))
    return h.value


def muon_destroy(handle: int) -> None:
    _check(load_library().muon_destroy(handle))


def muon_plan_describe(groups: Sequence[GroupLike], ns_steps: int = 5,
                       workspace_bytes_max: int = 0) -> dict:
    info = _PlanInfo()
    _check(load_library().muon_plan_describe(_groups(groups), len(groups), ns_steps,
                                             workspace_bytes_max, ctypes.byref(info)))
    return {f: getattr(info, f) for f, _ in _PlanInfo._fields_}


def muon_shard_momentum_cast(handle: int, shard_begin: int, shard_end: int, matrix_elems: int,
                             momentum, grad, mu: float, x_shard, sumsq, stream=None) -> None:
    _check(load_library().muon_shard_momentum_cast(handle, shard_begin, shard_end, matrix_elems,
                                                   _ptr(momentum), _ptr(grad), mu, _ptr(x_shard),
                                                   _ptr(sumsq), _stream(stream)))


def muon_norm_from_sumsq(handle: int, m: int, n: int, count: int, parts: int, sumsq, x_wide,
                         inv_norm, stream=None) -> None:
    _check(load_library().muon_norm_from_sumsq(handle, m, n, count, parts, _ptr(sumsq),
                                               _ptr(x_wide), _ptr(inv_norm), _stream(stream)))


def muon_transpose_bf16(handle: int, rows: int, cols: int, count: int, src, dst,
                        stream=None) -> None:
    _check(load_library().muon_transpose_bf16(handle, rows, cols, count, _ptr(src), _ptr(dst),
                                              _stream(stream)))


def muon_shard_apply(handle: int, n_elems: int, weights, o_shard, lr: float, wd: float,
                     scale: float = 1.0, stream=None) -> None:
    _check(load_library().muon_shard_apply(handle, n_elems, _ptr(weights), _ptr(o_shard), lr, wd,
                                           scale, _stream(stream)))


def muon_host_alloc(nbytes: int) -> int:
    """Page-locked host allocation (cudaHostAlloc); returns the address."""
    p = ctypes.c_void_p()
    _check(load_library().muon_host_alloc(nbytes, ctypes.byref(p)))
    return p.value


def muon_host_free(ptr: int) -> None:
    _check(load_library().muon_host_free(ptr))


def host_empty(shape, dtype=None):
    """A CPU torch tensor (FP32 by default) in page-locked memory from
    muon_host_alloc, freed when the tensor and its views are gone."""
    import weakref

    import numpy as np
    import torch
    dtype = dtype or torch.float32
    n = 1
    for d in shape:
        n *= int(d)
    itemsize = torch.empty((), dtype=dtype).element_size()
    nbytes = max(1, n * itemsize)
    ptr = muon_host_alloc(nbytes)
    raw = (ctypes.c_uint8 * nbytes).from_address(ptr)
    weakref.finalize(raw, muon_host_free, ptr)
    arr = np.frombuffer(raw, dtype=np.uint8, count=n * itemsize)
    return torch.from_numpy(arr).view(dtype).view(*shape)


def muon_partition(groups: Sequence[GroupLike], world: int, ns_steps: int = 5):
    """Whole-matrix split of a group list over `world` ranks.  Returns
    (slices, seconds): slices[r] is a list of (group index, first, count)
    of rank r's contiguous slices (count > 0 only); seconds[r] is rank r's
    estimated device time."""
    ng = len(groups)
    first = (ctypes.c_int64 * max(1, ng * world))()
    count = (ctypes.c_int32 * max(1, ng * world))()
    secs = (ctypes.c_double * max(1, world))()
    _check(load_library().muon_partition(_groups(groups), ng, ns_steps, world, first, count,
                                         secs))
    slices = [[(g, int(first[g * world + r]), int(count[g * world + r]))
               for g in range(ng) if count[g * world + r] > 0] for r in range(world)]
    return slices, [float(secs[r]) for r in range(world)]


def muon_step(handle: int, groups: Sequence[GroupLike], momentum: Sequence, grad: Sequence,
              weights: Sequence, lr: float, wd: float, mu: float, ns_steps: int = 5,
              stream=None) -> None:
    _check(load_library().muon_step(handle, _groups(groups), len(groups), _ptr_array(momentum),
                                    _ptr_array(grad), _ptr_array(weights), lr, wd, mu, ns_steps,
                                    _stream(stream)))


def muon_step_ex(handle: int, groups: Sequence[GroupLike], momentum: Sequence, grad: Sequence,
                 weights: Sequence, lr: float, wd: float, mu: float, ns_steps: int = 5,
                 nesterov: bool = False, coeffs: Optional[Sequence] = None,
                 scale_rule: int = SCALE_NONE, rms_target: float = 0.2, stream=None) -> None:
    """muon_step with variants; ``coeffs`` is a list of ns_steps (a, b, c)."""
    c = None
    if coeffs is not None:
        flat = [float(v) for t in coeffs for v in t]
        if len(flat) != 3 * ns_steps:
            raise ValueError("coeffs needs one (a, b, c) per iteration")
        c = (ctypes.c_float * len(flat))(*flat)
    opts = _Options(lr, wd, mu, ns_steps, 1 if nesterov else 0,
                    ctypes.cast(c, ctypes.POINTER(ctypes.c_float)) if c is not None else None,
                    scale_rule, rms_target)
    _check(load_library().muon_step_ex(handle, _groups(groups), len(groups), _ptr_array(momentum),
                                       _ptr_array(grad), _ptr_array(weights), ctypes.byref(opts),
                                       _stream(stream)))


def muon_step_host(handle: int, groups: Sequence[GroupLike], momentum: Sequence, grad: Sequence,
                   weights: Sequence, lr: float, wd: float, mu: float, ns_steps: int = 5,
                   stream=None) -> None:
    _check(load_library().muon_step_host(handle, _groups(groups), len(groups),
                                         _ptr_array(momentum), _ptr_array(grad),
                                         _ptr_array(weights), lr, wd, mu, ns_steps,
                                         _stream(stream)))


def muon_momentum_cast(handle: int, rows: int, cols: int, count: int, momentum, grad, mu: float,
                       x_wide, inv_norm, stream=None) -> None:
    _check(load_library().muon_momentum_cast(handle, rows, cols, count, _ptr(momentum),
                                             _ptr(grad), mu, _ptr(x_wide), _ptr(inv_norm),
                                             _stream(stream)))


def muon_newton_schulz_bf16(handle: int, m: int, n: int, count: int, x, out, inv_norm,
                            ns_steps: int = 5, coeffs: Optional[Sequence[float]] = None,
                            stream=None) -> None:
    c = None
    if coeffs is not None:
        c = (ctypes.c_float * 3)(*[float(v) for v in coeffs])
    _check(load_library().muon_newton_schulz_bf16(handle, m, n, count, _ptr(x), _ptr(out),
                                                  _ptr(inv_norm), ns_steps, c, _stream(stream)))


def muon_newton_schulz_bf16_static(m: int, n: int, count: int, x, out, inv_norm,
                                   ns_steps: int = 5, coeffs: Optional[Sequence[float]] = None,
                                   error_flag=None, stream=None) -> None:
    """Newton-Schulz with no allocation: scratch lives in the library's
    fixed static device array (for callers that cannot allocate)."""
    c = None
    if coeffs is not None:
        c = (ctypes.c_float * 3)(*[float(v) for v in coeffs])
    _check(load_library().muon_newton_schulz_bf16_static(m, n, count, _ptr(x), _ptr(out),
                                                         _ptr(inv_norm), ns_steps, c,
                                                         _ptr(error_flag), _stream(stream)))


def muon_apply_update(handle: int, rows: int, cols: int, count: int, weights, o_wide,
                      lr: float, wd: float, scale: float = 1.0, stream=None) -> None:
    _check(load_library().muon_apply_update(handle, rows, cols, count, _ptr(weights),
                                            _ptr(o_wide), lr, wd, scale, _stream(stream)))


def muon_last_device_error(handle: int, stream=None) -> None:
    _check(load_library().muon_last_device_error(handle, _stream(stream)))


def muon_adamw_step(handle: int, params: Sequence, grads: Sequence, exp_avg: Sequence,
                    exp_avg_sq: Sequence, lr: float, beta1: float, beta2: float, eps: float,
                    wd: float, step: int, stream=None) -> None:
    """AdamW on FP32 tensors (updated in place); ``step`` is 1-based."""
    n = len(params)
    numel = (ctypes.c_int64 * max(n, 1))(*[int(t.numel()) for t in params])
    opts = _AdamwOptions(lr, beta1, beta2, eps, wd, step)
    _check(load_library().muon_adamw_step(handle, n, numel, _ptr_array(params), _ptr_array(grads),
                                          _ptr_array(exp_avg), _ptr_array(exp_avg_sq),
                                          ctypes.byref(opts), _stream(stream)))


def muon_selftest_bounded_wait(handle: int, limit_ms: int = 50, stream=None) -> None:
    """Launch the bounded-wait self-test; muon_last_device_error then
    raises MUON_ERR_TIMEOUT."""
    _check(load_library().muon_selftest_bounded_wait(handle, limit_ms, _stream(stream)))


def muon_set_kernel_timing(handle: int, enable: bool) -> None:
    _check(load_library().muon_set_kernel_timing(handle, 1 if enable else 0))


def muon_kernel_stats(handle: int) -> dict:
    st = _Stats()
    _check(load_library().muon_kernel_stats(handle, ctypes.byref(st)))
    return {"total_ms": {k: st.total_ms[i] for i, k in enumerate(KERNEL_NAMES)},
            "launches": {k: st.launches[i] for i, k in enumerate(KERNEL_NAMES)},
            "total_launches": st.total_launches}


def muon_reset_kernel_stats(handle: int) -> None:
    _check(load_library().muon_reset_kernel_stats(handle))


class Handle:
    """Owning wrapper: ``with Handle() as h: muon_step(h.value, ...)``."""

    def __init__(self, device: int = -1, workspace_bytes_max: int = 0):
        self.value = muon_create(device, workspace_bytes_max)

    def close(self) -> None:
        if self.value:
            muon_destroy(self.value)
            self.value = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
