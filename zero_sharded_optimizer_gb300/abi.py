"""Thin ctypes binding over libzero_gb300.so (declared in include/zero_gb300.h).

Same names as the C entry points; this module only marshals arguments
(tensor data pointers, stream and event handles, sizes) and turns status codes
into exceptions. Every step of the computation runs in the library's CUDA
kernels. Importing this module raises if the library has not been built --
there is no fallback path.

PyTorch provides device memory, streams and events here; tensors passed to the
step must be contiguous CUDA tensors of the precision's storage type (float32,
or bfloat16 in mixed precision).
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libzero_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()' "
        "or python zero_sharded_optimizer_gb300/build.py)")

_lib = ctypes.CDLL(LIB_PATH)

ZERO_FP32 = 0
ZERO_BF16_MIXED = 1
ZERO_FP64_EMU = 2

ZERO_OK = 0
ZERO_EINVAL = -1
ZERO_EALIGN = -2
ZERO_ECUDA = -3
ZERO_ETIMEDOUT = -4
ZERO_ENOMEM = -5
ZERO_MAX_RANKS = 64

_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_u64 = ctypes.c_uint64
_dbl = ctypes.c_double
_vp = ctypes.c_void_p
_P = ctypes.POINTER

# Every symbol the header declares, with its signature.
_SIGNATURES = {
    "zero_shard_bounds": (ctypes.c_int, [_i64, _i32, _P(_i64)]),
    "zero_init_states": (ctypes.c_int, [_i64, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _P(_vp)]),
    "zero_init_states_ex": (ctypes.c_int, [_i64, _i32, _i32, _vp, _vp, _vp, _vp, _P(_i64), _vp,
                                           _P(_vp)]),
    "zero_tensor_shard_bounds": (ctypes.c_int, [_P(_i64), _i64, _i32, _P(_i64)]),
    "zero_memory_breakdown_ex": (ctypes.c_int, [_i64, _i32, _i32, _i32, _i32, _P(_i64),
                                                _P(_u64)]),
    "zero_free_states": (ctypes.c_int, [_vp]),
    "zero_states_info": (ctypes.c_int, [_vp, _P(_i64), _P(_i32), _P(_i32)]),
    "zero_state_view": (ctypes.c_int, [_vp, _i32, _P(_i64), _P(_i64), _P(_vp), _P(_vp), _P(_vp)]),
    "zero_step": (ctypes.c_int, [_P(_vp), _P(_vp), _vp, _i64, _dbl, _dbl, _dbl, _dbl, _dbl, _vp]),
    "zero_step_range": (ctypes.c_int, [_P(_vp), _P(_vp), _vp, _i64, _dbl, _dbl, _dbl, _dbl, _dbl,
                                       _i64, _i64, _vp]),
    "zero_bucket_count": (ctypes.c_int, [_i64, _i32, _i64, _P(_i64)]),
    "zero_bucket_range": (ctypes.c_int, [_i64, _i32, _i64, _i64, _P(_i64), _P(_i64)]),
    "zero_step_bucket": (ctypes.c_int, [_P(_vp), _P(_vp), _vp, _i64, _dbl, _dbl, _dbl, _dbl, _dbl,
                                        _i64, _i64, _vp, _vp]),
    "zero_step_bucketed": (ctypes.c_int, [_P(_vp), _P(_vp), _vp, _i64, _dbl, _dbl, _dbl, _dbl,
                                          _dbl, _i64, _P(_vp), _i64, _vp, _vp, _i64]),
    "zero_step_from_host": (ctypes.c_int, [_P(_vp), _P(_vp), _P(_vp), _vp, _i64, _dbl, _dbl, _dbl,
                                           _dbl, _dbl, _vp, _i64, _vp, _vp, _vp]),
    "zero_step_from_host_ex": (ctypes.c_int, [_P(_vp), _P(_vp), _P(_vp), _vp, _vp, _vp, _vp,
                                              _i64, _vp, _vp, _vp]),
    "ddp_allreduce_mean": (ctypes.c_int, [_P(_vp), _i64, _i32, _i32, _vp]),
    "ddp_allreduce_mean_from_host": (ctypes.c_int, [_P(_vp), _P(_vp), _i64, _i32, _i32, _vp,
                                                    _i64, _vp, _vp, _vp]),
    "zero_ddp_host_create": (ctypes.c_int, [_P(_vp)]),
    "zero_debug_fail_host_allocs": (ctypes.c_int, [_i32]),
    "zero_ddp_host_reset": (ctypes.c_int, [_vp]),
    "zero_ddp_host_free": (ctypes.c_int, [_vp]),
    "ddp_allreduce_mean_from_host_h": (ctypes.c_int, [_vp, _P(_vp), _P(_vp), _i64, _i32, _i32,
                                                      _vp, _i64, _vp, _vp, _vp]),
    "zero_memory_bytes": (ctypes.c_int, [_i64, _i32, _i32, _i32, _P(_u64)]),
    "zero_memory_breakdown": (ctypes.c_int, [_i64, _i32, _i32, _i32, _i32, _P(_u64)]),
    "zero_grad_norm_scratch_count": (ctypes.c_int, [_i64, _i32, _P(_i64)]),
    "zero_grad_norm_sq": (ctypes.c_int, [_P(_vp), _i64, _i32, _i32, _vp, _i64, _vp, _vp]),
    "zero_step_ex": (ctypes.c_int, [_P(_vp), _P(_vp), _vp, _vp, _vp]),
    "zero_gather": (ctypes.c_int, [_P(_vp), _vp, _i64, _i64, _vp]),
    "zero_step_sgd": (ctypes.c_int, [_P(_vp), _P(_vp), _vp, _vp, _vp]),
    "zero_grad_norm_sq_noalloc": (ctypes.c_int, [_P(_vp), _i64, _i32, _i32, _vp, _vp]),
    "zero_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "zero_last_error": (ctypes.c_char_p, []),
}

for _name, (_res, _args) in _SIGNATURES.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class ZeroError(RuntimeError):
    """A non-zero status from the library, with its code and message."""

    def __init__(self, code: int, func: str):
        self.code = code
        msg = _lib.zero_last_error().decode(errors="replace")
        super().__init__(f"{func}: {zero_strerror(code)} ({code}): {msg}")


def _check(code: int, func: str) -> None:
    if code != ZERO_OK:
        raise ZeroError(code, func)


def zero_strerror(code: int) -> str:
    return _lib.zero_strerror(code).decode()


# --------------------------------------------------------------- marshalling --

def _storage_dtype(precision: int):
    if precision == ZERO_FP32:
        return torch.float32
    if precision == ZERO_BF16_MIXED:
        return torch.bfloat16
    raise ValueError(f"no tensor storage type for precision {precision}")


def _ptr_array(tensors, n: int, dtype, what: str):
    arr = (_vp * len(tensors))()
    for i, t in enumerate(tensors):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{what}[{i}] must be a CUDA tensor")
        if t.dtype != dtype:
            raise TypeError(f"{what}[{i}] has dtype {t.dtype}, expected {dtype}")
        if not t.is_contiguous() or t.numel() < n:
            raise ValueError(f"{what}[{i}] must be contiguous with at least {n} elements")
        arr[i] = t.data_ptr()
    return arr


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _event_to_record(ev) -> int | None:
    """Handle of an event the library will record. torch creates the CUDA event
    on its first record, so a fresh event is recorded once here to exist."""
    if isinstance(ev, torch.cuda.Event) and not ev.cuda_event:
        ev.record()
    return _event(ev)


def _event(ev) -> int | None:
    if ev is None:
        return None
    if isinstance(ev, torch.cuda.Event):
        h = ev.cuda_event
        if not h:
            raise ValueError("event has never been recorded")
        return h
    return int(ev)


# ----------------------------------------------------------------- host calls --

def zero_shard_bounds(n: int, N: int) -> list[int]:
    out = (_i64 * (max(N, 0) + 1))()
    _check(_lib.zero_shard_bounds(n, N, out), "zero_shard_bounds")
    return list(out)


def zero_memory_bytes(n: int, N: int, stage: int, precision: int) -> int:
    out = _u64()
    _check(_lib.zero_memory_bytes(n, N, stage, precision, ctypes.byref(out)), "zero_memory_bytes")
    return out.value


def zero_memory_breakdown(n: int, N: int, stage: int, precision: int, rank: int) -> tuple:
    out = (_u64 * 3)()
    _check(_lib.zero_memory_breakdown(n, N, stage, precision, rank, out), "zero_memory_breakdown")
    return tuple(out)


def zero_tensor_shard_bounds(numels, N: int) -> list[int]:
    T = len(numels)
    arr = (_i64 * max(T, 1))(*[int(x) for x in numels])
    out = (_i64 * (max(N, 0) + 1))()
    _check(_lib.zero_tensor_shard_bounds(arr, T, N, out), "zero_tensor_shard_bounds")
    return list(out)


def _bounds_array(bounds):
    return None if bounds is None else (_i64 * len(bounds))(*[int(x) for x in bounds])


def zero_memory_breakdown_ex(n: int, N: int, stage: int, precision: int, rank: int,
                             bounds=None) -> tuple:
    out = (_u64 * 3)()
    _check(_lib.zero_memory_breakdown_ex(n, N, stage, precision, rank, _bounds_array(bounds),
                                         out), "zero_memory_breakdown_ex")
    return tuple(out)


def zero_bucket_count(n: int, precision: int, bucket_bytes: int) -> int:
    out = _i64()
    _check(_lib.zero_bucket_count(n, precision, bucket_bytes, ctypes.byref(out)),
           "zero_bucket_count")
    return out.value


def zero_bucket_range(n: int, precision: int, bucket_bytes: int, k: int) -> tuple:
    lo, hi = _i64(), _i64()
    _check(_lib.zero_bucket_range(n, precision, bucket_bytes, k, ctypes.byref(lo),
                                  ctypes.byref(hi)), "zero_bucket_range")
    return lo.value, hi.value


# ------------------------------------------------------------------- state --

class ZeroStates:
    """Owner of a zero_states_t handle; keeps the state tensors alive."""

    def __init__(self, handle: int, n: int, N: int, precision: int, tensors: dict):
        self.handle = handle
        self.n = n
        self.N = N
        self.precision = precision
        self.tensors = tensors

    def view(self, rank: int) -> dict:
        lo, hi = _i64(), _i64()
        m, v, master = _vp(), _vp(), _vp()
        _check(_lib.zero_state_view(self.handle, rank, ctypes.byref(lo), ctypes.byref(hi),
                                    ctypes.byref(m), ctypes.byref(v), ctypes.byref(master)),
               "zero_state_view")
        return {"lo": lo.value, "hi": hi.value, "m": m.value, "v": v.value,
                "master": master.value}

    def info(self) -> tuple:
        n, N, p = _i64(), _i32(), _i32()
        _check(_lib.zero_states_info(self.handle, ctypes.byref(n), ctypes.byref(N),
                                     ctypes.byref(p)), "zero_states_info")
        return n.value, N.value, p.value

    def close(self):
        if self.handle:
            _lib.zero_free_states(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def zero_init_states(n: int, N: int, precision: int, m, v, master=None, master_init=None,
                     stream=None, bounds=None) -> ZeroStates:
    """m, v (and master, master_init in mixed precision): contiguous float32 CUDA
    tensors of n elements. Returns the state handle."""
    def ptr(t, what):
        if t is None:
            return None
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
            raise TypeError(f"{what} must be a float32 CUDA tensor")
        if not t.is_contiguous() or t.numel() < n:
            raise ValueError(f"{what} must be contiguous with at least {n} elements")
        return t.data_ptr()
    h = _vp()
    if bounds is None:
        _check(_lib.zero_init_states(n, N, precision, ptr(m, "m"), ptr(v, "v"),
                                     ptr(master, "master"), ptr(master_init, "master_init"),
                                     _stream(stream), ctypes.byref(h)), "zero_init_states")
    else:
        if len(bounds) != N + 1:
            raise ValueError(f"need {N + 1} shard bounds")
        _check(_lib.zero_init_states_ex(n, N, precision, ptr(m, "m"), ptr(v, "v"),
                                        ptr(master, "master"), ptr(master_init, "master_init"),
                                        _bounds_array(bounds), _stream(stream), ctypes.byref(h)),
               "zero_init_states_ex")
    return ZeroStates(h.value, n, N, precision, {"m": m, "v": v, "master": master})


# -------------------------------------------------------------------- step --

def _step_ptrs(params, grads, st: ZeroStates):
    if len(params) != st.N or len(grads) != st.N:
        raise ValueError(f"need {st.N} params and {st.N} grads")
    dt = _storage_dtype(st.precision)
    return _ptr_array(params, st.n, dt, "params"), _ptr_array(grads, st.n, dt, "grads")


def zero_step(params, grads, st: ZeroStates, t: int, lr: float, beta1: float = 0.9,
              beta2: float = 0.999, eps: float = 1e-8, weight_decay: float = 0.0, stream=None):
    pp, gp = _step_ptrs(params, grads, st)
    _check(_lib.zero_step(pp, gp, st.handle, t, lr, beta1, beta2, eps, weight_decay,
                          _stream(stream)), "zero_step")


def zero_step_range(params, grads, st: ZeroStates, t: int, lr: float, beta1: float, beta2: float,
                    eps: float, weight_decay: float, lo: int, hi: int, stream=None):
    pp, gp = _step_ptrs(params, grads, st)
    _check(_lib.zero_step_range(pp, gp, st.handle, t, lr, beta1, beta2, eps, weight_decay, lo, hi,
                                _stream(stream)), "zero_step_range")


def zero_step_bucket(params, grads, st: ZeroStates, t: int, lr: float, beta1: float, beta2: float,
                     eps: float, weight_decay: float, bucket_bytes: int, k: int, ready=None,
                     side=None):
    pp, gp = _step_ptrs(params, grads, st)
    _check(_lib.zero_step_bucket(pp, gp, st.handle, t, lr, beta1, beta2, eps, weight_decay,
                                 bucket_bytes, k, _event(ready), _stream(side)), "zero_step_bucket")


def zero_step_bucketed(params, grads, st: ZeroStates, t: int, lr: float, beta1: float,
                       beta2: float, eps: float, weight_decay: float, bucket_bytes: int,
                       ready=None, side=None, done=None, timeout_ms: int = -1):
    """Raises ZeroError with code ZERO_ETIMEDOUT when the deadline passes."""
    pp, gp = _step_ptrs(params, grads, st)
    if ready is None:
        arr, count = None, 0
    else:
        arr = (_vp * len(ready))(*[_event(e) for e in ready])
        count = len(ready)
    _check(_lib.zero_step_bucketed(pp, gp, st.handle, t, lr, beta1, beta2, eps, weight_decay,
                                   bucket_bytes, arr, count, _stream(side), _event_to_record(done),
                                   timeout_ms), "zero_step_bucketed")


class StepOpts(ctypes.Structure):
    """zero_step_opts_t."""
    _fields_ = [("t", _i64), ("lr", _dbl), ("beta1", _dbl), ("beta2", _dbl), ("eps", _dbl),
                ("weight_decay", _dbl), ("grad_scale", _dbl), ("max_grad_norm", _dbl),
                ("norm_sq", _vp), ("lo", _i64), ("hi", _i64), ("owner_only", _i32),
                ("norm_scratch", _vp), ("norm_scratch_count", _i64)]


def _f64_device_ptr(t, count: int, what: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float64:
        raise TypeError(f"{what} must be a float64 CUDA tensor")
    if not t.is_contiguous() or t.numel() < count:
        raise ValueError(f"{what} must be contiguous with at least {count} elements")
    return t.data_ptr()


def zero_grad_norm_scratch_count(n: int, precision: int) -> int:
    out = _i64()
    _check(_lib.zero_grad_norm_scratch_count(n, precision, ctypes.byref(out)),
           "zero_grad_norm_scratch_count")
    return out.value


def zero_grad_norm_sq(grads, precision: int, scratch, norm_sq, n: int | None = None,
                      stream=None):
    """Queue ||mean of grads||^2 into the float64 CUDA scalar ``norm_sq``."""
    n = grads[0].numel() if n is None else n
    gp = _ptr_array(grads, n, _storage_dtype(precision), "grads")
    sp = _f64_device_ptr(scratch, 1, "scratch")
    op = _f64_device_ptr(norm_sq, 1, "norm_sq")
    _check(_lib.zero_grad_norm_sq(gp, n, len(grads), precision, sp, scratch.numel(), op,
                                  _stream(stream)), "zero_grad_norm_sq")


ZERO_NOALLOC_MAX_N = 2147450880


def zero_grad_norm_sq_noalloc(grads, precision: int, norm_sq, n: int | None = None,
                              stream=None):
    """zero_grad_norm_sq using the library's own scratch array (no allocation);
    for callers that cannot allocate device memory. n <= ZERO_NOALLOC_MAX_N."""
    n = grads[0].numel() if n is None else n
    gp = _ptr_array(grads, n, _storage_dtype(precision), "grads")
    op = _f64_device_ptr(norm_sq, 1, "norm_sq")
    _check(_lib.zero_grad_norm_sq_noalloc(gp, n, len(grads), precision, op, _stream(stream)),
           "zero_grad_norm_sq_noalloc")


def _scratch_args(norm_scratch):
    if norm_scratch is None:
        return None, 0
    return _f64_device_ptr(norm_scratch, 1, "norm_scratch"), norm_scratch.numel()


def zero_step_ex(params, grads, st: ZeroStates, t: int, lr: float, beta1: float = 0.9,
                 beta2: float = 0.999, eps: float = 1e-8, weight_decay: float = 0.0,
                 grad_scale: float = 1.0, max_grad_norm: float = 0.0, norm_sq=None,
                 lo: int = 0, hi: int = -1, stream=None, owner_only: bool = False,
                 norm_scratch=None):
    """``owner_only`` (ZeRO-3): write the new parameters into the owner's
    replica over its own shard only; ``zero_gather`` restores the replicas.
    Clipping: ``norm_sq`` is the squared norm from zero_grad_norm_sq, or, with
    ``norm_scratch`` (a float64 CUDA tensor of zero_grad_norm_scratch_count
    elements), the scalar this call computes the norm into itself."""
    pp, gp = _step_ptrs(params, grads, st)
    nq = None if norm_sq is None else _f64_device_ptr(norm_sq, 1, "norm_sq")
    sc, count = _scratch_args(norm_scratch)
    o = StepOpts(t, lr, beta1, beta2, eps, weight_decay, grad_scale, max_grad_norm, nq, lo, hi,
                 1 if owner_only else 0, sc, count)
    _check(_lib.zero_step_ex(pp, gp, st.handle, ctypes.byref(o), _stream(stream)), "zero_step_ex")


class SgdOpts(ctypes.Structure):
    """zero_sgd_opts_t."""
    _fields_ = [("t", _i64), ("lr", _dbl), ("momentum", _dbl), ("dampening", _dbl),
                ("weight_decay", _dbl), ("nesterov", _i32), ("grad_scale", _dbl),
                ("max_grad_norm", _dbl), ("norm_sq", _vp), ("lo", _i64), ("hi", _i64),
                ("owner_only", _i32), ("norm_scratch", _vp), ("norm_scratch_count", _i64)]


def zero_step_sgd(params, grads, st: ZeroStates, t: int, lr: float, momentum: float = 0.0,
                  dampening: float = 0.0, weight_decay: float = 0.0, nesterov: bool = False,
                  grad_scale: float = 1.0, max_grad_norm: float = 0.0, norm_sq=None,
                  lo: int = 0, hi: int = -1, stream=None, owner_only: bool = False,
                  norm_scratch=None):
    """The fused ZeRO step with momentum SGD (torch.optim.SGD semantics); the
    state's m is the momentum buffer. Clipping as in zero_step_ex."""
    pp, gp = _step_ptrs(params, grads, st)
    nq = None if norm_sq is None else _f64_device_ptr(norm_sq, 1, "norm_sq")
    sc, count = _scratch_args(norm_scratch)
    o = SgdOpts(t, lr, momentum, dampening, weight_decay, 1 if nesterov else 0, grad_scale,
                max_grad_norm, nq, lo, hi, 1 if owner_only else 0, sc, count)
    _check(_lib.zero_step_sgd(pp, gp, st.handle, ctypes.byref(o), _stream(stream)),
           "zero_step_sgd")


def zero_gather(params, st: ZeroStates, lo: int = 0, hi: int = -1, stream=None):
    """ZeRO-3 gather: copy every shard from its owner's replica into the others."""
    if len(params) != st.N:
        raise ValueError(f"need {st.N} params")
    pp = _ptr_array(params, st.n, _storage_dtype(st.precision), "params")
    _check(_lib.zero_gather(pp, st.handle, lo, hi, _stream(stream)), "zero_gather")


def _host_ptr_array(tensors, n: int, dtype, what: str):
    arr = (_vp * len(tensors))()
    for i, t in enumerate(tensors):
        if not isinstance(t, torch.Tensor) or t.is_cuda:
            raise TypeError(f"{what}[{i}] must be a host tensor")
        if t.dtype != dtype:
            raise TypeError(f"{what}[{i}] has dtype {t.dtype}, expected {dtype}")
        if not t.is_contiguous() or t.numel() < n:
            raise ValueError(f"{what}[{i}] must be contiguous with at least {n} elements")
        arr[i] = t.data_ptr()
    return arr


def zero_step_from_host(params, host_grads, staging, st: ZeroStates, t: int, lr: float,
                        beta1: float, beta2: float, eps: float, weight_decay: float,
                        host_params_out=None, chunk_bytes: int = 25 * 1024 * 1024,
                        compute=None, h2d=None, d2h=None):
    dt = _storage_dtype(st.precision)
    if len(host_grads) != st.N or len(staging) != st.N or len(params) != st.N:
        raise ValueError(f"need {st.N} params, host gradients and staging buffers")
    pp = _ptr_array(params, st.n, dt, "params")
    sp = _ptr_array(staging, st.n, dt, "staging")
    hp = _host_ptr_array(host_grads, st.n, dt, "host_grads")
    out = None
    if host_params_out is not None:
        out = _host_ptr_array([host_params_out], st.n, dt, "host_params_out")[0]
    _check(_lib.zero_step_from_host(pp, hp, sp, st.handle, t, lr, beta1, beta2, eps, weight_decay,
                                    out, chunk_bytes, _stream(compute), _stream(h2d), _stream(d2h)),
           "zero_step_from_host")


def zero_step_from_host_ex(params, host_grads, staging, st: ZeroStates, adamw=None, sgd=None,
                           host_params_out=None, chunk_bytes: int = 25 * 1024 * 1024,
                           compute=None, h2d=None, d2h=None):
    """zero_step_from_host with AdamW options (a StepOpts) or SGD options (an
    SgdOpts): exactly one of ``adamw`` and ``sgd``. With max_grad_norm > 0 the
    options' norm_sq is the device address of a float64 scalar that the call
    fills with the squared norm before the clipped step, and norm_scratch /
    norm_scratch_count the caller's float64 device buffer for its partial
    sums (zero_grad_norm_scratch_count elements)."""
    dt = _storage_dtype(st.precision)
    if len(host_grads) != st.N or len(staging) != st.N or len(params) != st.N:
        raise ValueError(f"need {st.N} params, host gradients and staging buffers")
    pp = _ptr_array(params, st.n, dt, "params")
    sp = _ptr_array(staging, st.n, dt, "staging")
    hp = _host_ptr_array(host_grads, st.n, dt, "host_grads")
    out = None
    if host_params_out is not None:
        out = _host_ptr_array([host_params_out], st.n, dt, "host_params_out")[0]
    _check(_lib.zero_step_from_host_ex(
        pp, hp, sp, st.handle, None if adamw is None else ctypes.byref(adamw),
        None if sgd is None else ctypes.byref(sgd), out, chunk_bytes, _stream(compute),
        _stream(h2d), _stream(d2h)), "zero_step_from_host_ex")


def ddp_allreduce_mean(grads, precision: int, n: int | None = None, stream=None):
    n = grads[0].numel() if n is None else n
    gp = _ptr_array(grads, n, _storage_dtype(precision), "grads")
    _check(_lib.ddp_allreduce_mean(gp, n, len(grads), precision, _stream(stream)),
           "ddp_allreduce_mean")


def ddp_allreduce_mean_from_host(host_grads, staging, precision: int, n: int | None = None,
                                 host_mean_out=None, chunk_bytes: int = 25 * 1024 * 1024,
                                 compute=None, h2d=None, d2h=None):
    """The DDP mean of host gradients, chunk-pipelined into the ``staging``
    CUDA buffers (which end holding the mean); ``host_mean_out`` (a host
    tensor) receives it too when given."""
    n = staging[0].numel() if n is None else n
    if len(host_grads) != len(staging):
        raise ValueError("need one staging buffer per host gradient")
    dt = _storage_dtype(precision)
    hp = _host_ptr_array(host_grads, n, dt, "host_grads")
    sp = _ptr_array(staging, n, dt, "staging")
    out = None
    if host_mean_out is not None:
        out = _host_ptr_array([host_mean_out], n, dt, "host_mean_out")[0]
    _check(_lib.ddp_allreduce_mean_from_host(hp, sp, n, len(staging), precision, out, chunk_bytes,
                                             _stream(compute), _stream(h2d), _stream(d2h)),
           "ddp_allreduce_mean_from_host")


class DdpHost:
    """A zero_ddp_host_t handle: back-to-back DDP means of host gradients on it
    chain chunk by chunk (see ddp_allreduce_mean_from_host_h)."""

    def __init__(self):
        h = _vp()
        _check(_lib.zero_ddp_host_create(ctypes.byref(h)), "zero_ddp_host_create")
        self.handle = h.value

    def reset(self):
        """The next call waits for everything queued on its compute stream."""
        _check(_lib.zero_ddp_host_reset(self.handle), "zero_ddp_host_reset")

    def mean_from_host(self, host_grads, staging, precision: int, n: int | None = None,
                       host_mean_out=None, chunk_bytes: int = 25 * 1024 * 1024, compute=None,
                       h2d=None, d2h=None):
        n = staging[0].numel() if n is None else n
        if len(host_grads) != len(staging):
            raise ValueError("need one staging buffer per host gradient")
        dt = _storage_dtype(precision)
        hp = _host_ptr_array(host_grads, n, dt, "host_grads")
        sp = _ptr_array(staging, n, dt, "staging")
        out = None
        if host_mean_out is not None:
            out = _host_ptr_array([host_mean_out], n, dt, "host_mean_out")[0]
        _check(_lib.ddp_allreduce_mean_from_host_h(
            self.handle, hp, sp, n, len(staging), precision, out, chunk_bytes, _stream(compute),
            _stream(h2d), _stream(d2h)), "ddp_allreduce_mean_from_host_h")

    def close(self):
        if self.handle:
            _lib.zero_ddp_host_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def zero_last_error() -> str:
    """The calling thread's most recent error message from the library."""
    return _lib.zero_last_error().decode(errors="replace")


def zero_debug_fail_host_allocs(count: int) -> None:
    """Failure injection: the calling thread's next ``count`` handle
    allocations fail with ZERO_ENOMEM (count <= 0 clears it)."""
    _check(_lib.zero_debug_fail_host_allocs(count), "zero_debug_fail_host_allocs")


def raw_call(name: str, *args) -> int:
    """Call an entry point with raw ctypes arguments and return its status
    (for callers that manage pointers themselves)."""
    return getattr(_lib, name)(*args)


def declared_symbols() -> list[str]:
    return sorted(_SIGNATURES)
