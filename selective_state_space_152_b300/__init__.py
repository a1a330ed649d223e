"""Python binding of libselscan (selective-scan forward, its gradients and the recurrent decode step on B300).

The functions here only marshal arguments: they check tensor types and
layouts, allocate missing outputs with torch, and call the C ABI declared in
``include/selscan.h``.  Every step of the computation runs in the library's
CUDA kernels.  There is no CPU or PyTorch fallback: if ``libselscan.so`` has
not been built, every call raises.

Build the library with ``python -m selective_state_space_152_b300.build``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libselscan.so")

SELSCAN_F32, SELSCAN_BF16 = 0, 1
STATUS = {0: "SELSCAN_OK", 1: "SELSCAN_ERR_NULL", 2: "SELSCAN_ERR_SHAPE", 3: "SELSCAN_ERR_ALIGN",
          4: "SELSCAN_ERR_UNSUPPORTED", 5: "SELSCAN_ERR_CUDA", 6: "SELSCAN_ERR_POINTER", 7: "SELSCAN_ERR_ALIAS",
          8: "SELSCAN_ERR_SCRATCH"}
EXPORTED = ("selscan_fwd", "selscan_step", "selscan_status_string", "selscan_last_cuda_error", "selscan_device_status",
            "selscan_abi_version", "selscan_fwd_noalloc", "selscan_fwd_ex", "selscan_fwd_conv", "selscan_probe_rate",
            "selscan_last_launch_count", "selscan_bwd", "selscan_bwd_workspace_size", "selscan_probe_wait_timeout",
            "selscan_fwd_ckpt", "selscan_bwd_ckpt", "selscan_probe_function")
# Units of selscan_probe_rate (include/selscan_probe.h).
PROBE_UNITS = {"ex2": 0, "lg2": 1, "rcp": 2, "tanh": 3, "ffma": 4, "ffma2": 5}
# Functions of selscan_probe_function (include/selscan_probe.h).
PROBE_FUNCTIONS = {"ex2": 0, "softplus": 1, "silu": 2, "softplus_bwd": 3, "sigmoid": 4, "zoh": 5}
SELSCAN_FLAG_REVERSE, SELSCAN_FLAG_ZOH = 1, 2


class SelscanError(RuntimeError):
    """A libselscan entry point returned a status other than SELSCAN_OK."""

    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class SelscanShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("dim", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int)]


_lib = None


def load_library(path: Optional[str] = None):
    """Load libselscan.so (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libselscan.so not found at {p}; build it with "
                           "`python -m selective_state_space_152_b300.build`")
    lib = ctypes.CDLL(p)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    shp = ctypes.POINTER(SelscanShape)
    lib.selscan_fwd.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp]
    lib.selscan_fwd.restype = i32
    lib.selscan_fwd_ex.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, ctypes.c_uint, vp]
    lib.selscan_fwd_ex.restype = i32
    lib.selscan_fwd_conv.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, ctypes.c_uint, vp]
    lib.selscan_fwd_conv.restype = i32
    lib.selscan_fwd_noalloc.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp]
    lib.selscan_fwd_noalloc.restype = i32
    lib.selscan_step.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp]
    lib.selscan_step.restype = i32
    lib.selscan_status_string.argtypes = [i32]
    lib.selscan_status_string.restype = ctypes.c_char_p
    lib.selscan_last_cuda_error.argtypes = []
    lib.selscan_last_cuda_error.restype = i32
    lib.selscan_device_status.argtypes = [i32]
    lib.selscan_device_status.restype = i32
    lib.selscan_abi_version.argtypes = []
    lib.selscan_abi_version.restype = i32
    lib.selscan_last_launch_count.argtypes = []
    lib.selscan_last_launch_count.restype = i32
    lib.selscan_bwd.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                vp, ctypes.c_size_t, vp]
    lib.selscan_bwd.restype = i32
    lib.selscan_fwd_ckpt.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp]
    lib.selscan_fwd_ckpt.restype = i32
    lib.selscan_bwd_ckpt.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                     vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.selscan_bwd_ckpt.restype = i32
    lib.selscan_bwd_workspace_size.argtypes = [shp]
    lib.selscan_bwd_workspace_size.restype = ctypes.c_size_t
    lib.selscan_probe_wait_timeout.argtypes = [ctypes.c_int64, ctypes.POINTER(ctypes.c_int)]
    lib.selscan_probe_wait_timeout.restype = i32
    lib.selscan_probe_rate.argtypes = [i32, ctypes.POINTER(ctypes.c_double)]
    lib.selscan_probe_rate.restype = i32
    lib.selscan_probe_function.argtypes = [i32, vp, vp, vp, ctypes.c_int64, vp]
    lib.selscan_probe_function.restype = i32
    if path is None:
        _lib = lib
    return lib


def selscan_status_string(status: int) -> str:
    return load_library().selscan_status_string(int(status)).decode()


def selscan_abi_version() -> int:
    return load_library().selscan_abi_version()


def selscan_last_cuda_error() -> int:
    return load_library().selscan_last_cuda_error()


def selscan_device_status(reset: bool = False) -> int:
    """0 if no kernel gave up a bounded wait since the last reset (synchronous read)."""
    return load_library().selscan_device_status(int(bool(reset)))


def selscan_last_launch_count() -> int:
    """Kernels enqueued by the last entry-point call on this host thread (see include/selscan.h)."""
    return load_library().selscan_last_launch_count()


def selscan_probe_rate(unit: str) -> float:
    """Measured results per clock per SM of one arithmetic unit on the current device (synchronous).

    ``unit`` is one of ``PROBE_UNITS``: "ex2", "lg2", "rcp", "tanh" (special-function unit), "ffma",
    "ffma2" (fp32 FMA pipe, scalar and packed; fp32 results counted).
    """
    r = ctypes.c_double(0.0)
    _check(load_library().selscan_probe_rate(PROBE_UNITS[unit], ctypes.byref(r)))
    return r.value


def selscan_probe_function(fn: str, x, x2=None, stream=None):
    """The kernels' own evaluation of one function (``PROBE_FUNCTIONS``) on a contiguous fp32 CUDA tensor
    ``x`` (``x2``: A for "zoh", same shape); returns a new fp32 tensor (see include/selscan_probe.h)."""
    import torch

    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()):
        raise SelscanError("x must be a contiguous float32 CUDA tensor")
    if x2 is not None and not (isinstance(x2, torch.Tensor) and x2.is_cuda and x2.dtype == torch.float32
                               and x2.is_contiguous() and x2.shape == x.shape):
        raise SelscanError("x2 must be a contiguous float32 CUDA tensor shaped like x")
    y = torch.empty_like(x)
    _check(load_library().selscan_probe_function(PROBE_FUNCTIONS[fn], x.data_ptr(),
                                                 None if x2 is None else x2.data_ptr(), y.data_ptr(), x.numel(),
                                                 _stream_handle(stream)))
    return y


def selscan_probe_wait_timeout(polls: int = 4096) -> int:
    """Run the forward kernels' bounded wait on a phase that never completes (see include/selscan_probe.h);
    returns the number of waits that completed (0 when the bound works).  Synchronous."""
    c = ctypes.c_int(-1)
    _check(load_library().selscan_probe_wait_timeout(int(polls), ctypes.byref(c)))
    return c.value


def _check(status: int):
    if status != 0:
        msg = selscan_status_string(status)
        if status == 5:
            msg += f" (cudaError {selscan_last_cuda_error()})"
        raise SelscanError(status, msg)


def _torch():
    import torch  # torch supplies device memory and streams only

    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t == torch.float32:
        return SELSCAN_F32
    if t == torch.bfloat16:
        return SELSCAN_BF16
    raise TypeError(f"unsupported dtype {t}; use torch.float32 or torch.bfloat16")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libselscan takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libselscan takes contiguous tensors")
    return t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _need_f32(name, t):
    torch = _torch()
    if t is not None and t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")


def selscan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus: bool = True, h0=None,
                out=None, h_last=None, stream=None, out_dtype=None, return_h_last: bool = False):
    """Selective-scan forward (see ``include/selscan.h``).

    u, delta, z: [B, D, L]; B, C: [B, N, L] (all float32 or all bfloat16);
    A: [D, N], D / delta_bias: [D], h0 / h_last: [B, D, N] (float32).
    ``out`` ([B, D, L]) is allocated if not given, with ``out_dtype``
    (default float32).  ``h_last`` is allocated when ``return_h_last``.
    Returns ``(out, h_last)`` (``h_last`` may be None).  The work is enqueued
    on ``stream`` (default: torch's current stream).
    """
    torch = _torch()
    lib = load_library()
    if u.dim() != 3 or B.dim() != 3:
        raise ValueError("u must be [B, D, L] and B must be [B, N, L]")
    Bsz, Dm, L = u.shape
    N = B.shape[1]
    for name, t in (("A", A), ("D", D), ("delta_bias", delta_bias), ("h0", h0), ("h_last", h_last)):
        _need_f32(name, t)
    for name, t in (("delta", delta), ("z", z), ("B", B), ("C", C)):
        if t is not None and t.dtype != u.dtype:
            raise TypeError(f"{name} must have u's dtype {u.dtype}")
    if out is None:
        out = torch.empty((Bsz, Dm, L), device=u.device, dtype=out_dtype or torch.float32)
    if h_last is None and return_h_last:
        h_last = torch.empty((Bsz, Dm, N), device=u.device, dtype=torch.float32)
    shape = SelscanShape(Bsz, Dm, L, N, _dtype_code(u.dtype), _dtype_code(out.dtype))
    st = lib.selscan_fwd(ctypes.byref(shape), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                         _ptr(delta_bias), int(bool(delta_softplus)), _ptr(h0), _ptr(out), _ptr(h_last),
                         _stream_handle(stream))
    _check(st)
    return out, h_last


def selscan_fwd_ckpt(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus: bool = True, h0=None,
                     out=None, h_last=None, ckpt=None, stream=None, out_dtype=None, return_h_last: bool = False):
    """``selscan_fwd`` that also keeps the state before every 16-step chunk for ``selscan_bwd(ckpt=...)``.

    Returns ``(out, h_last, ckpt)``, ``ckpt`` [B, D, ceil(L/16), 16] float32 (allocated if not given).
    """
    torch = _torch()
    lib = load_library()
    if u.dim() != 3 or B.dim() != 3:
        raise ValueError("u must be [B, D, L] and B must be [B, N, L]")
    Bsz, Dm, L = u.shape
    N = B.shape[1]
    for name, t in (("A", A), ("D", D), ("delta_bias", delta_bias), ("h0", h0), ("h_last", h_last), ("ckpt", ckpt)):
        _need_f32(name, t)
    for name, t in (("delta", delta), ("z", z), ("B", B), ("C", C)):
        if t is not None and t.dtype != u.dtype:
            raise TypeError(f"{name} must have u's dtype {u.dtype}")
    if out is None:
        out = torch.empty((Bsz, Dm, L), device=u.device, dtype=out_dtype or torch.float32)
    if h_last is None and return_h_last:
        h_last = torch.empty((Bsz, Dm, N), device=u.device, dtype=torch.float32)
    if ckpt is None:
        ckpt = torch.empty((Bsz, Dm, (L + 15) // 16, 16), device=u.device, dtype=torch.float32)
    shape = SelscanShape(Bsz, Dm, L, N, _dtype_code(u.dtype), _dtype_code(out.dtype))
    st = lib.selscan_fwd_ckpt(ctypes.byref(shape), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                              _ptr(delta_bias), int(bool(delta_softplus)), _ptr(h0), _ptr(out), _ptr(h_last),
                              _ptr(ckpt), _stream_handle(stream))
    _check(st)
    return out, h_last, ckpt


def selscan_fwd_ex(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus: bool = True, h0=None,
                   out=None, h_last=None, stream=None, out_dtype=None, return_h_last: bool = False,
                   reverse: bool = False, zoh: bool = False):
    """selscan_fwd with options: ``reverse`` scans from the last step to the first (h_last is the
    state after step 0); ``zoh`` uses the exact zero-order-hold input matrix (exp(ΔA) - 1)/A·B
    instead of Δ·B.  Arguments and return value as for ``selscan_fwd``."""
    torch = _torch()
    lib = load_library()
    if u.dim() != 3 or B.dim() != 3:
        raise ValueError("u must be [B, D, L] and B must be [B, N, L]")
    Bsz, Dm, L = u.shape
    N = B.shape[1]
    for name, t in (("A", A), ("D", D), ("delta_bias", delta_bias), ("h0", h0), ("h_last", h_last)):
        _need_f32(name, t)
    for name, t in (("delta", delta), ("z", z), ("B", B), ("C", C)):
        if t is not None and t.dtype != u.dtype:
            raise TypeError(f"{name} must have u's dtype {u.dtype}")
    if out is None:
        out = torch.empty((Bsz, Dm, L), device=u.device, dtype=out_dtype or torch.float32)
    if h_last is None and return_h_last:
        h_last = torch.empty((Bsz, Dm, N), device=u.device, dtype=torch.float32)
    flags = (SELSCAN_FLAG_REVERSE if reverse else 0) | (SELSCAN_FLAG_ZOH if zoh else 0)
    shape = SelscanShape(Bsz, Dm, L, N, _dtype_code(u.dtype), _dtype_code(out.dtype))
    st = lib.selscan_fwd_ex(ctypes.byref(shape), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                            _ptr(delta_bias), int(bool(delta_softplus)), _ptr(h0), _ptr(out), _ptr(h_last), flags,
                            _stream_handle(stream))
    _check(st)
    return out, h_last


def selscan_fwd_conv(x, conv_w, conv_b, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus: bool = True,
                     h0=None, out=None, h_last=None, stream=None, out_dtype=None, return_h_last: bool = False,
                     zoh: bool = False):
    """The forward with the convolution front: u = silu(conv_b + causal conv1d(x, conv_w [D, 4])),
    computed in the kernel.  Other arguments and the return value as for ``selscan_fwd``."""
    torch = _torch()
    lib = load_library()
    if x.dim() != 3 or B.dim() != 3:
        raise ValueError("x must be [B, D, L] and B must be [B, N, L]")
    Bsz, Dm, L = x.shape
    N = B.shape[1]
    for name, t in (("conv_w", conv_w), ("conv_b", conv_b), ("A", A), ("D", D), ("delta_bias", delta_bias),
                    ("h0", h0), ("h_last", h_last)):
        _need_f32(name, t)
    for name, t in (("delta", delta), ("z", z), ("B", B), ("C", C)):
        if t is not None and t.dtype != x.dtype:
            raise TypeError(f"{name} must have x's dtype {x.dtype}")
    if out is None:
        out = torch.empty((Bsz, Dm, L), device=x.device, dtype=out_dtype or torch.float32)
    if h_last is None and return_h_last:
        h_last = torch.empty((Bsz, Dm, N), device=x.device, dtype=torch.float32)
    shape = SelscanShape(Bsz, Dm, L, N, _dtype_code(x.dtype), _dtype_code(out.dtype))
    st = lib.selscan_fwd_conv(ctypes.byref(shape), _ptr(x), _ptr(conv_w), _ptr(conv_b), _ptr(delta), _ptr(A), _ptr(B),
                              _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(h0),
                              _ptr(out), _ptr(h_last), SELSCAN_FLAG_ZOH if zoh else 0, _stream_handle(stream))
    _check(st)
    return out, h_last


def selscan_fwd_noalloc(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus: bool = True, h0=None,
                        out=None, h_last=None, stream=None):
    """Selective-scan forward that allocates no device memory inside the library.

    For callers that must not allocate while they run.  ``out`` (and
    ``h_last`` if wanted) must be given: this function allocates nothing,
    not even through torch.  The time-block scratch lives in one fixed
    buffer of the library (see ``include/selscan.h``); calls whose work
    overlaps on the GPU race on it.  Raises ``SelscanError`` with status
    ``SELSCAN_ERR_SCRATCH`` if the problem needs more than that buffer holds.
    """
    lib = load_library()
    if out is None:
        raise ValueError("selscan_fwd_noalloc allocates nothing: pass `out`")
    if u.dim() != 3 or B.dim() != 3:
        raise ValueError("u must be [B, D, L] and B must be [B, N, L]")
    Bsz, Dm, L = u.shape
    N = B.shape[1]
    for name, t in (("A", A), ("D", D), ("delta_bias", delta_bias), ("h0", h0), ("h_last", h_last)):
        _need_f32(name, t)
    for name, t in (("delta", delta), ("z", z), ("B", B), ("C", C)):
        if t is not None and t.dtype != u.dtype:
            raise TypeError(f"{name} must have u's dtype {u.dtype}")
    shape = SelscanShape(Bsz, Dm, L, N, _dtype_code(u.dtype), _dtype_code(out.dtype))
    st = lib.selscan_fwd_noalloc(ctypes.byref(shape), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                 _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(h0), _ptr(out),
                                 _ptr(h_last), _stream_handle(stream))
    _check(st)
    return out, h_last


def selscan_step(u, delta, A, B, C, state, D=None, z=None, delta_bias=None, delta_softplus: bool = True,
                 out=None, stream=None, out_dtype=None):
    """One recurrent decode step, updating ``state`` [B, D, N] (float32) in place.

    u, delta, z: [B, D]; B, C: [B, N]; returns ``out`` [B, D].
    """
    torch = _torch()
    lib = load_library()
    if u.dim() != 2 or B.dim() != 2:
        raise ValueError("u must be [B, D] and B must be [B, N]")
    Bsz, Dm = u.shape
    N = B.shape[1]
    for name, t in (("A", A), ("D", D), ("delta_bias", delta_bias), ("state", state)):
        _need_f32(name, t)
    for name, t in (("delta", delta), ("z", z), ("B", B), ("C", C)):
        if t is not None and t.dtype != u.dtype:
            raise TypeError(f"{name} must have u's dtype {u.dtype}")
    if out is None:
        out = torch.empty((Bsz, Dm), device=u.device, dtype=out_dtype or torch.float32)
    shape = SelscanShape(Bsz, Dm, 1, N, _dtype_code(u.dtype), _dtype_code(out.dtype))
    st = lib.selscan_step(ctypes.byref(shape), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                          _ptr(delta_bias), int(bool(delta_softplus)), _ptr(state), _ptr(out),
                          _stream_handle(stream))
    _check(st)
    return out


def selscan_bwd_workspace_size(Bsz: int, Dm: int, L: int, N: int) -> int:
    """Bytes of workspace ``selscan_bwd`` needs for a [Bsz, Dm, L] problem with N states."""
    shape = SelscanShape(Bsz, Dm, L, N, SELSCAN_F32, SELSCAN_F32)
    return int(load_library().selscan_bwd_workspace_size(ctypes.byref(shape)))


def selscan_bwd(u, delta, A, B, C, dout, D=None, z=None, delta_bias=None, delta_softplus: bool = True, h0=None,
                dh_last=None, grads=None, workspace=None, stream=None, want_dh0: bool = True, ckpt=None):
    """Gradients of ``selscan_fwd`` for ``dout`` = ∂loss/∂out (and ``dh_last`` = ∂loss/∂h_last, or None).

    Returns a dict with "u", "delta" and "z" ([B, D, L], u's dtype; "z" None without z), "A" [D, N],
    "B", "C" ([B, N, L], float32), "D", "delta_bias" ([D], float32) and "h0" ([B, D, N], float32; None
    unless ``want_dh0``).  ``grads`` may hold preallocated outputs under the same keys.  ``workspace`` is
    a CUDA tensor of at least ``selscan_bwd_workspace_size`` bytes (or None: the library takes it from
    the stream's memory pool).  ``ckpt`` (from ``selscan_fwd_ckpt`` on the same inputs) makes it rerun
    chunks from the forward's checkpoints (``selscan_bwd_ckpt``) instead of recomputing them.
    """
    torch = _torch()
    lib = load_library()
    if u.dim() != 3 or B.dim() != 3:
        raise ValueError("u must be [B, D, L] and B must be [B, N, L]")
    Bsz, Dm, L = u.shape
    N = B.shape[1]
    for name, t in (("A", A), ("D", D), ("delta_bias", delta_bias), ("h0", h0), ("dh_last", dh_last)):
        _need_f32(name, t)
    for name, t in (("delta", delta), ("z", z), ("B", B), ("C", C)):
        if t is not None and t.dtype != u.dtype:
            raise TypeError(f"{name} must have u's dtype {u.dtype}")
    g = dict(grads or {})
    dev = u.device

    def out(key, shp, dt):
        if g.get(key) is None:
            g[key] = torch.empty(shp, device=dev, dtype=dt)

    out("u", (Bsz, Dm, L), u.dtype)
    out("delta", (Bsz, Dm, L), u.dtype)
    if z is not None:
        out("z", (Bsz, Dm, L), u.dtype)
    else:
        g["z"] = None
    out("A", (Dm, N), torch.float32)
    out("B", (Bsz, N, L), torch.float32)
    out("C", (Bsz, N, L), torch.float32)
    out("D", (Dm,), torch.float32)
    out("delta_bias", (Dm,), torch.float32)
    if want_dh0:
        out("h0", (Bsz, Dm, N), torch.float32)
    else:
        g["h0"] = None
    for key in ("A", "B", "C", "D", "delta_bias", "h0"):
        _need_f32("grad of " + key, g.get(key))
    shape = SelscanShape(Bsz, Dm, L, N, _dtype_code(u.dtype), _dtype_code(dout.dtype))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    head = (ctypes.byref(shape), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            int(bool(delta_softplus)), _ptr(h0), _ptr(dout), _ptr(dh_last))
    tail = (_ptr(g["u"]), _ptr(g["delta"]), _ptr(g["z"]), _ptr(g["A"]), _ptr(g["B"]), _ptr(g["C"]), _ptr(g["D"]),
            _ptr(g["delta_bias"]), _ptr(g["h0"]), _ptr(workspace), ws_bytes, _stream_handle(stream))
    if ckpt is None:
        st = lib.selscan_bwd(*head, *tail)
    else:
        _need_f32("ckpt", ckpt)
        st = lib.selscan_bwd_ckpt(*head, _ptr(ckpt), *tail)
    _check(st)
    return g


__all__ = ["selscan_fwd", "selscan_fwd_ckpt", "selscan_bwd", "selscan_bwd_workspace_size", "selscan_probe_wait_timeout", "selscan_fwd_ex", "selscan_fwd_conv", "selscan_fwd_noalloc", "selscan_step",
           "selscan_status_string", "selscan_abi_version", "selscan_last_cuda_error", "selscan_device_status",
           "selscan_probe_rate", "selscan_last_launch_count", "SelscanError", "SelscanShape", "load_library", "LIB_PATH", "EXPORTED",
           "PROBE_UNITS", "PROBE_FUNCTIONS", "selscan_probe_function"]
