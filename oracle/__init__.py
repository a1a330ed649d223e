"""fp64 CPU oracle for the selective scan — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product (the CUDA library and its Python binding) never imports it, and this
package imports nothing from the product: the two share only the seeded input
arrays produced by ``seeded_inputs``.

The arithmetic lives in ``selscan_oracle.c`` (plain C, fp64, sequential in t);
this module compiles it with gcc and marshals numpy arrays to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "selscan_oracle.c")
LIB = os.path.join(_HERE, "liboracle_selscan.so")

F32, BF16 = 0, 1
_DT = {"f32": F32, "bf16": BF16}

_lib = None


def compile_oracle(src: str = SRC, out: str = LIB, extra: Sequence[str] = ()) -> str:
    """Compile the oracle C source into a shared library (gcc, -O2)."""
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-pthread", *extra, src, "-lm", "-o", out]
    subprocess.run(cmd, check=True)
    return out


def build() -> str:
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        compile_oracle()
    return LIB


def _bind(lib):
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.oracle_selscan_fwd.argtypes = [i64, i64, i64, i64, i32, p, p, p, p, p, p, p, p, i32, p, p, i32, i32, p, p, i64, p,
                                       p, i32]
    lib.oracle_conv_silu.argtypes = [i64, i64, i64, i64, i32, p, p, p, p]
    lib.oracle_conv_silu.restype = i32
    lib.oracle_selscan_fwd.restype = i32
    lib.oracle_selscan_bwd.argtypes = [i64, i64, i64, i64, i32, p, p, p, p, p, p, p, p, i32, p, p, p, p, p, p, p, p,
                                       p, p, p, p, i32]
    lib.oracle_selscan_bwd.restype = i32
    lib.oracle_selscan_step.argtypes = [i64, i64, i64, i32, p, p, p, p, p, p, p, p, i32, p, p]
    lib.oracle_selscan_step.restype = i32
    lib.oracle_softplus.argtypes = [ctypes.c_double]
    lib.oracle_softplus.restype = ctypes.c_double
    lib.oracle_silu.argtypes = [ctypes.c_double]
    lib.oracle_silu.restype = ctypes.c_double
    lib.oracle_load_bf16.argtypes = [ctypes.c_uint16]
    lib.oracle_load_bf16.restype = ctypes.c_double
    return lib


def load(path: Optional[str] = None):
    """Load the oracle library (building it first if needed).  ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _in(a, dtype):
    if a is None:
        return None
    want = np.uint16 if dtype == "bf16" else np.float32
    return np.ascontiguousarray(a, dtype=want)


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def selscan_fwd(inp: Dict[str, object], delta_softplus: bool = True, rows: Optional[Sequence[int]] = None,
                reverse: bool = False, nthreads: Optional[int] = None, h0_f64: Optional[np.ndarray] = None, lib=None,
                zoh: bool = False, u_f64: Optional[np.ndarray] = None):
    """Run the fp64 forward on an input dict (see ``seeded_inputs.make_inputs``).

    Returns ``(out, h_last)`` as float64 arrays shaped ``[B, D, L]`` and
    ``[B, D, N]`` — or, when ``rows`` (flat b*D + d indices) is given,
    ``[len(rows), L]`` and ``[len(rows), N]``.  ``h0_f64`` (float64
    ``[B, D, N]``) replaces ``inp["h0"]`` as the start state, so that a
    carried fp64 state can be fed back without rounding.
    """
    lib = lib or load()
    Bsz, Dm, L, N = inp["shape"]
    dt = inp["in_dtype"]
    u, delta, z = _in(inp["u"], dt), _in(inp["delta"], dt), _in(inp.get("z"), dt)
    Bm, Cm = _in(inp["B"], dt), _in(inp["C"], dt)
    A, D, bias, h0 = _f32(inp["A"]), _f32(inp.get("D")), _f32(inp.get("delta_bias")), _f32(inp.get("h0"))
    if rows is not None:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.zeros((len(r), L), dtype=np.float64)
        hl = np.zeros((len(r), N), dtype=np.float64)
        rp, nr = _ptr(r), len(r)
    else:
        out = np.zeros((Bsz, Dm, L), dtype=np.float64)
        hl = np.zeros((Bsz, Dm, N), dtype=np.float64)
        rp, nr = None, 0
    nth = nthreads if nthreads is not None else (os.cpu_count() or 1)
    rc = lib.oracle_selscan_fwd(Bsz, Dm, L, N, _DT[dt], _ptr(u), _ptr(delta), _ptr(A), _ptr(Bm), _ptr(Cm),
                                _ptr(D), _ptr(z), _ptr(bias), int(bool(delta_softplus)), _ptr(h0),
                                _ptr(None if h0_f64 is None else np.ascontiguousarray(h0_f64, dtype=np.float64)),
                                int(bool(reverse)), int(bool(zoh)),
                                _ptr(None if u_f64 is None else np.ascontiguousarray(u_f64, dtype=np.float64)),
                                rp, nr, _ptr(out), _ptr(hl), int(nth))
    if rc != 0:
        raise ValueError("oracle_selscan_fwd rejected its arguments")
    return out, hl


def selscan_bwd(inp: Dict[str, object], dout: np.ndarray, dh_last: Optional[np.ndarray] = None,
                delta_softplus: bool = True, nthreads: Optional[int] = None, lib=None) -> Dict[str, np.ndarray]:
    """Gradients of the fp64 forward for a loss with gradient ``dout`` [B, D, L] with respect to out and
    ``dh_last`` [B, D, N] (or None: zero) with respect to h_last.

    Returns float64 arrays keyed "u", "delta", "z" (None without z), "A", "B", "C", "D", "delta_bias"
    (None when the input is absent) and "h0" (the gradient with respect to the start state, returned
    also when h0 is absent, i.e. zero).
    """
    lib = lib or load()
    Bsz, Dm, L, N = inp["shape"]
    dt = inp["in_dtype"]
    u, delta, z = _in(inp["u"], dt), _in(inp["delta"], dt), _in(inp.get("z"), dt)
    Bm, Cm = _in(inp["B"], dt), _in(inp["C"], dt)
    A, D, bias, h0 = _f32(inp["A"]), _f32(inp.get("D")), _f32(inp.get("delta_bias")), _f32(inp.get("h0"))
    go = np.ascontiguousarray(dout, dtype=np.float64)
    gh = None if dh_last is None else np.ascontiguousarray(dh_last, dtype=np.float64)
    res = {"u": np.zeros((Bsz, Dm, L)), "delta": np.zeros((Bsz, Dm, L)),
           "z": None if z is None else np.zeros((Bsz, Dm, L)), "A": np.zeros((Dm, N)),
           "B": np.zeros((Bsz, N, L)), "C": np.zeros((Bsz, N, L)),
           "D": None if D is None else np.zeros(Dm), "delta_bias": None if bias is None else np.zeros(Dm),
           "h0": np.zeros((Bsz, Dm, N))}
    nth = nthreads if nthreads is not None else (os.cpu_count() or 1)
    rc = lib.oracle_selscan_bwd(Bsz, Dm, L, N, _DT[dt], _ptr(u), _ptr(delta), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(D),
                                _ptr(z), _ptr(bias), int(bool(delta_softplus)), _ptr(h0), _ptr(go), _ptr(gh),
                                _ptr(res["u"]), _ptr(res["delta"]), _ptr(res["z"]), _ptr(res["A"]), _ptr(res["B"]),
                                _ptr(res["C"]), _ptr(res["D"]), _ptr(res["delta_bias"]), _ptr(res["h0"]), int(nth))
    if rc != 0:
        raise ValueError("oracle_selscan_bwd rejected its arguments or ran out of memory")
    return res


def conv_silu(x, w, cb, in_dtype: str, lib=None) -> np.ndarray:
    """u = silu(causal depthwise conv1d(x; w [D, K]) + cb) in fp64, for x [B, D, L] of ``in_dtype``."""
    lib = lib or load()
    xin = _in(x, in_dtype)
    Bsz, Dm, L = xin.shape
    w32 = np.ascontiguousarray(w, dtype=np.float32)
    out = np.zeros((Bsz, Dm, L), dtype=np.float64)
    rc = lib.oracle_conv_silu(Bsz, Dm, L, w32.shape[1], _DT[in_dtype], _ptr(xin), _ptr(w32), _ptr(_f32(cb)), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_conv_silu rejected its arguments")
    return out


def selscan_step(inp: Dict[str, object], state: np.ndarray, step: int = 0, delta_softplus: bool = True, lib=None):
    """One decode step on a float64 state [B, D, N] (updated in place); returns out [B, D].

    ``inp`` is a decode input dict (per-step tensors with a leading [steps]
    axis); ``step`` selects the slice.
    """
    lib = lib or load()
    Bsz, Dm, _, N = inp["shape"]
    dt = inp["in_dtype"]

    def sl(name):
        a = inp.get(name)
        return None if a is None else _in(a[step], dt)

    assert state.dtype == np.float64 and state.flags["C_CONTIGUOUS"] and state.shape == (Bsz, Dm, N)
    out = np.zeros((Bsz, Dm), dtype=np.float64)
    rc = lib.oracle_selscan_step(Bsz, Dm, N, _DT[dt], _ptr(sl("u")), _ptr(sl("delta")), _ptr(_f32(inp["A"])),
                                 _ptr(sl("B")), _ptr(sl("C")), _ptr(_f32(inp.get("D"))), _ptr(sl("z")),
                                 _ptr(_f32(inp.get("delta_bias"))), int(bool(delta_softplus)), _ptr(state), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_selscan_step rejected its arguments")
    return out


def softplus(x: float) -> float:
    return load().oracle_softplus(float(x))


def silu(z: float) -> float:
    return load().oracle_silu(float(z))


def load_bf16(bits: int) -> float:
    return load().oracle_load_bf16(int(bits))
