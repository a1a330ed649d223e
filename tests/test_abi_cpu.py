"""libselscan loads, exports every symbol that include/*.h declares, and rejects bad arguments on the host.

These run without a GPU: every call below fails a host-side check (shape,
dtype, null pointer or alignment) before the library makes any CUDA call.
"""
import ctypes
import glob
import os
import re

import pytest

import selective_state_space_152_b300 as ss

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b(\w+)\s*\(", text, flags=re.M):
            name = m.group(1)
            if name not in ("if", "defined", "extern") and not name.isupper():
                names.add(name)
    return names


@pytest.fixture(scope="module")
def lib():
    from selective_state_space_152_b300 import build

    build.build()
    return ss.load_library()


def test_header_declares_the_entry_points():
    assert _declared_functions() == set(ss.EXPORTED)


def test_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_abi_version(lib):
    assert ss.selscan_abi_version() == 1


def test_status_strings(lib):
    for code, name in ss.STATUS.items():
        assert ss.selscan_status_string(code).startswith(name)
    assert "unknown" in ss.selscan_status_string(99)


def _shape(B=2, D=3, L=8, N=4, i=0, o=0):
    return ss.SelscanShape(B, D, L, N, i, o)


FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: every call below fails earlier


def _fwd(lib, shape, **kw):
    args = dict(u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, bias=None, sp=1, h0=None, out=FAKE,
                h_last=None)
    args.update(kw)
    return lib.selscan_fwd(ctypes.byref(shape) if shape is not None else None, args["u"], args["delta"], args["A"],
                           args["B"], args["C"], args["D"], args["z"], args["bias"], args["sp"], args["h0"],
                           args["out"], args["h_last"], None)


def _step(lib, shape, **kw):
    args = dict(u=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, bias=None, sp=1, state=FAKE, out=FAKE)
    args.update(kw)
    return lib.selscan_step(ctypes.byref(shape), args["u"], args["delta"], args["A"], args["B"], args["C"],
                            args["D"], args["z"], args["bias"], args["sp"], args["state"], args["out"], None)


def test_null_shape(lib):
    assert _fwd(lib, None) == 1


@pytest.mark.parametrize("bad", [dict(B=-1), dict(D=-2), dict(L=-1), dict(N=0)])
def test_bad_sizes(lib, bad):
    assert _fwd(lib, _shape(**bad)) == 2


def test_overflowing_sizes(lib):
    assert _fwd(lib, _shape(B=2 ** 40, D=2 ** 40, L=2)) == 2


@pytest.mark.parametrize("bad", [dict(N=17), dict(N=64), dict(i=2), dict(o=7)])
def test_unsupported(lib, bad):
    assert _fwd(lib, _shape(**bad)) == 4


@pytest.mark.parametrize("which", ["u", "delta", "A", "B", "C", "out"])
def test_required_pointer_null(lib, which):
    assert _fwd(lib, _shape(), **{which: None}) == 1


@pytest.mark.parametrize("which,dt", [("u", 0), ("A", 0), ("out", 0), ("u", 1), ("B", 1)])
def test_misaligned(lib, which, dt):
    bad = ctypes.c_void_p(0x10001)
    assert _fwd(lib, _shape(i=dt), **{which: bad}) == 3


def test_fwd_ex_rejects_unknown_flags(lib):
    shape = _shape()
    assert lib.selscan_fwd_ex(ctypes.byref(shape), FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, 1, None, FAKE,
                              None, 4, None) == 4  # an unknown flag bit: SELSCAN_ERR_UNSUPPORTED


def test_fwd_conv_rejects_reverse_and_missing_taps(lib):
    shape = _shape()
    # the front is causal: the reverse flag is refused before anything else is checked
    assert lib.selscan_fwd_conv(ctypes.byref(shape), FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, None, None, 1,
                                None, FAKE, None, 1, None) == 4
    assert lib.selscan_fwd_conv(ctypes.byref(shape), FAKE, None, None, FAKE, FAKE, FAKE, FAKE, None, None, None, 1,
                                None, FAKE, None, 0, None) == 1


def test_step_needs_seqlen_one(lib):
    assert _step(lib, _shape(L=2)) == 2
    assert _step(lib, _shape(L=1), state=None) == 1
    assert _step(lib, _shape(L=1, N=20)) == 4


def test_binding_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    u = torch.zeros(1, 2, 4)
    with pytest.raises((ValueError, RuntimeError)):
        ss.selscan_fwd(u, u, torch.zeros(2, 1), torch.zeros(1, 1, 4), torch.zeros(1, 1, 4),
                       out=torch.zeros(1, 2, 4), stream=0)


def test_probe_function_checks_its_arguments(lib):
    # (fn, x, x2, y, n): every case fails before the library touches the GPU
    assert lib.selscan_probe_function(6, FAKE, FAKE, FAKE, 4, None) == 4  # unknown function: UNSUPPORTED
    assert lib.selscan_probe_function(-1, FAKE, FAKE, FAKE, 4, None) == 4
    assert lib.selscan_probe_function(0, FAKE, None, FAKE, -1, None) == 2  # n < 0: SHAPE
    assert lib.selscan_probe_function(0, None, None, FAKE, 4, None) == 1  # no x: NULL
    assert lib.selscan_probe_function(2, FAKE, None, None, 4, None) == 1  # no y: NULL
    assert lib.selscan_probe_function(5, FAKE, None, FAKE, 4, None) == 1  # ZOH without A: NULL
    assert lib.selscan_probe_function(0, None, None, None, 0, None) == 0  # nothing to do: OK, no launch


def test_probe_wait_timeout_checks_its_arguments(lib):
    c = ctypes.c_int(-1)
    assert lib.selscan_probe_wait_timeout(4, None) == 1
    assert lib.selscan_probe_wait_timeout(0, ctypes.byref(c)) == 2
    assert lib.selscan_probe_wait_timeout((1 << 20) + 1, ctypes.byref(c)) == 2
