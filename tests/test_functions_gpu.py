"""The kernels' own arithmetic of the functions they approximate, held against float64 over each input range.

Every Ā of the scan is 2^(Δ·A·log2 e) on the special-function unit ("Mamba架构与SSM模型：高效序列建模技术
解析" §2.1), Δ is softplus(δ + Δ_bias) (§2.2 of the same page), the gate is x·σ(x) ("Mamba状态空间模型深度
解析：挑战Transformer的下一代序列建模范式" §3.1), the backward needs σ as the derivative of softplus, and the
exact zero-order-hold option needs (exp(ΔA) − 1)/A.  selscan_probe_function evaluates the kernels' own code
for each of them; the references are numpy float64 evaluations at the same fp32 inputs.

Bounds (relative to the reference, and growing with |x| where the argument x·log2 e is rounded to fp32 before
the exponential: an argument of magnitude m carries an absolute error up to m·2^-24, which becomes a relative
error of m·2^-24·ln 2 in the result):
  ex2       2^-21 relative                        (the unit's approximation; its argument is exact here)
  softplus  2^-21 + |x|·2^-23 relative, plus 2^-22 absolute: for e = exp(-|x|) ≥ 1/16 it takes
            log1p(e) as lg2(1 + e)·ln 2 on the unit, whose error there is about 2^-22 in absolute terms
            (measured: 1.9e-7 at the branch point, where softplus is 0.060)
  silu      2^-20 + |x|·2^-23 relative
  sigmoid   2^-20 + |x|·2^-23 relative
  zoh       2^-18 relative: below |ΔA| = 1/16 the series errs by less than (ΔA)^4/120; above it Ā − 1 loses
            up to 2^-22/(1/16) = 2^-18 of its value to cancellation
"""
from __future__ import annotations

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _eval(fn, x, x2=None):
    import torch

    import selective_state_space_152_b300 as ss

    xt = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    x2t = None if x2 is None else torch.from_numpy(np.ascontiguousarray(x2, dtype=np.float32)).cuda()
    y = ss.selscan_probe_function(fn, xt, x2t)
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


def _grid(lo, hi, n=1 << 20):
    """n fp32 values spread over [lo, hi], plus every fp32 value in a small window around 0."""
    x = np.linspace(lo, hi, n, dtype=np.float64).astype(np.float32)
    near0 = np.linspace(-1e-3, 1e-3, 4097, dtype=np.float64).astype(np.float32)
    return np.unique(np.concatenate([x, near0]))


def _worst(got, ref, bound):
    frac = np.abs(got - ref) / bound
    i = int(np.argmax(frac))
    return float(frac[i]), i


def test_ex2():
    x = _grid(-120.0, 60.0)
    x64 = x.astype(np.float64)
    ref = np.exp2(x64)
    got = _eval("ex2", x)
    w, i = _worst(got, ref, 2.0 ** -21 * ref)
    assert w <= 1.0, f"ex2 at x={x[i]!r}: got {got[i]!r} ref {ref[i]!r} ({w:.2f} of the bound)"


def _softplus64(x):
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


@pytest.mark.parametrize("fn", ["softplus", "softplus_bwd"])
def test_softplus(fn):
    # Past |x| = 88 the series term underflows in fp32 (exactly: it is below 2^-126); the grid stops there.
    x = np.concatenate([_grid(-80.0, 80.0), np.float32([-np.log(16.0), np.log(16.0)])])  # the branch points
    x64 = x.astype(np.float64)
    ref = _softplus64(x64)
    got = _eval(fn, x)
    bound = (2.0 ** -21 + np.abs(x64) * 2.0 ** -23) * ref + 2.0 ** -22
    w, i = _worst(got, ref, bound)
    assert w <= 1.0, f"{fn} at x={x[i]!r}: got {got[i]!r} ref {ref[i]!r} ({w:.2f} of the bound)"


def test_silu():
    x = _grid(-80.0, 80.0)
    x64 = x.astype(np.float64)
    ref = x64 / (1.0 + np.exp(-x64))
    got = _eval("silu", x)
    bound = (2.0 ** -20 + np.abs(x64) * 2.0 ** -23) * np.abs(ref) + 1e-300
    w, i = _worst(got, ref, bound)
    assert w <= 1.0, f"silu at x={x[i]!r}: got {got[i]!r} ref {ref[i]!r} ({w:.2f} of the bound)"


def test_sigmoid():
    x = _grid(-80.0, 80.0)
    x64 = x.astype(np.float64)
    ref = 1.0 / (1.0 + np.exp(-x64))
    got = _eval("sigmoid", x)
    bound = (2.0 ** -20 + np.abs(x64) * 2.0 ** -23) * ref
    w, i = _worst(got, ref, bound)
    assert w <= 1.0, f"sigmoid at x={x[i]!r}: got {got[i]!r} ref {ref[i]!r} ({w:.2f} of the bound)"


def test_zoh_input_factor():
    """(exp(ΔA) − 1)/A over Δ log-uniform in [1e-4, 10] and A in −[0.01, 20] (and A = 0: the limit Δ), dense
    around the branch |ΔA| = 1/16."""
    rng = np.random.Generator(np.random.PCG64(7))
    n = 1 << 20
    dl = np.exp(rng.uniform(np.log(1e-4), np.log(10.0), n)).astype(np.float32)
    a = (-np.exp(rng.uniform(np.log(0.01), np.log(20.0), n))).astype(np.float32)
    near = (-0.0625 * np.exp(rng.uniform(-0.05, 0.05, 1 << 16)) / dl[: 1 << 16]).astype(np.float32)
    dl = np.concatenate([dl, dl[: 1 << 16], np.float32([0.5, 2.0])])
    a = np.concatenate([a, near, np.float32([0.0, 0.0])])
    d64, a64 = dl.astype(np.float64), a.astype(np.float64)
    with np.errstate(invalid="ignore", divide="ignore"):
        ref = np.where(a64 == 0.0, d64, np.expm1(d64 * a64) / a64)
    got = _eval("zoh", dl, a)
    w, i = _worst(got, ref, 2.0 ** -18 * np.abs(ref))
    assert w <= 1.0, f"zoh at Δ={dl[i]!r} A={a[i]!r}: got {got[i]!r} ref {ref[i]!r} ({w:.2f} of the bound)"
