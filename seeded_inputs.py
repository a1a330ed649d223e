"""Seeded synthetic inputs for the selective scan (shared by the oracle, the tests and the bench).

This module only draws and stores numbers. It holds none of the scan's
arithmetic: no softplus, no exponentials of the state matrix, no recurrence.
Both the CUDA library and the fp64 oracle consume exactly the arrays returned
here (bf16 tensors as their raw uint16 bit patterns), so neither side ever
sees a value the other did not.

Workloads follow the shapes and value distributions of the Mamba selective
SSM layer described on the pages:

* "Mamba架构与SSM模型：高效序列建模技术解析" §3.2 (the ``Mamba(d_model=768,
  d_state=16, d_conv=4, expand=2)`` example) gives d_state = 16 and the
  expand-2 inner width; §2.2 gives Δ = softplus(Linear(x) + param_Δ).
* "Mamba架构深度剖析：如何以线性时间重塑序列建模" §6 says the step size is
  started around 0.001, which is the low end of the log-uniform range used
  for the Δ bias here.

Random streams: every tensor has its own numpy PCG64 stream keyed by
``(seed, tensor_id)`` via ``numpy.random.SeedSequence``; the fixed tensor ids
are listed in ``TENSOR_IDS``.  Normal values are drawn in fp32 and, for bf16
tensors, rounded to bf16 with round-to-nearest-even on the bit pattern.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

TENSOR_IDS = {"u": 0, "delta": 1, "z": 2, "B": 3, "C": 4, "D": 5, "delta_bias": 6, "h0": 7, "A": 8}

BASE_SEED = 0x5E1EC7


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic selective-scan problem.

    Layout (row-major, last index fastest): u, delta, z, out are
    ``[batch, dim, seqlen]``; B, C are ``[batch, dstate, seqlen]``; A is
    ``[dim, dstate]``; D and delta_bias are ``[dim]``; h0 / h_last are
    ``[batch, dim, dstate]``.  For a decode workload (``steps > 0``) the
    per-step tensors get a leading ``[steps]`` axis and ``seqlen`` is 1.
    """

    name: str
    batch: int
    dim: int
    seqlen: int
    dstate: int
    in_dtype: str  # "f32" or "bf16" for u, delta, z, B, C
    a_init: str  # "neg_n1": A = -(n+1);  "neg_exp_log": A = -exp(log(n+1)) in fp32
    d_init: str  # "normal" or "ones"
    h0_init: str  # "zeros", "none" or "normal"
    has_z: bool = True
    steps: int = 0  # > 0: recurrent decode, one selscan_step per step
    returns_h_last: bool = True

    @property
    def elements(self) -> int:
        """Units of work: B·D·L (for decode: B·D per step times the steps)."""
        if self.steps:
            return self.batch * self.dim * self.steps
        return self.batch * self.dim * self.seqlen


# The five workloads: a tiny fp32 case, a Mamba-130M-like layer, a long
# sequence, a 2.8B-width layer and the recurrent decode step.
WORKLOADS: Dict[str, Workload] = {
    "tiny_fp32": Workload("tiny_fp32", 1, 16, 256, 4, "f32", "neg_n1", "normal", "zeros"),
    "mamba130m_layer": Workload("mamba130m_layer", 8, 1536, 2048, 16, "bf16", "neg_exp_log", "ones", "none"),
    "long_seq_65k": Workload("long_seq_65k", 1, 1536, 65536, 16, "bf16", "neg_exp_log", "ones", "none"),
    "width_2p8b": Workload("width_2p8b", 4, 5120, 4096, 16, "bf16", "neg_n1", "normal", "none"),
    "decode_step": Workload("decode_step", 256, 5120, 1, 16, "bf16", "neg_n1", "normal", "normal", steps=64),
}
WORKLOAD_ORDER = ["tiny_fp32", "mamba130m_layer", "long_seq_65k", "width_2p8b", "decode_step"]


def _rng(seed: int, name: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, TENSOR_IDS[name]])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 (used for host-side reporting only)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal(seed: int, name: str, shape, dtype: str) -> np.ndarray:
    """N(0,1) draws in fp32; bf16 tensors are returned as uint16 bit patterns."""
    x = _rng(seed, name).standard_normal(size=shape, dtype=np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    return x


def delta_bias_init(seed: int, dim: int, dt_min: float = 1e-3, dt_max: float = 1e-1) -> np.ndarray:
    """Per-channel Δ bias: the inverse softplus of dt drawn log-uniform in [dt_min, dt_max].

    dt = exp(U(ln dt_min, ln dt_max)); bias = log(expm1(dt)) = dt + log(-expm1(-dt)),
    evaluated in fp64 and stored as fp32.  This is input preparation (a
    parameter initialisation), not part of the scan.
    """
    uu = _rng(seed, "delta_bias").random(dim)
    dt = np.exp(np.log(dt_min) + uu * (np.log(dt_max) - np.log(dt_min)))
    return (dt + np.log(-np.expm1(-dt))).astype(np.float32)


def a_init(kind: str, dim: int, dstate: int) -> np.ndarray:
    n1 = np.arange(1, dstate + 1, dtype=np.float32)
    if kind == "neg_n1":
        row = -n1
    elif kind == "neg_exp_log":
        a_log = np.log(n1).astype(np.float32)  # A_log = log(n+1) stored in fp32
        row = -np.exp(a_log).astype(np.float32)  # A = -exp(A_log) evaluated in fp32
    else:
        raise ValueError(kind)
    return np.ascontiguousarray(np.broadcast_to(row, (dim, dstate)), dtype=np.float32)


def make_inputs(w: Workload, seed: Optional[int] = None, batch: Optional[int] = None,
                seqlen: Optional[int] = None, steps: Optional[int] = None) -> Dict[str, object]:
    """Draw every input tensor of workload ``w``.

    ``batch``/``seqlen``/``steps`` override the workload's sizes (for smaller
    cases with the same value distributions).  Returns a dict of numpy arrays
    keyed by argument name plus ``"shape"``: (batch, dim, seqlen, dstate).
    Absent optional tensors are ``None``.
    """
    seed = BASE_SEED + WORKLOAD_ORDER.index(w.name) if seed is None else seed
    bsz = w.batch if batch is None else batch
    L = w.seqlen if seqlen is None else seqlen
    T = w.steps if steps is None else steps
    Dm, N = w.dim, w.dstate
    if T:
        lead = (T, bsz, Dm)
        bc = (T, bsz, N)
    else:
        lead = (bsz, Dm, L)
        bc = (bsz, N, L)
    out: Dict[str, object] = {}
    out["u"] = normal(seed, "u", lead, w.in_dtype)
    out["delta"] = normal(seed, "delta", lead, w.in_dtype)
    out["z"] = normal(seed, "z", lead, w.in_dtype) if w.has_z else None
    out["B"] = normal(seed, "B", bc, w.in_dtype)
    out["C"] = normal(seed, "C", bc, w.in_dtype)
    if w.d_init == "normal":
        out["D"] = _rng(seed, "D").standard_normal(Dm, dtype=np.float32)
    else:
        out["D"] = np.ones(Dm, dtype=np.float32)
    out["delta_bias"] = delta_bias_init(seed, Dm)
    out["A"] = a_init(w.a_init, Dm, N)
    if w.h0_init == "zeros":
        out["h0"] = np.zeros((bsz, Dm, N), dtype=np.float32)
    elif w.h0_init == "normal":
        out["h0"] = _rng(seed, "h0").standard_normal((bsz, Dm, N), dtype=np.float32)
    else:
        out["h0"] = None
    out["shape"] = (bsz, Dm, 1 if T else L, N)
    out["in_dtype"] = w.in_dtype
    out["steps"] = T
    return out


def random_case(seed: int, batch: int, dim: int, seqlen: int, dstate: int, in_dtype: str = "f32",
                has_z: bool = True, has_D: bool = True, has_bias: bool = True, has_h0: bool = True,
                a_scale: float = 1.0) -> Dict[str, object]:
    """A small random problem with arbitrary sizes (for ragged-shape and edge-case tests).

    A is drawn as -(a_scale · U(0.5, n+1)) per (d, n) — a general diagonal
    A, not the structured -(n+1) — so that nothing can rely on that pattern.
    """
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0xCA5E])))

    def draw(shape):
        x = rng.standard_normal(size=shape, dtype=np.float32)
        return f32_to_bf16_bits(x) if in_dtype == "bf16" else x

    n1 = np.arange(1, dstate + 1, dtype=np.float32)
    A = -(a_scale * rng.uniform(0.5, 1.0, size=(dim, dstate)).astype(np.float32) * n1).astype(np.float32)
    out: Dict[str, object] = {
        "u": draw((batch, dim, seqlen)),
        "delta": draw((batch, dim, seqlen)),
        "z": draw((batch, dim, seqlen)) if has_z else None,
        "B": draw((batch, dstate, seqlen)),
        "C": draw((batch, dstate, seqlen)),
        "A": np.ascontiguousarray(A),
        "D": rng.standard_normal(dim, dtype=np.float32) if has_D else None,
        "delta_bias": None,
        "h0": rng.standard_normal((batch, dim, dstate), dtype=np.float32) if has_h0 else None,
        "shape": (batch, dim, seqlen, dstate),
        "in_dtype": in_dtype,
        "steps": 0,
    }
    if has_bias:
        uu = rng.random(dim)
        dt = np.exp(np.log(1e-3) + uu * (np.log(1e-1) - np.log(1e-3)))
        out["delta_bias"] = (dt + np.log(-np.expm1(-dt))).astype(np.float32)
    return out


def random_cotangents(seed: int, batch: int, dim: int, seqlen: int, dstate: int, dout_dtype: str = "f32",
                      has_dh_last: bool = True) -> Dict[str, object]:
    """Seeded gradients of a loss with respect to the forward's outputs, for backward tests:
    "dout" [B, D, L] (N(0,1), fp32 or bf16 bit patterns) and "dh_last" [B, D, N] (N(0,1) fp32 or None)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0xB4C])))
    go = rng.standard_normal(size=(batch, dim, seqlen), dtype=np.float32)
    return {"dout": f32_to_bf16_bits(go) if dout_dtype == "bf16" else go,
            "dh_last": rng.standard_normal(size=(batch, dim, dstate), dtype=np.float32) if has_dh_last else None,
            "dout_dtype": dout_dtype}
