"""Pins for the fp64 oracle: checks against facts that do not come from the oracle itself.

Each ``pin_*`` function takes an oracle library handle (``oracle.load()`` or
a build of a deliberately broken copy) and raises ``AssertionError`` when the
oracle disagrees with the closed form, brute force, library routine or
invariant that the pin computes on its own.  No pin retypes the oracle's
recurrence: each computes the same quantity by a different route.

Sources on the pages (by page title and section):
 * "Mamba状态空间模型深度解析：挑战Transformer的下一代序列建模范式" §2.1 — the
   selective recurrence; with B, C, Δ fixed in time it is the time-invariant
   (S4) form.
 * "Mamba: Linear-Time Sequence Modeling with Selective SSMs", "S4的关键思想" —
   a time-invariant SSM is a 1-D convolution with a fixed kernel; and
   "选择性扫描要点" — block-wise scanning with the end state carried to the
   next block.
 * "Mamba架构深度剖析：如何以线性时间重塑序列建模" §3 — the same model runs as a
   recurrence (RNN mode, constant state) or in parallel (convolution mode).
 * "Mamba架构与SSM模型：高效序列建模技术解析" §2.1 — Ā = exp(ΔA); §2.2 —
   Δ = softplus(· + param_Δ).
 * "Mamba状态空间模型深度解析" §2.1 — the selective SSM is a linear time-varying
   system (linear in its input and initial state for fixed Δ, B, C).
 * "Mamba架构与SSM模型：高效序列建模技术解析" §2.1 — the zero-order hold that
   discretises the continuous system h' = A h + B u (exact when the input is
   held over each step), and §3.2 — a bidirectional (reverse-direction) option.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy.special import expit

import oracle
import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _case(seed, Bsz, Dm, L, N, **kw):
    return si.random_case(seed, Bsz, Dm, L, N, in_dtype="f32", **kw)


def _softplus_lib(x):
    # numpy's logaddexp(0, x) = log(e^0 + e^x): a library evaluation of softplus
    return np.logaddexp(0.0, x)


def _rel_close(got, want, rtol, atol=0.0, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    bound = atol + rtol * np.maximum(np.abs(want), np.max(np.abs(want)) * 1e-3 + 1e-300)
    if not np.all(err <= bound):
        i = int(np.argmax(err - bound))
        raise AssertionError(f"{what}: max excess at flat {i}: got {got.flat[i]!r} want {want.flat[i]!r}")


def brute_force(inp, delta_softplus=True):
    """y through the materialised causal matrix, independently of any recurrence.

    For one (b, d) row with S_t = Σ_{r≤t} Δ_r (inclusive prefix sum of the step sizes):
      ∏_{s<r≤t} Ā_r[n] = exp(A[n]·(S_t - S_s))
      M[t,s] = Σ_n C_t[n] · exp(A[n](S_t - S_s)) · Δ_s B_s[n]     (s ≤ t)
      y_t    = Σ_s M[t,s] u_s + D u_t + Σ_n C_t[n] exp(A[n] S_t) h0[n]
      h_last[n] = Σ_s exp(A[n](S_{L-1} - S_s)) Δ_s B_s[n] u_s + exp(A[n] S_{L-1}) h0[n]
    and out = y · z·σ(z) when z is given.
    """
    Bsz, Dm, L, N = inp["shape"]
    u = np.asarray(inp["u"], np.float64)
    x = np.asarray(inp["delta"], np.float64)
    if inp.get("delta_bias") is not None:
        x = x + np.asarray(inp["delta_bias"], np.float64)[None, :, None]
    dt = _softplus_lib(x) if delta_softplus else x
    Bm = np.asarray(inp["B"], np.float64)
    Cm = np.asarray(inp["C"], np.float64)
    A = np.asarray(inp["A"], np.float64)
    Dv = np.zeros(Dm) if inp.get("D") is None else np.asarray(inp["D"], np.float64)
    h0 = np.zeros((Bsz, Dm, N)) if inp.get("h0") is None else np.asarray(inp["h0"], np.float64)
    out = np.zeros((Bsz, Dm, L))
    hl = np.zeros((Bsz, Dm, N))
    tri = np.tril(np.ones((L, L), dtype=bool))
    for b in range(Bsz):
        for d in range(Dm):
            S = np.cumsum(dt[b, d])
            y = Dv[d] * u[b, d].copy()
            for n in range(N):
                decay = np.where(tri, np.exp(A[d, n] * np.where(tri, S[:, None] - S[None, :], 0.0)), 0.0)
                M = Cm[b, n][:, None] * decay * (dt[b, d] * Bm[b, n])[None, :]
                y += M @ u[b, d] + Cm[b, n] * np.exp(A[d, n] * S) * h0[b, d, n]
                hl[b, d, n] = np.sum(np.exp(A[d, n] * (S[-1] - S)) * dt[b, d] * Bm[b, n] * u[b, d]) + \
                    np.exp(A[d, n] * S[-1]) * h0[b, d, n]
            if inp.get("z") is not None:
                zz = np.asarray(inp["z"], np.float64)[b, d]
                y = y * zz * expit(zz)
            out[b, d] = y
    return out, hl


def pin_brute_force(lib):
    """Oracle == materialised causal matrix on tiny random inputs (gate, bias, h0, D all on)."""
    for seed, shape in [(1, (2, 3, 24, 3)), (2, (1, 2, 17, 1)), (3, (1, 2, 9, 5))]:
        inp = _case(seed, *shape)
        got, ghl = oracle.selscan_fwd(inp, lib=lib, nthreads=1)
        want, whl = brute_force(inp)
        _rel_close(got, want, 1e-11, what=f"brute force out {shape}")
        _rel_close(ghl, whl, 1e-11, what=f"brute force h_last {shape}")


def pin_lti_convolution(lib):
    """Constant Δ, B, C: y = K * u + D·u with K_k = Σ_n C_n Ā_n^k Δ B_n (time-invariant SSM as a convolution)."""
    rng = np.random.default_rng(11)
    Bsz, Dm, L, N = 1, 2, 40, 4
    inp = _case(12, Bsz, Dm, L, N, has_z=False, has_bias=False, has_h0=False)
    c = np.float32(0.375)  # Δ, exactly representable; delta_softplus off so Δ = δ
    inp["delta"] = np.full((Bsz, Dm, L), c, dtype=np.float32)
    Bn = rng.standard_normal(N).astype(np.float32)
    Cn = rng.standard_normal(N).astype(np.float32)
    inp["B"] = np.ascontiguousarray(np.broadcast_to(Bn[None, :, None], (Bsz, N, L)), dtype=np.float32)
    inp["C"] = np.ascontiguousarray(np.broadcast_to(Cn[None, :, None], (Bsz, N, L)), dtype=np.float32)
    got, _ = oracle.selscan_fwd(inp, delta_softplus=False, lib=lib, nthreads=1)
    A = np.asarray(inp["A"], np.float64)
    k = np.arange(L)
    for d in range(Dm):
        abar = np.exp(float(c) * A[d])  # [N]
        K = (Cn[None, :].astype(np.float64) * np.power(abar[None, :], k[:, None]) * float(c) * Bn[None, :]).sum(1)
        uu = np.asarray(inp["u"][0, d], np.float64)
        want = np.convolve(uu, K)[:L] + float(inp["D"][d]) * uu
        _rel_close(got[0, d], want, 1e-11, what=f"LTI convolution d={d}")


def pin_delta_to_zero(lib):
    """Δ → 0: Ā → 1 and Δ·B → 0, so y = C·h0 + D·u and h_last = h0 (y = D·u when h0 = 0)."""
    inp = _case(21, 1, 3, 30, 4, has_z=False)
    # (a) exact: softplus off, δ = 0, bias = 0 -> Δ = 0 exactly
    inp["delta"] = np.zeros_like(inp["delta"])
    inp["delta_bias"] = None
    got, hl = oracle.selscan_fwd(inp, delta_softplus=False, lib=lib, nthreads=1)
    h0 = np.asarray(inp["h0"], np.float64)
    want = np.einsum("nt,dn->dt", np.asarray(inp["C"][0], np.float64), h0[0]) + \
        np.asarray(inp["D"], np.float64)[:, None] * np.asarray(inp["u"][0], np.float64)
    _rel_close(got[0], want, 1e-14, what="Δ=0 out")
    assert np.array_equal(hl, h0), "Δ=0: h_last must equal h0 exactly"
    # (b) limit: softplus with bias -40 -> Δ ≈ e^-40 ~ 4e-18; h0 = 0 -> y = D·u
    inp2 = _case(22, 1, 3, 30, 4, has_z=False, has_h0=False)
    inp2["delta_bias"] = np.full(3, -40.0, dtype=np.float32)
    got2, hl2 = oracle.selscan_fwd(inp2, lib=lib, nthreads=1)
    want2 = np.asarray(inp2["D"], np.float64)[:, None] * np.asarray(inp2["u"][0], np.float64)
    _rel_close(got2[0], want2, 1e-12, atol=1e-14, what="Δ→0 out")
    assert np.max(np.abs(hl2)) < 1e-14, "Δ→0: h_last must vanish with h0 = 0"


def pin_prefix_sum(lib):
    """A = 0, N = 1, Δ = δ: Ā = 1 and h_t = h0 + Σ_{s≤t} Δ_s B_s u_s, a cumulative sum; y = C_t h_t."""
    Bsz, Dm, L, N = 2, 2, 50, 1
    inp = _case(31, Bsz, Dm, L, N, has_z=False, has_D=False, has_bias=False)
    inp["A"] = np.zeros((Dm, N), dtype=np.float32)
    got, hl = oracle.selscan_fwd(inp, delta_softplus=False, lib=lib, nthreads=1)
    for b in range(Bsz):
        for d in range(Dm):
            terms = np.asarray(inp["delta"][b, d], np.float64) * np.asarray(inp["B"][b, 0], np.float64) * \
                np.asarray(inp["u"][b, d], np.float64)
            h = float(inp["h0"][b, d, 0]) + np.cumsum(terms)
            _rel_close(got[b, d], np.asarray(inp["C"][b, 0], np.float64) * h, 1e-12, atol=1e-13,
                       what="prefix sum out")
            _rel_close(hl[b, d, 0], h[-1], 1e-12, what="prefix sum h_last")


def pin_memoryless(lib):
    """Very negative A with Δ bounded below: Ā underflows to 0, so y_t = Δ_t u_t Σ_n C_t[n] B_t[n] + D u_t."""
    Bsz, Dm, L, N = 1, 3, 20, 4
    inp = _case(41, Bsz, Dm, L, N, has_z=False, has_bias=False)
    inp["A"] = np.full((Dm, N), -1e6, dtype=np.float32)  # Δ ≥ softplus(-6) ≈ 2.5e-3 -> ΔA ≤ -2500
    inp["delta"] = np.clip(inp["delta"], -6, 6).astype(np.float32)
    got, hl = oracle.selscan_fwd(inp, lib=lib, nthreads=1)
    dt = _softplus_lib(np.asarray(inp["delta"][0], np.float64))
    u = np.asarray(inp["u"][0], np.float64)
    cb = (np.asarray(inp["C"][0], np.float64) * np.asarray(inp["B"][0], np.float64)).sum(0)  # [L]
    want = dt * u * cb[None, :] + np.asarray(inp["D"], np.float64)[:, None] * u
    _rel_close(got[0], want, 1e-13, atol=1e-15, what="memoryless out")
    wh = dt[:, -1:] * u[:, -1:] * np.asarray(inp["B"][0, :, -1], np.float64)[None, :]
    _rel_close(hl[0], wh, 1e-13, atol=1e-15, what="memoryless h_last")


def pin_gate(lib):
    """SiLU gate: z = 0 gives out = 0; and the gate equals z·σ(z) with σ from scipy."""
    inp = _case(51, 1, 2, 16, 3)
    inp["z"] = np.zeros_like(inp["z"])
    got, _ = oracle.selscan_fwd(inp, lib=lib, nthreads=1)
    assert np.all(got == 0.0), "z = 0 must zero the output"
    inp2 = _case(52, 1, 2, 16, 3)
    g_on, _ = oracle.selscan_fwd(inp2, lib=lib, nthreads=1)
    inp2_off = dict(inp2)
    inp2_off["z"] = None
    g_off, _ = oracle.selscan_fwd(inp2_off, lib=lib, nthreads=1)
    zz = np.asarray(inp2["z"], np.float64)
    _rel_close(g_on, g_off * zz * expit(zz), 1e-14, atol=1e-300, what="gate = y·z·σ(z)")


def pin_scalar_functions(lib):
    """softplus against numpy's logaddexp(0, x); silu against z·expit(z); bf16 widening on known bit patterns."""
    xs = np.concatenate([np.linspace(-60, 60, 241), [-700.0, -30.5, -1e-9, 0.0, 1e-9, 33.0, 700.0]])
    for x in xs:
        want = float(np.logaddexp(0.0, x))
        got = lib.oracle_softplus(float(x))
        assert abs(got - want) <= 2e-16 * max(abs(want), 1e-300) + 1e-320, (x, got, want)
    assert lib.oracle_softplus(0.0) == np.log(2.0)
    for zv in np.linspace(-40, 40, 161):
        want = float(zv * expit(zv))
        got = lib.oracle_silu(float(zv))
        assert abs(got - want) <= 4e-16 * abs(want) + 1e-300, (zv, got, want)
    known = {0x3F80: 1.0, 0xC000: -2.0, 0x3F81: 1.0078125, 0x0000: 0.0, 0x0001: 2.0 ** -133,
             0x7F7F: 3.3895313892515355e38, 0x3E80: 0.25, 0xBF40: -0.75}
    for bits, val in known.items():
        assert lib.oracle_load_bf16(bits) == val, (hex(bits), lib.oracle_load_bf16(bits), val)


def pin_carry(lib):
    """Block carry: fwd over L equals fwd over L1 then fwd over L2 started from the carried end state."""
    inp = _case(61, 2, 3, 70, 4)
    full, hfull = oracle.selscan_fwd(inp, lib=lib, nthreads=1)
    for L1 in (1, 23, 69):
        a = {k: (v[..., :L1].copy() if k in ("u", "delta", "z", "B", "C") and v is not None else v)
             for k, v in inp.items()}
        a["shape"] = (2, 3, L1, 4)
        b = {k: (v[..., L1:].copy() if k in ("u", "delta", "z", "B", "C") and v is not None else v)
             for k, v in inp.items()}
        b["shape"] = (2, 3, 70 - L1, 4)
        o1, h1 = oracle.selscan_fwd(a, lib=lib, nthreads=1)
        o2, h2 = oracle.selscan_fwd(b, lib=lib, nthreads=1, h0_f64=h1)
        _rel_close(np.concatenate([o1, o2], axis=-1), full, 1e-13, atol=1e-300, what=f"carry out L1={L1}")
        _rel_close(h2, hfull, 1e-13, what=f"carry h_last L1={L1}")


def pin_step_equals_fwd(lib):
    """RNN mode: T decode steps carrying the state reproduce the forward over T steps."""
    Bsz, Dm, T, N = 2, 3, 12, 4
    inp = _case(71, Bsz, Dm, T, N)
    full, hfull = oracle.selscan_fwd(inp, lib=lib, nthreads=1)
    dec = {"shape": (Bsz, Dm, 1, N), "in_dtype": "f32", "steps": T, "A": inp["A"], "D": inp["D"],
           "delta_bias": inp["delta_bias"]}
    for k in ("u", "delta", "z"):
        dec[k] = np.ascontiguousarray(np.moveaxis(inp[k], -1, 0))  # [T, B, D]
    for k in ("B", "C"):
        dec[k] = np.ascontiguousarray(np.moveaxis(inp[k], -1, 0))  # [T, B, N]
    state = np.asarray(inp["h0"], np.float64).copy()
    for t in range(T):
        o = oracle.selscan_step(dec, state, step=t, lib=lib)
        _rel_close(o, full[..., t], 1e-13, atol=1e-300, what=f"step {t}")
    _rel_close(state, hfull, 1e-13, what="step final state")


def pin_linearity(lib):
    """Superposition in (u, h0) for fixed Δ, B, C and no gate (linear time-varying system)."""
    Bsz, Dm, L, N = 1, 2, 33, 3
    base = _case(81, Bsz, Dm, L, N, has_z=False)
    rng = np.random.default_rng(82)

    def grid(shape):  # multiples of 2^-10 in [-4, 4): sums stay exact in fp32
        return (rng.integers(-4096, 4096, size=shape) / 1024.0).astype(np.float32)

    u1, u2 = grid((Bsz, Dm, L)), grid((Bsz, Dm, L))
    h1, h2 = grid((Bsz, Dm, N)), grid((Bsz, Dm, N))

    def run(u, h):
        c = dict(base)
        c["u"], c["h0"] = u, h
        return oracle.selscan_fwd(c, lib=lib, nthreads=1)

    o1, hl1 = run(u1, h1)
    o2, hl2 = run(u2, h2)
    o12, hl12 = run((u1 + u2).astype(np.float32), (h1 + h2).astype(np.float32))
    _rel_close(o12, o1 + o2, 1e-12, atol=1e-12, what="linearity out")
    _rel_close(hl12, hl1 + hl2, 1e-12, atol=1e-12, what="linearity h_last")
    o3, _ = run((3 * u1).astype(np.float32), (3 * h1).astype(np.float32))
    _rel_close(o3, 3 * o1, 1e-12, atol=1e-12, what="homogeneity out")


def pin_causality(lib):
    """Changing u at t0 leaves every output before t0 bit-identical, and changes the output at t0."""
    inp = _case(91, 1, 2, 40, 3)
    o, _ = oracle.selscan_fwd(inp, lib=lib, nthreads=1)
    for t0 in (0, 17, 39):
        p = dict(inp)
        p["u"] = inp["u"].copy()
        p["u"][..., t0] += 1.0
        op, _ = oracle.selscan_fwd(p, lib=lib, nthreads=1)
        assert np.array_equal(op[..., :t0], o[..., :t0]), f"output before t0={t0} changed"
        assert np.all(op[..., t0] != o[..., t0]), f"output at t0={t0} did not change"


def _closed_form(exprs):
    """Evaluate the fixture's closed-form expressions (arithmetic in ln2 and ln3 only)."""
    env = {"__builtins__": {}, "ln2": math.log(2.0), "ln3": math.log(3.0)}
    return np.array([float(eval(e, env)) for e in exprs])


def pin_worked_examples(lib):
    """Hand-derived sequences stored under tests/golden/ (values from the definitions, not from code)."""
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        L = len(c["u"])
        N = len(c["A"])
        inp = {
            "shape": (1, 1, L, N), "in_dtype": "f32", "steps": 0,
            "u": np.array(c["u"], np.float32).reshape(1, 1, L),
            "delta": np.array(c["delta"], np.float32).reshape(1, 1, L),
            "z": None if c.get("z") is None else np.array(c["z"], np.float32).reshape(1, 1, L),
            "B": np.array(c["B"], np.float32).reshape(1, N, L),
            "C": np.array(c["C"], np.float32).reshape(1, N, L),
            "A": np.array(c["A"], np.float32).reshape(1, N),
            "D": np.array([c["D"]], np.float32),
            "delta_bias": None if c.get("delta_bias") is None else np.array([c["delta_bias"]], np.float32),
            "h0": np.array(c["h0"], np.float32).reshape(1, 1, N),
        }
        out, hl = oracle.selscan_fwd(inp, delta_softplus=c["delta_softplus"], lib=lib, nthreads=1)
        _rel_close(out[0, 0], _closed_form(c["expect_out"]), c["rtol"], atol=c["rtol"], what=c["name"] + " out")
        _rel_close(hl[0, 0], _closed_form(c["expect_h_last"]), c["rtol"], atol=c["rtol"],
                   what=c["name"] + " h_last")


def pin_row_subset(lib):
    """Computing a listed subset of rows gives the same rows as the full computation."""
    inp = _case(101, 2, 5, 19, 3)
    full, hl = oracle.selscan_fwd(inp, lib=lib, nthreads=3)
    rows = [7, 0, 9, 4]
    sub, shl = oracle.selscan_fwd(inp, rows=rows, lib=lib, nthreads=2)
    assert np.array_equal(sub, full.reshape(10, 19)[rows]) and np.array_equal(shl, hl.reshape(10, 3)[rows])


def brute_force_reverse(inp, delta_softplus=True):
    """The reverse-direction scan through its materialised anti-causal matrix.

    Scanning from t = L-1 down to 0, h_t = Ā_t h_{t+1} + Δ_t B_t u_t with h_L = h0.  With the
    exclusive prefix sum P_t = Σ_{r<t} Δ_r, ∏_{t≤r<s} Ā_r[n] = exp(A[n](P_s - P_t)), so
      h_t[n] = Σ_{s≥t} exp(A[n](P_s - P_t)) Δ_s B_s[n] u_s + exp(A[n](P_L - P_t)) h0[n]
    and y_t = Σ_n C_t[n] h_t[n] + D u_t (gated by silu(z)); h_last is h_0.
    """
    Bsz, Dm, L, N = inp["shape"]
    u = np.asarray(inp["u"], np.float64)
    x = np.asarray(inp["delta"], np.float64)
    if inp.get("delta_bias") is not None:
        x = x + np.asarray(inp["delta_bias"], np.float64)[None, :, None]
    dt = _softplus_lib(x) if delta_softplus else x
    Bm = np.asarray(inp["B"], np.float64)
    Cm = np.asarray(inp["C"], np.float64)
    A = np.asarray(inp["A"], np.float64)
    Dv = np.zeros(Dm) if inp.get("D") is None else np.asarray(inp["D"], np.float64)
    h0 = np.zeros((Bsz, Dm, N)) if inp.get("h0") is None else np.asarray(inp["h0"], np.float64)
    out = np.zeros((Bsz, Dm, L))
    hl = np.zeros((Bsz, Dm, N))
    upper = np.triu(np.ones((L, L), dtype=bool))  # s >= t
    for b in range(Bsz):
        for d in range(Dm):
            P = np.concatenate([[0.0], np.cumsum(dt[b, d])])  # P_0 .. P_L
            y = Dv[d] * u[b, d].copy()
            for n in range(N):
                gap = np.where(upper, P[None, :L] - P[:L, None], 0.0)  # P_s - P_t for s >= t
                decay = np.where(upper, np.exp(A[d, n] * gap), 0.0)
                hn = decay @ (dt[b, d] * Bm[b, n] * u[b, d]) + np.exp(A[d, n] * (P[L] - P[:L])) * h0[b, d, n]
                y += Cm[b, n] * hn
                hl[b, d, n] = hn[0]
            if inp.get("z") is not None:
                zz = np.asarray(inp["z"], np.float64)[b, d]
                y = y * zz * expit(zz)
            out[b, d] = y
    return out, hl


def pin_reverse_brute_force(lib):
    """Reverse-direction oracle == materialised anti-causal matrix (gate, bias, h0, D all on)."""
    for seed, shape in [(81, (2, 3, 21, 3)), (82, (1, 2, 13, 1)), (83, (1, 2, 9, 5))]:
        inp = _case(seed, *shape)
        got, ghl = oracle.selscan_fwd(inp, reverse=True, lib=lib, nthreads=1)
        want, whl = brute_force_reverse(inp)
        _rel_close(got, want, 1e-11, what=f"reverse brute force out {shape}")
        _rel_close(ghl, whl, 1e-11, what=f"reverse brute force h_last {shape}")


def _rk4_zoh_reference(A, Bv, u, dt, h0, substeps=400):
    """The continuous system h'(τ) = A h + B_t u_t, held constant over each interval of length Δ_t
    (a zero-order hold of the input), integrated numerically with classical RK4."""
    h = np.array(h0, dtype=np.float64)
    hs = []
    for t in range(len(dt)):
        f = Bv[:, t] * u[t]
        k = dt[t] / substeps
        for _ in range(substeps):
            k1 = A * h + f
            k2 = A * (h + 0.5 * k * k1) + f
            k3 = A * (h + 0.5 * k * k2) + f
            k4 = A * (h + k * k3) + f
            h = h + (k / 6.0) * (k1 + 2 * k2 + 2 * k3 + k4)
        hs.append(h.copy())
    return np.array(hs)  # [L, N]: state at the end of each interval


def pin_zoh_matches_ode(lib):
    """With zoh, the recurrence samples the continuous SSM exactly: each step advances the state of
    h' = A h + B u over Δ_t with the input held constant, which RK4 reproduces to ~1e-10."""
    Bsz, Dm, L, N = 1, 2, 12, 3
    inp = _case(91, Bsz, Dm, L, N, has_z=False, has_bias=False)
    inp["delta"] = (np.abs(inp["delta"]) * 0.7 + 0.05).astype(np.float32)  # Δ = δ (softplus off), 0.05..~2.5
    got, hl = oracle.selscan_fwd(inp, delta_softplus=False, zoh=True, lib=lib, nthreads=1)
    for d in range(Dm):
        A = np.asarray(inp["A"][d], np.float64)
        dt = np.asarray(inp["delta"][0, d], np.float64)
        u = np.asarray(inp["u"][0, d], np.float64)
        hs = _rk4_zoh_reference(A, np.asarray(inp["B"][0], np.float64), u, dt, inp["h0"][0, d])
        y = (np.asarray(inp["C"][0], np.float64).T * hs).sum(1) + float(inp["D"][d]) * u
        _rel_close(got[0, d], y, 1e-9, atol=1e-12, what="zoh out vs ODE")
        _rel_close(hl[0, d], hs[-1], 1e-9, atol=1e-12, what="zoh h_last vs ODE")


def pin_zoh_limits(lib):
    """zoh at A = 0 is exactly the Δ·B scan (the limit of (e^{ΔA} - 1)/A), and for small Δ|A| the two
    agree to first order: their difference shrinks like Δ²."""
    inp = _case(92, 1, 3, 20, 4, has_z=False)
    inp["A"] = np.zeros_like(inp["A"])
    a, ah = oracle.selscan_fwd(inp, zoh=True, lib=lib, nthreads=1)
    b, bh = oracle.selscan_fwd(inp, zoh=False, lib=lib, nthreads=1)
    assert np.array_equal(a, b) and np.array_equal(ah, bh), "zoh at A = 0 must equal the Δ·B scan"
    inp2 = _case(93, 1, 2, 8, 2, has_z=False, has_bias=False, has_h0=False)
    diffs = []
    for scale in (1e-2, 1e-3):
        inp2["delta"] = np.full_like(inp2["delta"], scale)
        z, _ = oracle.selscan_fwd(inp2, delta_softplus=False, zoh=True, lib=lib, nthreads=1)
        e, _ = oracle.selscan_fwd(inp2, delta_softplus=False, zoh=False, lib=lib, nthreads=1)
        diffs.append(np.max(np.abs(z - e)) / np.max(np.abs(e)))
    assert 50 < diffs[0] / diffs[1] < 200, f"zoh minus Δ·B should shrink like Δ²: {diffs}"


def pin_conv_silu(lib):
    """The conv front against numpy's full convolution (first L outputs: causal, zero history) plus the
    bias, and scipy's logistic for the SiLU: u = z·σ(z), z = cb + Σ_k w[k] x[t-3+k]."""
    rng = np.random.default_rng(101)
    Bsz, Dm, L, K = 2, 3, 37, 4
    x = rng.standard_normal((Bsz, Dm, L)).astype(np.float32)
    w = rng.standard_normal((Dm, K)).astype(np.float32)
    cb = rng.standard_normal(Dm).astype(np.float32)
    got = oracle.conv_silu(x, w, cb, "f32", lib=lib)
    for b in range(Bsz):
        for d in range(Dm):
            zz = np.convolve(x[b, d].astype(np.float64), w[d, ::-1].astype(np.float64))[:L] + float(cb[d])
            _rel_close(got[b, d], zz * expit(zz), 1e-13, atol=1e-15, what="conv+silu")
    # an impulse at t0 reads the taps back in causal order: z_{t0+j} = w[K-1-j] for j < K, 0 after
    imp = np.zeros((1, 1, 12), dtype=np.float32)
    imp[0, 0, 5] = 1.0
    wi = np.array([[0.25, -0.5, 2.0, 1.5]], dtype=np.float32)
    gi = oracle.conv_silu(imp, wi, None, "f32", lib=lib)[0, 0]
    zi = np.zeros(12)
    zi[5:9] = [1.5, 2.0, -0.5, 0.25]
    _rel_close(gi, zi * expit(zi), 1e-15, atol=1e-300, what="conv impulse response")


def pin_conv_feeds_scan(lib):
    """The scan with an fp64 u override equals the scan on that u stored in fp32 to fp32 rounding."""
    inp = _case(102, 1, 2, 30, 3)
    u64 = np.asarray(inp["u"], np.float64) * 0.5
    inp32 = dict(inp)
    inp32["u"] = u64.astype(np.float32)  # exact: halving an fp32 value only changes its exponent
    a, ah = oracle.selscan_fwd(inp, u_f64=u64, lib=lib, nthreads=1)
    b, bh = oracle.selscan_fwd(inp32, lib=lib, nthreads=1)
    assert np.array_equal(a, b) and np.array_equal(ah, bh), "u_f64 must replace u exactly"


# ---- the backward (gradients) -------------------------------------------------------------------
#
# The pages describe training with the states recomputed in the backward pass instead of stored
# ("Mamba状态空间模型深度解析：挑战Transformer的下一代序列建模范式" §2.2); the gradients themselves are
# fixed by the forward.  Three independent routes pin them: central differences of the forward oracle,
# the transpose of the materialised causal matrix (the forward is linear in u and h0 for fixed Δ), and
# suffix sums in the prefix-sum special case.

def _fd_loss(inp, w, v, lib, delta_softplus):
    out, hl = oracle.selscan_fwd(inp, delta_softplus=delta_softplus, lib=lib, nthreads=1)
    return float(np.sum(w * out) + np.sum(v * hl))


def pin_bwd_finite_differences(lib):
    """Every gradient == central differences of the forward oracle, L = Σ w·out + Σ v·h_last."""
    rng = np.random.default_rng(41)
    for seed, shape, sp in [(11, (2, 3, 10, 3), True), (12, (1, 2, 9, 2), False)]:
        inp = _case(seed, *shape)
        if not sp:  # keep Δ = δ positive without softplus
            inp["delta_bias"] = None
            inp["delta"] = (np.abs(inp["delta"]) * 0.05 + 0.01).astype(np.float32)
        Bsz, Dm, L, N = shape
        w = rng.standard_normal((Bsz, Dm, L))
        v = rng.standard_normal((Bsz, Dm, N))
        g = oracle.selscan_bwd(inp, w, dh_last=v, delta_softplus=sp, lib=lib, nthreads=1)
        for name in ("u", "delta", "z", "A", "B", "C", "D", "delta_bias", "h0"):
            arr = inp.get(name)
            if arr is None:
                continue
            arr = np.asarray(arr, dtype=np.float32)
            flat = np.arange(arr.size)
            pick = flat if arr.size <= 24 else rng.choice(flat, size=12, replace=False)
            for i in pick:
                x = float(arr.flat[i])
                hstep = 2.0 ** -12 * 2.0 ** max(0, math.floor(math.log2(abs(x) + 1.0)))
                vals = []
                for sgn in (1.0, -1.0):
                    a2 = arr.copy()
                    a2.flat[i] = np.float32(x + sgn * hstep)
                    vals.append((float(a2.flat[i]), _fd_loss(dict(inp, **{name: a2}), w, v, lib, sp)))
                fd = (vals[0][1] - vals[1][1]) / (vals[0][0] - vals[1][0])
                got = float(g[name].flat[i])
                scale = float(np.max(np.abs(g[name]))) + 1e-12
                if not abs(got - fd) <= 2e-5 * scale + 1e-6 * abs(fd):
                    raise AssertionError(f"d{name}[{i}] {shape}: oracle {got!r}, central difference {fd!r}")


def pin_bwd_adjoint_matrix(lib):
    """du and dh0 == the transposes of the materialised maps u -> (out, h_last) and h0 -> (out, h_last)."""
    rng = np.random.default_rng(43)
    for seed, shape in [(13, (2, 2, 14, 3)), (14, (1, 3, 9, 1))]:
        inp = _case(seed, *shape, has_z=False)
        Bsz, Dm, L, N = shape
        w = rng.standard_normal((Bsz, Dm, L))
        v = rng.standard_normal((Bsz, Dm, N))
        g = oracle.selscan_bwd(inp, w, dh_last=v, lib=lib, nthreads=1)
        x = np.asarray(inp["delta"], np.float64) + np.asarray(inp["delta_bias"], np.float64)[None, :, None]
        dt = _softplus_lib(x)
        Bm, Cm = np.asarray(inp["B"], np.float64), np.asarray(inp["C"], np.float64)
        A, Dv = np.asarray(inp["A"], np.float64), np.asarray(inp["D"], np.float64)
        tri = np.tril(np.ones((L, L), dtype=bool))
        for b in range(Bsz):
            for d in range(Dm):
                S = np.cumsum(dt[b, d])
                M = np.diag(np.full(L, Dv[d]))
                du_hl = np.zeros(L)
                dh0 = np.zeros(N)
                for n in range(N):
                    decay = np.where(tri, np.exp(A[d, n] * np.where(tri, S[:, None] - S[None, :], 0.0)), 0.0)
                    M = M + Cm[b, n][:, None] * decay * (dt[b, d] * Bm[b, n])[None, :]
                    Hrow = np.exp(A[d, n] * (S[-1] - S)) * dt[b, d] * Bm[b, n]  # u_s -> h_last[n]
                    du_hl += Hrow * v[b, d, n]
                    dh0[n] = np.sum(Cm[b, n] * np.exp(A[d, n] * S) * w[b, d]) + np.exp(A[d, n] * S[-1]) * v[b, d, n]
                _rel_close(g["u"][b, d], M.T @ w[b, d] + du_hl, 1e-10, what=f"du adjoint {shape}")
                _rel_close(g["h0"][b, d], dh0, 1e-10, what=f"dh0 adjoint {shape}")


def pin_bwd_prefix_sum(lib):
    """A = 0, N = 1, no softplus, no gate: every gradient by suffix sums of the cumulative-sum model."""
    inp = _case(15, 2, 3, 16, 1, has_z=False)
    inp["A"] = np.zeros_like(inp["A"])
    inp["delta_bias"] = None
    rng = np.random.default_rng(44)
    Bsz, Dm, L, _ = inp["shape"]
    w = rng.standard_normal((Bsz, Dm, L))
    v = rng.standard_normal((Bsz, Dm, 1))
    # three worker threads over the six rows: the sums over rows are formed per worker and then added
    g = oracle.selscan_bwd(inp, w, dh_last=v, delta_softplus=False, lib=lib, nthreads=3)
    u = np.asarray(inp["u"], np.float64)
    dt = np.asarray(inp["delta"], np.float64)
    Bm, Cm = np.asarray(inp["B"], np.float64)[:, 0], np.asarray(inp["C"], np.float64)[:, 0]
    Dv, h0 = np.asarray(inp["D"], np.float64), np.asarray(inp["h0"], np.float64)[..., 0]
    h = h0[..., None] + np.cumsum(dt * Bm[:, None, :] * u, axis=-1)            # h_t
    hprev = np.concatenate([h0[..., None], h[..., :-1]], axis=-1)              # h_{t-1}
    R = np.flip(np.cumsum(np.flip(Cm[:, None, :] * w, -1), -1), -1) + v        # Σ_{t' ≥ t} C w + v
    _rel_close(g["u"], dt * Bm[:, None, :] * R + Dv[None, :, None] * w, 1e-11, what="du prefix sum")
    _rel_close(g["delta"], Bm[:, None, :] * u * R, 1e-11, what="ddelta prefix sum")
    _rel_close(g["B"][:, 0], np.sum(dt * u * R, axis=1), 1e-11, what="dB prefix sum")
    _rel_close(g["C"][:, 0], np.sum(w * h, axis=1), 1e-11, what="dC prefix sum")
    _rel_close(g["D"], np.sum(w * u, axis=(0, 2)), 1e-11, what="dD prefix sum")
    _rel_close(g["A"][:, 0], np.sum(R * hprev * dt, axis=(0, 2)), 1e-11, what="dA prefix sum")
    _rel_close(g["h0"][..., 0], R[..., 0], 1e-11, what="dh0 prefix sum")


ALL_PINS = [pin_brute_force, pin_lti_convolution, pin_delta_to_zero, pin_prefix_sum, pin_memoryless, pin_gate,
            pin_scalar_functions, pin_carry, pin_step_equals_fwd, pin_linearity, pin_causality,
            pin_worked_examples, pin_row_subset, pin_reverse_brute_force, pin_zoh_matches_ode, pin_zoh_limits,
            pin_conv_silu, pin_conv_feeds_scan, pin_bwd_finite_differences, pin_bwd_adjoint_matrix,
            pin_bwd_prefix_sum]
