"""Helpers for GPU-vs-oracle parity tests: numpy inputs -> CUDA tensors -> libselscan -> numpy."""
from __future__ import annotations

import numpy as np

FP32_TOL = (1e-4, 1e-4)  # fp32 inputs: |out - ref| <= 1e-4 + 1e-4·|ref|
BF16_TOL = (2e-3, 2e-3)  # bf16 inputs, fp32 state: |out - ref| <= 2e-3 + 2e-3·|ref|
H_RTOL = 1e-4  # h_last: |h - ref| <= 1e-4 · max_n |ref[b, d, :]|, relative to each channel's state vector


def to_dev(a, in_dtype=None, device="cuda"):
    """numpy -> torch CUDA tensor; uint16 arrays are bf16 bit patterns."""
    import torch

    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def gpu_fwd(inp, delta_softplus=True, out_dtype="f32", h_last=True, stream=None, **over):
    import torch

    import selective_state_space_152_b300 as ss

    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    t.update(over)
    od = torch.float32 if out_dtype == "f32" else torch.bfloat16
    out, hl = ss.selscan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                             delta_bias=t["delta_bias"], delta_softplus=delta_softplus, h0=t["h0"], out_dtype=od,
                             return_h_last=h_last, stream=stream)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), (None if hl is None else hl.cpu().numpy().astype(np.float64))


def gpu_fwd_ex(inp, reverse=False, zoh=False, delta_softplus=True, out_dtype="f32"):
    """selscan_fwd_ex (reverse and/or exact zero-order hold) on an input dict; float64 numpy results."""
    import torch

    import selective_state_space_152_b300 as ss

    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    od = torch.float32 if out_dtype == "f32" else torch.bfloat16
    out, hl = ss.selscan_fwd_ex(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                                delta_bias=t["delta_bias"], delta_softplus=delta_softplus, h0=t["h0"],
                                out_dtype=od, return_h_last=True, reverse=reverse, zoh=zoh)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), hl.cpu().numpy().astype(np.float64)


def gpu_fwd_conv(inp, conv_w, conv_b, zoh=False, delta_softplus=True):
    """selscan_fwd_conv with x = inp["u"] and the given taps and bias; float64 numpy results."""
    import torch

    import selective_state_space_152_b300 as ss

    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    w = torch.from_numpy(np.ascontiguousarray(conv_w, dtype=np.float32)).cuda()
    cb = None if conv_b is None else torch.from_numpy(np.ascontiguousarray(conv_b, dtype=np.float32)).cuda()
    out, hl = ss.selscan_fwd_conv(t["u"], w, cb, t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                                  delta_bias=t["delta_bias"], delta_softplus=delta_softplus, h0=t["h0"],
                                  return_h_last=True, zoh=zoh)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), hl.cpu().numpy().astype(np.float64)


def tol_for(in_dtype):
    return FP32_TOL if in_dtype == "f32" else BF16_TOL


def check_out(got, ref, in_dtype, what="out", extra_rel=0.0):
    atol, rtol = tol_for(in_dtype)
    err = np.abs(got - ref)
    bound = atol + (rtol + extra_rel) * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = int(np.argmax(np.where(bad, err - bound, -np.inf)))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at flat {i}: "
                             f"got {got.flat[i]!r} ref {ref.flat[i]!r} (max err {err.max():.3e})")
    return float(err.max())


def check_h(got, ref, what="h_last"):
    """Relative error of each channel's final state vector in the max norm over its N states.

    A state entry near zero is the difference of terms as large as the vector's largest entry, so its
    fp32 error is set by that scale; the bound is therefore relative to max_n |ref| of the channel.
    """
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    scale = np.max(np.abs(ref), axis=-1, keepdims=True)
    err = np.abs(got - ref)
    bound = H_RTOL * np.broadcast_to(scale, ref.shape)
    bad = ~(err <= bound)
    if bad.any():
        i = int(np.argmax(np.where(bad, err - bound, -np.inf)))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at flat {i}: "
                             f"got {got.flat[i]!r} ref {ref.flat[i]!r} "
                             f"(channel scale {np.broadcast_to(scale, ref.shape).flat[i]:.3e})")
    return float(np.max(err / np.maximum(np.broadcast_to(scale, ref.shape), 1e-300)))


def sample_rows(Bsz, Dm, k, seed=0):
    """k flat row indices b*D + d, always including the first and last row."""
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(Bsz * Dm, size=min(k, Bsz * Dm), replace=False).tolist())
    rows.update({0, Bsz * Dm - 1})
    return sorted(rows)


def decode_as_forward(inp):
    """A decode input ([T, B, D] / [T, B, N] per-step tensors) as one forward problem over its T steps:
    u, delta, z become [B, D, T] and B, C [B, N, T]; h0 stays the start state.  T decode steps carrying
    the state equal the forward over those T steps (an oracle pin), so the oracle can check every row of
    a full-size decode run with its threaded forward."""
    T = inp["steps"]
    Bsz, Dm, _, N = inp["shape"]
    mv = lambda a: None if a is None else np.ascontiguousarray(np.moveaxis(np.asarray(a), 0, -1))  # noqa: E731
    return {"shape": (Bsz, Dm, T, N), "in_dtype": inp["in_dtype"], "steps": 0,
            "u": mv(inp["u"]), "delta": mv(inp["delta"]), "z": mv(inp.get("z")), "B": mv(inp["B"]),
            "C": mv(inp["C"]), "A": inp["A"], "D": inp.get("D"), "delta_bias": inp.get("delta_bias"),
            "h0": inp.get("h0")}


def decode_as_sequences(inp, rows):
    """Rearrange a decode input ([T, B, D] / [T, B, N]) into forward problems over its steps.

    Returns one forward input dict of shape (1, 1, T, N) per listed flat row
    b*D + d: the row's T decode steps become a length-T sequence.  T decode
    steps carrying the state equal the forward over those T steps (an oracle
    pin), so the oracle can check sampled rows of a full-size decode run.
    """
    T = inp["steps"]
    Bsz, Dm, _, N = inp["shape"]
    out = []
    for r in rows:
        b, d = divmod(r, Dm)
        case = {"shape": (1, 1, T, N), "in_dtype": inp["in_dtype"], "steps": 0,
                "u": np.ascontiguousarray(inp["u"][:, b, d]).reshape(1, 1, T),
                "delta": np.ascontiguousarray(inp["delta"][:, b, d]).reshape(1, 1, T),
                "z": None if inp.get("z") is None else np.ascontiguousarray(inp["z"][:, b, d]).reshape(1, 1, T),
                "B": np.ascontiguousarray(inp["B"][:, b, :].T).reshape(1, N, T),
                "C": np.ascontiguousarray(inp["C"][:, b, :].T).reshape(1, N, T),
                "A": np.ascontiguousarray(inp["A"][d:d + 1]),
                "D": None if inp.get("D") is None else np.ascontiguousarray(inp["D"][d:d + 1]),
                "delta_bias": None if inp.get("delta_bias") is None else
                np.ascontiguousarray(inp["delta_bias"][d:d + 1]),
                "h0": None if inp.get("h0") is None else np.ascontiguousarray(inp["h0"][b, d]).reshape(1, 1, N)}
        out.append(case)
    return out


# Gradients (selscan_bwd): |g - ref| <= a·max|ref| + r·|ref| per tensor, (a, r) by the type the gradient
# is written in.  fp32 gradients carry the fp32 rounding of sums over up to B·L·N terms (relative 1e-5
# at these sizes) and the approximate exp2 of the recomputed states; bf16 gradients (du, dδ, dz of bf16
# inputs) are rounded to 8 significant bits (relative 2^-9) on top.
GRAD_TOL = {"f32": (1e-4, 1e-4), "bf16": (1e-3, 4e-3)}


def gpu_bwd(inp, cot, delta_softplus=True, workspace=None, want_dh0=True, ckpt=None):
    """selscan_bwd on an input dict and a cotangent dict; float64 numpy gradients keyed like
    oracle.selscan_bwd."""
    import torch

    import selective_state_space_152_b300 as ss

    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    go = to_dev(cot["dout"])
    gh = to_dev(cot.get("dh_last"))
    g = ss.selscan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], go, D=t["D"], z=t["z"],
                       delta_bias=t["delta_bias"], delta_softplus=delta_softplus, h0=t["h0"], dh_last=gh,
                       workspace=workspace, want_dh0=want_dh0, ckpt=ckpt)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.float().cpu().numpy().astype(np.float64)) for k, v in g.items()}


def oracle_cotangent(cot):
    """The cotangents as float64 arrays for oracle.selscan_bwd (bf16 bit patterns widened exactly)."""
    import seeded_inputs as si

    go = cot["dout"]
    go = si.bf16_bits_to_f32(go) if go.dtype == np.uint16 else go
    gh = cot.get("dh_last")
    return go.astype(np.float64), (None if gh is None else gh.astype(np.float64))


def check_grads(got, ref, in_dtype, what=""):
    """Compare every gradient the oracle returns (keys whose oracle value is None are skipped); returns
    the worst error of each tensor as a fraction of its bound."""
    worst = {}
    for key, r in ref.items():
        if r is None:
            continue
        g = got[key]
        assert g is not None, f"{what} grad {key} missing"
        assert g.shape == r.shape, f"{what} grad {key} shape {g.shape} != {r.shape}"
        assert np.isfinite(r).all(), f"{what} grad {key}: the oracle's gradient is not finite (bad test input)"
        kind = in_dtype if key in ("u", "delta", "z") else "f32"
        a, rr = GRAD_TOL[kind]
        scale = float(np.abs(r).max()) if r.size else 0.0
        err = np.abs(g - r)
        bound = a * scale + rr * np.abs(r)
        bad = ~(err <= bound)
        if bad.any():
            i = int(np.argmax(np.where(bad, err - bound, -np.inf)))
            raise AssertionError(f"{what} grad {key}: {int(bad.sum())} of {bad.size} outside tolerance; worst at flat "
                                 f"{i}: got {g.flat[i]!r} ref {r.flat[i]!r} (bound {bound.flat[i]:.3e}, scale "
                                 f"{scale:.3e})")
        worst[key] = float((err / np.maximum(bound, 1e-300)).max()) if r.size else 0.0
    return worst
