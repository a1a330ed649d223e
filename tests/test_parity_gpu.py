"""libselscan on the GPU against the fp64 oracle, element by element on the same seeded inputs.

Tolerances (written here, derived from the required accuracy of the scan):
  fp32 inputs:            |out - ref| <= 1e-4 + 1e-4·|ref|
  bf16 inputs, fp32 state: |out - ref| <= 2e-3 + 2e-3·|ref|
  h_last:                 |h - ref| <= 1e-4 · max_n |ref| of the channel (relative, in the max norm
                          of each channel's state vector)
Every case is compared in full, every element of every output, including the
full-size workloads in the launch configuration that bench.py times (the
oracle runs on all host cores) and all 64 steps of the decode workload.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import (check_h, check_out, decode_as_forward, gpu_fwd, gpu_fwd_conv, gpu_fwd_ex, sample_rows,
                      to_dev)

pytestmark = pytest.mark.gpu

# The forward kernels: "rows" is the row-sequential kernel with the warp-specialised copy pipeline
# (the library's choice wherever every input row is 16-byte aligned; elsewhere these cases fall back to
# "seq"); "seq" is the older sequential kernel (rows spread over lanes, in-CTA staging), "chunk" splits
# each row's sequence over lanes and joins them with a scan.  The tests force each one through the
# SELSCAN_KERNEL override.  "chunk_direct" is the chunked kernel with its tensor-copy staging turned off
# (SELSCAN_STAGING=0), so that its direct-load path is also covered on aligned inputs.
KERNELS = ["rows", "seq", "chunk", "chunk_direct"]


@pytest.fixture(params=KERNELS)
def kernel(request, monkeypatch):
    monkeypatch.setenv("SELSCAN_KERNEL", {"rows": "rows", "seq": "seq"}.get(request.param, "chunk"))
    if request.param == "chunk_direct":
        monkeypatch.setenv("SELSCAN_STAGING", "0")
    else:
        monkeypatch.delenv("SELSCAN_STAGING", raising=False)
    return request.param


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_152_b300 as ss

    ss.load_library()  # fails loudly if the library was not built


def test_tiny_fp32_workload_full(kernel):
    w = si.WORKLOADS["tiny_fp32"]
    inp = si.make_inputs(w)
    ref, href = oracle.selscan_fwd(inp)
    got, hl = gpu_fwd(inp)
    check_out(got, ref, "f32")
    check_h(hl, href)


SMALL = [
    # (seed, B, D, L, N, dtype, z, D, bias, h0, softplus)
    (1, 1, 1, 1, 1, "f32", True, True, True, True, True),
    (2, 2, 3, 7, 3, "f32", True, True, True, True, True),
    (3, 1, 5, 33, 4, "f32", False, True, True, False, True),
    (4, 2, 9, 255, 5, "f32", True, False, False, True, True),
    (5, 1, 4, 512, 8, "f32", True, True, True, True, False),
    (6, 2, 6, 513, 16, "f32", True, True, True, True, True),
    (7, 3, 7, 1000, 16, "bf16", True, True, True, True, True),
    (8, 1, 3, 1537, 2, "bf16", False, False, True, True, True),
    (9, 2, 5, 2048, 16, "bf16", True, True, True, False, True),
    (10, 1, 2, 4099, 12, "f32", True, True, True, True, True),
]


@pytest.mark.parametrize("case", SMALL, ids=[f"s{c[0]}_B{c[1]}D{c[2]}L{c[3]}N{c[4]}_{c[5]}" for c in SMALL])
def test_small_shapes_full(case, kernel):
    seed, Bsz, Dm, L, N, dt, hz, hD, hb, hh, sp = case
    inp = si.random_case(seed, Bsz, Dm, L, N, in_dtype=dt, has_z=hz, has_D=hD, has_bias=hb, has_h0=hh)
    if not sp:  # without softplus Δ = δ + bias must stay positive, else Ā > 1 and the state overflows
        inp["delta_bias"] = None
        d = np.abs(si.bf16_bits_to_f32(inp["delta"]) if dt == "bf16" else inp["delta"]) * 0.05
        inp["delta"] = si.f32_to_bf16_bits(d) if dt == "bf16" else d.astype(np.float32)
    ref, href = oracle.selscan_fwd(inp, delta_softplus=sp)
    got, hl = gpu_fwd(inp, delta_softplus=sp)
    check_out(got, ref, dt)
    check_h(hl, href)


# Shapes for the chunked kernel's tensor-copy staging, forced onto 4, 8 and 16 lanes per channel
# (channel blocks of 32, 16 and 8 rows; chunks of 64, 128 and 256 steps).  They cover ragged last
# chunks, channel counts that leave part of the last block past `dim` (its rows read the next batch
# entry's rows, or zeros past the tensor), dstate below the tile's 4/8/16 states, and both dtypes.
STAGED = [
    (31, 2, 40, 1000, 16, "bf16"),
    (32, 3, 17, 264, 12, "bf16"),
    (33, 1, 8, 4096, 16, "bf16"),
    (34, 2, 24, 300, 5, "f32"),
    (35, 1, 33, 772, 16, "f32"),
    (36, 2, 16, 64, 3, "bf16"),
]


@pytest.mark.parametrize("lanes", ["4", "8", "16"])
@pytest.mark.parametrize("case", STAGED, ids=[f"s{c[0]}_B{c[1]}D{c[2]}L{c[3]}N{c[4]}_{c[5]}" for c in STAGED])
def test_chunked_staged_shapes(case, lanes, monkeypatch):
    monkeypatch.setenv("SELSCAN_KERNEL", "chunk")
    monkeypatch.setenv("SELSCAN_LANES", lanes)
    monkeypatch.delenv("SELSCAN_STAGING", raising=False)
    seed, Bsz, Dm, L, N, dt = case
    inp = si.random_case(seed, Bsz, Dm, L, N, in_dtype=dt)
    ref, href = oracle.selscan_fwd(inp)
    got, hl = gpu_fwd(inp)
    check_out(got, ref, dt)
    check_h(hl, href)


# The row-sequential kernel's geometry, forced: 4 or 8 states per lane (4 or 2 lanes per row), 1, 3
# or 15 consumer warps per CTA, 2 or 4 pipeline stages.  Lengths are whole 16-byte rows (so the kernel
# can stage them) but ragged against its 32-step chunks; channel counts leave the last CTA's rows partly
# past `dim`; dstate below the 4/8/16-state tile; both dtypes; with and without the gate.
ROWS_CASES = [
    (101, 2, 40, 1000, 16, "bf16", True),
    (102, 3, 17, 264, 12, "bf16", True),
    (103, 1, 8, 4096, 16, "bf16", False),
    (104, 2, 24, 300, 5, "f32", True),
    (105, 1, 33, 772, 16, "f32", True),
    (106, 2, 16, 64, 3, "bf16", True),
    (107, 1, 130, 96, 8, "f32", False),
    (108, 2, 70, 200, 4, "bf16", True),
]
ROWS_GEOM = [("4", "1", "2"), ("4", "3", "4"), ("8", "15", "3"), ("8", "2", "2"), ("4", "15", "2")]


@pytest.mark.parametrize("geom", ROWS_GEOM, ids=[f"spl{g[0]}_w{g[1]}_s{g[2]}" for g in ROWS_GEOM])
@pytest.mark.parametrize("case", ROWS_CASES, ids=[f"s{c[0]}_B{c[1]}D{c[2]}L{c[3]}N{c[4]}_{c[5]}" for c in ROWS_CASES])
def test_rows_kernel_geometry(case, geom, monkeypatch):
    monkeypatch.setenv("SELSCAN_KERNEL", "rows")
    monkeypatch.setenv("SELSCAN_ROWS_SPL", geom[0])
    monkeypatch.setenv("SELSCAN_ROWS_WARPS", geom[1])
    monkeypatch.setenv("SELSCAN_ROWS_STAGES", geom[2])
    seed, Bsz, Dm, L, N, dt, hz = case
    inp = si.random_case(seed, Bsz, Dm, L, N, in_dtype=dt, has_z=hz)
    ref, href = oracle.selscan_fwd(inp)
    got, hl = gpu_fwd(inp)
    check_out(got, ref, dt)
    check_h(hl, href)
    got16, _ = gpu_fwd(inp, out_dtype="bf16", h_last=False)
    check_out(got16, ref, dt, what="bf16 out", extra_rel=2.0 ** -8)


# Time blocks: the sequence is cut into blocks joined by a summary pass (each block's zero-start end
# state and ΣΔ) and a carry pass.  Forced block counts on ragged lengths, with and without h0, softplus
# on and off, fp32 and bf16, for the row-sequential kernel (lengths of whole 16-byte rows) and the older
# sequential kernel.
TBLOCKED = [
    (41, 2, 5, 1500, 16, "bf16", True, True),
    (42, 1, 3, 2049, 4, "f32", True, False),
    (43, 3, 4, 1100, 12, "f32", False, True),
    (44, 1, 40, 4096, 16, "bf16", True, True),
    (45, 2, 5, 1504, 16, "bf16", True, True),
    (46, 1, 3, 2048, 4, "f32", True, False),
    (47, 3, 4, 1104, 12, "f32", False, True),
    (48, 1, 20, 1000, 8, "bf16", True, True),
]


@pytest.mark.parametrize("kern", ["rows", "seq"])
@pytest.mark.parametrize("nblocks", ["2", "3", "7"])
@pytest.mark.parametrize("case", TBLOCKED, ids=[f"s{c[0]}_B{c[1]}D{c[2]}L{c[3]}N{c[4]}_{c[5]}" for c in TBLOCKED])
def test_time_blocked_sequential(case, nblocks, kern, monkeypatch):
    monkeypatch.setenv("SELSCAN_KERNEL", kern)
    monkeypatch.setenv("SELSCAN_TBLOCKS", nblocks)
    seed, Bsz, Dm, L, N, dt, hh, sp = case
    inp = si.random_case(seed, Bsz, Dm, L, N, in_dtype=dt, has_h0=hh)
    if not sp:  # keep Δ = δ + bias positive without softplus
        inp["delta_bias"] = None
        d = np.abs(si.bf16_bits_to_f32(inp["delta"]) if dt == "bf16" else inp["delta"]) * 0.05
        inp["delta"] = si.f32_to_bf16_bits(d) if dt == "bf16" else d.astype(np.float32)
    ref, href = oracle.selscan_fwd(inp, delta_softplus=sp)
    got, hl = gpu_fwd(inp, delta_softplus=sp)
    check_out(got, ref, dt)
    check_h(hl, href)


# selscan_fwd_ex: the reverse direction and the exact zero-order-hold input matrix, alone and
# together, in one pass and in time blocks, against the oracle run with the same options.
EX_CASES = [
    (51, 2, 5, 1000, 16, "bf16"),
    (52, 1, 3, 777, 4, "f32"),
    (53, 2, 6, 2049, 12, "f32"),
]


@pytest.mark.parametrize("opts", ["rev", "zoh", "rev_zoh", "none"])
@pytest.mark.parametrize("nblocks", ["1", "3"])
@pytest.mark.parametrize("case", EX_CASES, ids=[f"s{c[0]}_B{c[1]}D{c[2]}L{c[3]}N{c[4]}_{c[5]}" for c in EX_CASES])
def test_fwd_ex_options(case, nblocks, opts, monkeypatch):
    monkeypatch.setenv("SELSCAN_TBLOCKS", nblocks)
    rev, zoh = "rev" in opts, "zoh" in opts
    seed, Bsz, Dm, L, N, dt = case
    inp = si.random_case(seed, Bsz, Dm, L, N, in_dtype=dt)
    ref, href = oracle.selscan_fwd(inp, reverse=rev, zoh=zoh)
    got, hl = gpu_fwd_ex(inp, reverse=rev, zoh=zoh)
    check_out(got, ref, dt, what=f"fwd_ex {opts} out")
    check_h(hl, href, what=f"fwd_ex {opts} h_last")


@pytest.mark.parametrize("opts", ["rev", "zoh"])
def test_fwd_ex_long_sequence_sampled(opts):
    """The 65k-step workload (time blocks chosen by the library) in reverse and with exact ZOH."""
    w = si.WORKLOADS["long_seq_65k"]
    inp = si.make_inputs(w)
    Bsz, Dm, L, N = inp["shape"]
    got, hl = gpu_fwd_ex(inp, reverse=opts == "rev", zoh=opts == "zoh")
    rows = sample_rows(Bsz, Dm, 8, seed=7)
    ref, href = oracle.selscan_fwd(inp, rows=rows, reverse=opts == "rev", zoh=opts == "zoh")
    check_out(got.reshape(Bsz * Dm, L)[rows], ref, w.in_dtype, what=f"long {opts} out")
    check_h(hl.reshape(Bsz * Dm, N)[rows], href, what=f"long {opts} h_last")


# selscan_fwd_conv: the causal conv1d (width 4) + SiLU front computed in the kernel from x, against
# the oracle's conv front feeding its scan (u in fp64).
def _conv_params(seed, Dm, with_bias=True):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((Dm, 4)) * 0.5).astype(np.float32)
    cb = (rng.standard_normal(Dm) * 0.5).astype(np.float32) if with_bias else None
    return w, cb


CONV_CASES = [
    (61, 2, 5, 1000, 16, "bf16", True),
    (62, 1, 3, 777, 4, "f32", False),
    (63, 2, 6, 2049, 12, "f32", True),
]


@pytest.mark.parametrize("zoh", [False, True])
@pytest.mark.parametrize("nblocks", ["1", "3"])
@pytest.mark.parametrize("case", CONV_CASES, ids=[f"s{c[0]}_B{c[1]}D{c[2]}L{c[3]}N{c[4]}_{c[5]}" for c in CONV_CASES])
def test_fwd_conv_front(case, nblocks, zoh, monkeypatch):
    monkeypatch.setenv("SELSCAN_TBLOCKS", nblocks)
    seed, Bsz, Dm, L, N, dt, with_bias = case
    inp = si.random_case(seed, Bsz, Dm, L, N, in_dtype=dt)
    w, cb = _conv_params(seed, Dm, with_bias)
    u64 = oracle.conv_silu(inp["u"], w, cb, dt)
    ref, href = oracle.selscan_fwd(inp, u_f64=u64, zoh=zoh)
    got, hl = gpu_fwd_conv(inp, w, cb, zoh=zoh)
    check_out(got, ref, dt, what="fwd_conv out")
    check_h(hl, href, what="fwd_conv h_last")


def test_fwd_conv_long_sequence_sampled():
    """The 65k-step workload with the conv front (time blocks chosen by the library)."""
    w_ = si.WORKLOADS["long_seq_65k"]
    inp = si.make_inputs(w_)
    Bsz, Dm, L, N = inp["shape"]
    w, cb = _conv_params(64, Dm)
    got, hl = gpu_fwd_conv(inp, w, cb)
    assert Bsz == 1
    ch = np.array(sample_rows(Bsz, Dm, 8, seed=9))
    # The sampled channels as a problem of their own (batch 1, 8 channels) for the oracle.
    sub = dict(inp)
    for k in ("u", "delta", "z"):
        sub[k] = None if inp.get(k) is None else np.ascontiguousarray(np.asarray(inp[k])[:, ch])
    for k in ("A", "D", "delta_bias"):
        sub[k] = None if inp.get(k) is None else np.ascontiguousarray(np.asarray(inp[k])[ch])
    sub["h0"] = None if inp.get("h0") is None else np.ascontiguousarray(np.asarray(inp["h0"])[:, ch])
    sub["shape"] = (1, len(ch), L, N)
    u64 = oracle.conv_silu(sub["u"], w[ch], cb[ch], w_.in_dtype)
    ref, href = oracle.selscan_fwd(sub, u_f64=u64)
    check_out(got[:, ch], ref, w_.in_dtype, what="long conv out")
    check_h(hl[:, ch], href, what="long conv h_last")


@pytest.mark.parametrize("name", ["mamba130m_layer", "long_seq_65k", "width_2p8b"])
def test_workload_full(name):
    """Every element of the full-size workload, in the launch configuration the bench times, against
    the oracle on all host cores."""
    w = si.WORKLOADS[name]
    inp = si.make_inputs(w)
    got, hl = gpu_fwd(inp)
    ref, href = oracle.selscan_fwd(inp)
    check_out(got, ref, w.in_dtype, what=f"{name} out")
    check_h(hl, href, what=f"{name} h_last")


def test_bf16_output(kernel):
    inp = si.random_case(21, 2, 5, 700, 16, in_dtype="bf16")
    ref, _ = oracle.selscan_fwd(inp)
    got, _ = gpu_fwd(inp, out_dtype="bf16")
    # bf16 rounding of the output adds up to 2^-8 relative on top of the bf16-input tolerance
    check_out(got, ref, "bf16", extra_rel=2.0 ** -8)


def test_carry_across_calls(kernel):
    import torch

    import selective_state_space_152_b300 as ss

    inp = si.random_case(31, 2, 6, 1500, 16, in_dtype="f32")
    ref, href = oracle.selscan_fwd(inp)
    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    outs = []
    h = t["h0"].clone()
    for a, b in [(0, 1), (1, 700), (700, 1100), (1100, 1500)]:
        sl = {k: t[k][..., a:b].contiguous() for k in ("u", "delta", "z", "B", "C")}
        o, _ = ss.selscan_fwd(sl["u"], sl["delta"], t["A"], sl["B"], sl["C"], D=t["D"], z=sl["z"],
                              delta_bias=t["delta_bias"], h0=h, h_last=h)  # in-place carry: h_last aliases h0
        outs.append(o)
    torch.cuda.synchronize()
    got = torch.cat(outs, dim=-1).cpu().numpy().astype(np.float64)
    check_out(got, ref, "f32", what="chunked-call out")
    check_h(h.cpu().numpy().astype(np.float64), href, what="chunked-call h_last")


@pytest.mark.parametrize("kern", ["rows", "seq"])
@pytest.mark.parametrize("reverse", [False, True])
def test_inplace_carry_with_time_blocks(kern, reverse, monkeypatch):
    """h_last aliasing h0 (the in-place carry the header allows) while the sequence runs in time blocks:
    the first block's start state must be read before the last block's end state overwrites it."""
    import torch

    import selective_state_space_152_b300 as ss

    monkeypatch.setenv("SELSCAN_KERNEL", kern)
    monkeypatch.setenv("SELSCAN_TBLOCKS", "5")
    inp = si.random_case(121, 2, 40, 2048, 16, in_dtype="bf16")
    ref, href = oracle.selscan_fwd(inp, reverse=reverse)
    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    h = t["h0"].clone()
    out, _ = ss.selscan_fwd_ex(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                               delta_bias=t["delta_bias"], h0=h, h_last=h, reverse=reverse)
    torch.cuda.synchronize()
    check_out(out.cpu().numpy().astype(np.float64), ref, "bf16", what="in-place carry out")
    check_h(h.cpu().numpy().astype(np.float64), href, what="in-place carry h_last")


def test_decode_step_workload_full():
    """The decode workload as stated: all 64 steps over the full 256 x 5120 batch, carrying the state.
    Every output of every step and the final state are compared with the oracle.  T decode steps
    carrying the state equal the forward over those T steps (an oracle pin), so the oracle runs the
    whole decode as one threaded forward over [B, D, T]."""
    import torch

    import selective_state_space_152_b300 as ss

    w = si.WORKLOADS["decode_step"]
    inp = si.make_inputs(w)
    Bsz, Dm, _, N = inp["shape"]
    T = inp["steps"]
    assert T == 64
    dev = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    state = dev["h0"].clone()
    out = torch.empty((T, Bsz, Dm), device="cuda", dtype=torch.float32)
    for s in range(T):
        ss.selscan_step(dev["u"][s], dev["delta"][s], dev["A"], dev["B"][s], dev["C"][s], state, D=dev["D"],
                        z=dev["z"][s], delta_bias=dev["delta_bias"], out=out[s])
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)  # [T, B, D]
    hs = state.cpu().numpy().astype(np.float64)
    seq = decode_as_forward(inp)
    ref, href = oracle.selscan_fwd(seq)  # [B, D, T], [B, D, N]
    check_out(np.moveaxis(got, 0, -1), ref, "bf16", what="decode out (all steps)")
    check_h(hs, href, what="decode state after 64 steps")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_step_rows_spanning_batch_entries(dt):
    """The one-thread-per-row decode kernel with 300 channels: CTAs of 256 rows span two batch entries,
    whose B and C each CTA stages separately; 5 steps carrying the state, against the forward oracle."""
    import torch

    import selective_state_space_152_b300 as ss

    inp = si.random_case(131, 3, 300, 5, 16, in_dtype=dt)
    ref, href = oracle.selscan_fwd(inp)
    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    state = t["h0"].clone()
    outs = []
    for s in range(5):
        outs.append(ss.selscan_step(t["u"][..., s].contiguous(), t["delta"][..., s].contiguous(), t["A"],
                                    t["B"][..., s].contiguous(), t["C"][..., s].contiguous(), state, D=t["D"],
                                    z=t["z"][..., s].contiguous(), delta_bias=t["delta_bias"]))
    torch.cuda.synchronize()
    got = torch.stack(outs, dim=-1).cpu().numpy().astype(np.float64)
    check_out(got, ref, dt, what="decode rows spanning batch entries")
    check_h(state.cpu().numpy().astype(np.float64), href, what="decode state")


# (batch, dim, steps, in_dtype, has_z, out_dtype)
STEP_CASES = [(5, 100, 4, "bf16", True, "f32"), (5, 192, 4, "f32", False, "f32"), (1400, 256, 3, "bf16", True, "f32"),
              (3, 384, 3, "f32", False, "f32"), (2, 512, 3, "bf16", True, "bf16")]


@pytest.mark.parametrize("kern", ["quad", "row", "generic"])
@pytest.mark.parametrize("case", STEP_CASES, ids=lambda c: "x".join(map(str, c[:3])) + f"-{c[3]}-z{int(c[4])}-{c[5]}")
def test_step_kernels(case, kern, monkeypatch):
    """Each decode kernel, a few steps carrying the state, against the forward oracle (D = 100 puts a
    batch-entry boundary inside CTAs of the quad kernel, whose 64 rows then span two entries)."""
    import torch

    import selective_state_space_152_b300 as ss

    monkeypatch.setenv("SELSCAN_STEP", kern)
    Bsz, Dm, T, dt, has_z, odt = case
    inp = si.random_case(137 + Bsz, Bsz, Dm, T, 16, in_dtype=dt, has_z=has_z)
    ref, href = oracle.selscan_fwd(inp)
    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    state = t["h0"].clone()
    outs = []
    for s in range(T):
        z = None if t["z"] is None else t["z"][..., s].contiguous()
        outs.append(ss.selscan_step(t["u"][..., s].contiguous(), t["delta"][..., s].contiguous(), t["A"],
                                    t["B"][..., s].contiguous(), t["C"][..., s].contiguous(), state, D=t["D"],
                                    z=z, delta_bias=t["delta_bias"],
                                    out_dtype=torch.bfloat16 if odt == "bf16" else torch.float32))
        assert ss.selscan_last_launch_count() == 1
    torch.cuda.synchronize()
    got = torch.stack(outs, dim=-1).float().cpu().numpy().astype(np.float64)
    # a bf16 output adds its own rounding (2^-8 relative) to the bound
    check_out(got, ref, dt, what=f"decode {kern}", extra_rel=2.0 ** -8 if odt == "bf16" else 0.0)
    check_h(state.cpu().numpy().astype(np.float64), href, what=f"decode {kern} state")
    assert ss.selscan_device_status() == 0


def test_step_small_fp32_odd_dstate():
    import torch

    import selective_state_space_152_b300 as ss

    for N in (1, 3, 4, 6, 16):
        inp = si.random_case(40 + N, 3, 5, 9, N, in_dtype="f32")
        ref, href = oracle.selscan_fwd(inp)
        t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
        state = t["h0"].clone()
        outs = []
        for s in range(9):
            outs.append(ss.selscan_step(t["u"][..., s].contiguous(), t["delta"][..., s].contiguous(), t["A"],
                                        t["B"][..., s].contiguous(), t["C"][..., s].contiguous(), state, D=t["D"],
                                        z=t["z"][..., s].contiguous(), delta_bias=t["delta_bias"]))
        torch.cuda.synchronize()
        got = torch.stack(outs, dim=-1).cpu().numpy().astype(np.float64)
        check_out(got, ref, "f32", what=f"step N={N}")
        check_h(state.cpu().numpy().astype(np.float64), href, what=f"step state N={N}")


def test_causality_bitwise(kernel):
    inp = si.random_case(51, 1, 4, 1200, 16, in_dtype="bf16")
    base, _ = gpu_fwd(inp)
    for t0 in (0, 511, 512, 777, 1199):
        p = dict(inp)
        u = si.bf16_bits_to_f32(inp["u"]).copy()
        u[..., t0] += 1.0
        p["u"] = si.f32_to_bf16_bits(u)
        got, _ = gpu_fwd(p)
        assert np.array_equal(got[..., :t0], base[..., :t0]), f"outputs before t0={t0} changed"


def test_delta_to_zero_limit(kernel):
    inp = si.random_case(61, 1, 3, 300, 8, in_dtype="f32", has_z=False, has_h0=False)
    inp["delta_bias"] = np.full(3, -40.0, dtype=np.float32)
    got, hl = gpu_fwd(inp)
    want = np.asarray(inp["D"], np.float64)[None, :, None] * np.asarray(inp["u"], np.float64)
    check_out(got, want, "f32", what="Δ→0 gives D·u")
    assert np.max(np.abs(hl)) < 1e-12


def test_extreme_values(kernel):
    inp = si.random_case(71, 2, 3, 400, 16, in_dtype="f32")
    rng = np.random.default_rng(72)
    inp["delta"] = (rng.standard_normal(inp["delta"].shape) * 30).astype(np.float32)  # softplus far on both sides
    inp["z"] = (rng.standard_normal(inp["z"].shape) * 60).astype(np.float32)  # gate saturates and underflows
    ref, href = oracle.selscan_fwd(inp)
    got, hl = gpu_fwd(inp)
    check_out(got, ref, "f32")
    check_h(hl, href)


def test_empty_and_zero_length():
    import torch

    import selective_state_space_152_b300 as ss

    inp = si.random_case(81, 2, 3, 0, 4, in_dtype="f32")
    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    hl = torch.full_like(t["h0"], 7.0)
    ss.selscan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"], h0=t["h0"], h_last=hl)
    torch.cuda.synchronize()
    assert torch.equal(hl, t["h0"]), "L = 0 must pass h0 through"
    hl2 = torch.full_like(t["h0"], 7.0)
    ss.selscan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], h_last=hl2)
    torch.cuda.synchronize()
    assert torch.count_nonzero(hl2) == 0, "L = 0 without h0 gives a zero state"
    e = torch.empty(0, 3, 5, device="cuda")
    out, _ = ss.selscan_fwd(e, e, t["A"], torch.empty(0, 4, 5, device="cuda"), torch.empty(0, 4, 5, device="cuda"))
    assert out.shape == (0, 3, 5)


def test_host_side_rejections():
    import torch

    import selective_state_space_152_b300 as ss

    inp = si.random_case(91, 1, 4, 64, 4, in_dtype="f32")
    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    # output aliasing an input
    with pytest.raises(ss.SelscanError) as e:
        ss.selscan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], out=t["u"])
    assert e.value.status == 7
    # a tensor whose stated extent runs past the end of its allocation: a 4 MiB cudaMalloc (not the
    # caching allocator, whose segments can be larger), with u placed 40 bytes before its end while
    # the shape needs 1 KiB.  The call must be refused before any launch.
    import ctypes

    lib = ss.load_library()
    shape = ss.SelscanShape(1, 4, 64, 4, 0, 0)
    out = torch.empty(1, 4, 64, device="cuda")
    torch.cuda.synchronize()
    cudart = ctypes.CDLL("libcudart.so.13")
    buf = ctypes.c_void_p()
    assert cudart.cudaMalloc(ctypes.byref(buf), ctypes.c_size_t(4 << 20)) == 0
    try:
        tail = buf.value + (4 << 20) - 40
        st = lib.selscan_fwd(ctypes.byref(shape), tail, t["delta"].data_ptr(), t["A"].data_ptr(),
                             t["B"].data_ptr(), t["C"].data_ptr(), None, None, None, 1, None, out.data_ptr(), None,
                             None)
        assert st == 6, ss.selscan_status_string(st)
        # the same call with u at the start of the allocation is accepted
        assert cudart.cudaMemset(buf, 0, ctypes.c_size_t(4 << 20)) == 0
        st = lib.selscan_fwd(ctypes.byref(shape), buf.value, t["delta"].data_ptr(), t["A"].data_ptr(),
                             t["B"].data_ptr(), t["C"].data_ptr(), None, None, None, 1, None, out.data_ptr(), None,
                             None)
        assert st == 0
        torch.cuda.synchronize()
    finally:
        cudart.cudaFree(buf)
    # host memory that the device cannot reach
    host = np.zeros(4 * 64, np.float32)
    st = lib.selscan_fwd(ctypes.byref(shape), host.ctypes.data, t["delta"].data_ptr(), t["A"].data_ptr(),
                         t["B"].data_ptr(), t["C"].data_ptr(), None, None, None, 1, None, out.data_ptr(), None, None)
    assert st == 6
    torch.cuda.synchronize()
