"""Parity of the backward (selscan_bwd) with the fp64 oracle's gradients, element by element.

The oracle's gradients are pinned against central finite differences of its forward and against the
adjoint of the materialised causal matrix (tests/oracle_pins.py).  Every case here runs the CUDA
kernel through the C ABI and compares every gradient tensor: du, dδ, dz, dA, dB, dC, dD, dΔ_bias, dh0.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import check_grads, gpu_bwd, oracle_cotangent, to_dev

pytestmark = pytest.mark.gpu

# (batch, dim, seqlen, dstate, in_dtype, dout_dtype, options)
CASES = [
    (2, 40, 100, 16, "f32", "f32", {}),                      # ragged chunk and ragged CTA, every input
    (2, 64, 128, 16, "bf16", "bf16", {}),                    # whole chunks, vector loads and stores
    (1, 37, 33, 12, "bf16", "f32", {}),                      # N not a multiple of 4, odd L
    (3, 33, 47, 1, "f32", "f32", {}),                        # one state
    (1, 8, 1, 4, "f32", "f32", {}),                          # one step
    (1, 8, 16, 8, "f32", "bf16", {}),                        # exactly one chunk
    (1, 70, 260, 16, "f32", "f32", {"has_z": False, "has_D": False, "has_bias": False, "has_h0": False,
                                    "has_dh_last": False}),  # no optional input
    (2, 48, 300, 16, "f32", "f32", {"softplus": False}),     # Δ = δ + Δ_bias (no softplus)
    (2, 96, 2048, 16, "bf16", "bf16", {}),                   # 128 chunks, three CTAs per batch entry
    (2, 20, 96, 3, "bf16", "bf16", {}),                      # checkpoints by the one-lane-per-row forward pass
    (1, 44, 200, 8, "f32", "bf16", {}),                      # checkpoints by the 8-state forward pass
]


def _case(i, B, Dm, L, N, dt, gdt, opt):
    inp = si.random_case(500 + i, B, Dm, L, N, in_dtype=dt, has_z=opt.get("has_z", True),
                         has_D=opt.get("has_D", True), has_bias=opt.get("has_bias", True),
                         has_h0=opt.get("has_h0", True))
    if not opt.get("softplus", True):
        # keep Δ = δ + Δ_bias positive without the softplus: δ = |N(0,1)|·0.1, Δ_bias = |Δ_bias|·0.01
        inp["delta_bias"] = (np.abs(inp["delta_bias"]) * np.float32(0.01)).astype(np.float32)
        d = inp["delta"]
        if dt == "bf16":
            f = si.bf16_bits_to_f32(d)
            inp["delta"] = si.f32_to_bf16_bits(np.abs(f) * np.float32(0.1))
        else:
            inp["delta"] = (np.abs(d) * np.float32(0.1)).astype(np.float32)
    cot = si.random_cotangents(900 + i, B, Dm, L, N, dout_dtype=gdt, has_dh_last=opt.get("has_dh_last", True))
    return inp, cot


@pytest.mark.parametrize("i", range(len(CASES)))
def test_bwd_matches_oracle(i):
    B, Dm, L, N, dt, gdt, opt = CASES[i]
    inp, cot = _case(i, B, Dm, L, N, dt, gdt, opt)
    sp = opt.get("softplus", True)
    got = gpu_bwd(inp, cot, delta_softplus=sp)
    go, gh = oracle_cotangent(cot)
    ref = oracle.selscan_bwd(inp, go, gh, delta_softplus=sp)
    check_grads(got, ref, dt, what=f"case {CASES[i][:6]}")


# (batch, dim, seqlen, dstate, in_dtype, dout_dtype, options) run in forced time blocks
TBLOCK_CASES = [
    (1, 40, 700, 16, "f32", "f32", {}),
    (2, 33, 517, 12, "bf16", "bf16", {}),
    (1, 64, 1000, 16, "f32", "f32", {"has_z": False, "has_h0": False}),
    (1, 24, 333, 4, "f32", "f32", {"softplus": False, "has_dh_last": False}),
]


@pytest.mark.parametrize("nblocks", ["2", "3", "7"])
@pytest.mark.parametrize("i", range(len(TBLOCK_CASES)))
def test_bwd_time_blocks(i, nblocks, monkeypatch):
    """Time blocks (summary, carry and block-wise passes) give every gradient of the one-block run, up to
    rounding: the carried start states and end gradients are exact in real arithmetic."""
    monkeypatch.setenv("SELSCAN_BWD_TBLOCKS", nblocks)
    B, Dm, L, N, dt, gdt, opt = TBLOCK_CASES[i]
    inp, cot = _case(700 + i, B, Dm, L, N, dt, gdt, opt)
    sp = opt.get("softplus", True)
    got = gpu_bwd(inp, cot, delta_softplus=sp)
    go, gh = oracle_cotangent(cot)
    ref = oracle.selscan_bwd(inp, go, gh, delta_softplus=sp)
    check_grads(got, ref, dt, what=f"time blocks {nblocks} case {TBLOCK_CASES[i][:6]}")


def test_bwd_absent_optional_inputs_give_gradient_at_zero():
    """dD and dΔ_bias are returned even without D and Δ_bias: they equal the gradients at D = 0 and
    Δ_bias = 0, which the oracle computes when given explicit zeros."""
    inp, cot = _case(40, 2, 40, 90, 16, "f32", "f32", {"has_D": False, "has_bias": False})
    got = gpu_bwd(inp, cot)
    z = dict(inp)
    z["D"] = np.zeros(40, np.float32)
    z["delta_bias"] = np.zeros(40, np.float32)
    go, gh = oracle_cotangent(cot)
    ref = oracle.selscan_bwd(z, go, gh)
    check_grads(got, ref, "f32", what="zero D / bias")


def test_bwd_workspace_given_or_pooled():
    import torch

    import selective_state_space_152_b300 as ss

    inp, cot = _case(41, 2, 40, 200, 16, "bf16", "f32", {})
    need = ss.selscan_bwd_workspace_size(2, 40, 200, 16)
    assert need == 2 * 40 * ((200 + 15) // 16) * 16 * 4
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    a = gpu_bwd(inp, cot, workspace=ws)
    b = gpu_bwd(inp, cot)
    go, gh = oracle_cotangent(cot)
    ref = oracle.selscan_bwd(inp, go, gh)
    check_grads(a, ref, "bf16", what="given workspace")
    check_grads(b, ref, "bf16", what="pooled workspace")
    for k in ("u", "delta", "z", "h0"):  # no atomics in these: identical bits
        assert np.array_equal(a[k], b[k]), k
    with pytest.raises(ss.SelscanError) as e:
        gpu_bwd(inp, cot, workspace=ws[: need - 16])
    assert e.value.status == 8  # SELSCAN_ERR_SCRATCH


def test_bwd_empty_sequence_and_no_rows():
    import torch

    import selective_state_space_152_b300 as ss

    inp, cot = _case(42, 2, 8, 0, 4, "f32", "f32", {})
    got = gpu_bwd(inp, cot)
    assert got["u"].shape == (2, 8, 0) and got["B"].shape == (2, 4, 0)
    assert np.all(got["A"] == 0) and np.all(got["D"] == 0) and np.all(got["delta_bias"] == 0)
    assert np.array_equal(got["h0"], cot["dh_last"].astype(np.float64))  # the state's gradient passes through
    inp, cot = _case(43, 2, 0, 50, 4, "f32", "f32", {})
    got = gpu_bwd(inp, cot)
    assert np.all(got["B"] == 0) and np.all(got["C"] == 0) and got["A"].shape == (0, 4)

def test_bwd_requires_dz_with_z():
    """The C ABI refuses a call with z but no dz (SELSCAN_ERR_NULL) and enqueues nothing."""
    import ctypes

    import torch

    import selective_state_space_152_b300 as ss

    inp, cot = _case(45, 1, 8, 32, 4, "f32", "f32", {})
    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A")}
    go = to_dev(cot["dout"])
    g = {k: torch.zeros_like(t[k], dtype=torch.float32) for k in ("u", "delta", "A", "B", "C")}
    lib = ss.load_library()
    shape = ss.SelscanShape(1, 8, 32, 4, 0, 0)
    p = lambda x: None if x is None else x.data_ptr()  # noqa: E731
    st = lib.selscan_bwd(ctypes.byref(shape), p(t["u"]), p(t["delta"]), p(t["A"]), p(t["B"]), p(t["C"]), None,
                         p(t["z"]), None, 1, None, p(go), None, p(g["u"]), p(g["delta"]), None, p(g["A"]),
                         p(g["B"]), p(g["C"]), None, None, None, None, 0, None)
    assert st == 1  # SELSCAN_ERR_NULL
    assert ss.selscan_last_launch_count() == 0


def test_bwd_launch_count(monkeypatch):
    """The checkpointing forward pass first when the row-sequential kernel can stage the rows in one pass
    (else the backward forms its checkpoints itself), then one kernel for one time block and three
    (summary, carry, block-wise backward) for several."""
    import selective_state_space_152_b300 as ss

    inp, cot = _case(44, 1, 32, 64, 16, "f32", "f32", {})  # whole 16-byte rows: the pass applies
    ragged, rcot = _case(45, 1, 32, 66, 16, "f32", "f32", {})  # 66 fp32 steps: rows the copies cannot stage
    for blocks, own in (("1", 1), ("2", 3)):
        monkeypatch.setenv("SELSCAN_BWD_TBLOCKS", blocks)
        gpu_bwd(inp, cot)
        assert ss.selscan_last_launch_count() == 1 + own
        gpu_bwd(ragged, rcot)
        assert ss.selscan_last_launch_count() == own


@pytest.mark.parametrize("name", ["mamba130m_layer", "width_2p8b", "long_seq_65k"])
def test_bwd_workload_full(name):
    """Every gradient of a full-size workload against the oracle on all host cores."""
    w = si.WORKLOADS[name]
    inp = si.make_inputs(w)
    B, Dm, L, N = inp["shape"]
    cot = si.random_cotangents(77, B, Dm, L, N, dout_dtype="bf16")
    got = gpu_bwd(inp, cot)
    go, gh = oracle_cotangent(cot)
    ref = oracle.selscan_bwd(inp, go, gh)
    check_grads(got, ref, w.in_dtype, what=name)


def _truncated(inp, steps):
    """The input dict cut to its first `steps` steps (the forward oracle's state after them is h_last)."""
    out = dict(inp)
    for k in ("u", "delta", "z", "B", "C"):
        if out.get(k) is not None:
            out[k] = np.ascontiguousarray(out[k][..., :steps])
    B, Dm, _, N = inp["shape"]
    out["shape"] = (B, Dm, steps, N)
    return out


# (batch, dim, seqlen, dstate, in_dtype, forward time blocks)
CKPT_CASES = [(2, 40, 200, 16, "bf16", None), (1, 24, 100, 16, "f32", "3"), (2, 33, 96, 4, "f32", None),
              (1, 20, 136, 8, "bf16", "2")]


@pytest.mark.parametrize("i", range(len(CKPT_CASES)))
def test_fwd_ckpt_keeps_the_oracle_states(i, monkeypatch):
    """selscan_fwd_ckpt's checkpoint c is the state after the first 16·c steps (the oracle's h_last of the
    sequence cut there), in one pass and in forced time blocks; its out and h_last are selscan_fwd's."""
    import torch

    import selective_state_space_152_b300 as ss
    from gpu_util import check_h, check_out

    B, Dm, L, N, dt, tb = CKPT_CASES[i]
    if tb:
        monkeypatch.setenv("SELSCAN_TBLOCKS", tb)
    inp = si.random_case(800 + i, B, Dm, L, N, in_dtype=dt)
    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    out, hl, ck = ss.selscan_fwd_ckpt(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                                      delta_bias=t["delta_bias"], h0=t["h0"], return_h_last=True)
    torch.cuda.synchronize()
    assert ck.shape == (B, Dm, (L + 15) // 16, 16)
    ref, href = oracle.selscan_fwd(inp)
    check_out(out.cpu().numpy().astype(np.float64), ref, dt, what="fwd_ckpt out")
    check_h(hl.cpu().numpy().astype(np.float64), href, what="fwd_ckpt h_last")
    ckh = ck.cpu().numpy().astype(np.float64)
    assert np.array_equal(ckh[:, :, 0, :N], inp["h0"].astype(np.float64))  # before step 0: h0 itself
    for c in sorted({1, (L // 16) // 2, (L - 1) // 16}):
        if c < 1:
            continue
        _, hc = oracle.selscan_fwd(_truncated(inp, 16 * c))
        check_h(ckh[:, :, c, :N], hc, what=f"checkpoint {c}")


def _check_fwd_ckpt(inp, dt, chunks, what):
    """selscan_fwd_ckpt on inp: out and h_last against the oracle, and checkpoint c (c in chunks) against
    the oracle's state after the first 16·c steps."""
    import torch

    import selective_state_space_152_b300 as ss
    from gpu_util import check_h, check_out

    N = inp["shape"][3]
    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    out, hl, ck = ss.selscan_fwd_ckpt(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                                      delta_bias=t["delta_bias"], h0=t["h0"], return_h_last=True)
    torch.cuda.synchronize()
    ref, href = oracle.selscan_fwd(inp)
    check_out(out.cpu().numpy().astype(np.float64), ref, dt, what=f"{what} out")
    check_h(hl.cpu().numpy().astype(np.float64), href, what=f"{what} h_last")
    ckh = ck.cpu().numpy().astype(np.float64)
    for c in chunks:
        _, hc = oracle.selscan_fwd(_truncated(inp, 16 * c))
        check_h(ckh[:, :, c, :N], hc, what=f"{what} checkpoint {c}")


@pytest.mark.parametrize("spl", ["4", "8"])
def test_fwd_ckpt_both_lane_geometries(spl, monkeypatch):
    """The checkpointing forward with four and with eight states per lane (its two 16-state
    instantiations), over a ragged last chunk and enough rows for several CTAs."""
    monkeypatch.setenv("SELSCAN_ROWS_SPL", spl)
    inp = si.random_case(830 + int(spl), 2, 200, 296, 16, in_dtype="bf16")  # 296 = 9·32 + 8: a ragged last chunk
    _check_fwd_ckpt(inp, "bf16", [1, 9, 18], f"spl {spl}")


def test_fwd_ckpt_workload_full():
    """The checkpointing forward on the full 130M-like layer: every output and the final state against the
    oracle, and the checkpoints after 16, 1024 and 2032 steps."""
    w = si.WORKLOADS["mamba130m_layer"]
    _check_fwd_ckpt(si.make_inputs(w), w.in_dtype, [1, 64, 127], "mamba130m_layer")


@pytest.mark.parametrize("bwd_blocks", ["1", "3"])
@pytest.mark.parametrize("i", range(len(CKPT_CASES)))
def test_bwd_from_forward_checkpoints(i, bwd_blocks, monkeypatch):
    """selscan_bwd_ckpt from selscan_fwd_ckpt's checkpoints gives every gradient of the oracle, in one
    time block and in three (the carries then run without the backward's own forward pass)."""
    import selective_state_space_152_b300 as ss

    B, Dm, L, N, dt, tb = CKPT_CASES[i]
    if tb:
        monkeypatch.setenv("SELSCAN_TBLOCKS", tb)
    monkeypatch.setenv("SELSCAN_BWD_TBLOCKS", bwd_blocks)
    inp = si.random_case(820 + i, B, Dm, L, N, in_dtype=dt)
    cot = si.random_cotangents(840 + i, B, Dm, L, N, dout_dtype=dt)
    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    _, _, ck = ss.selscan_fwd_ckpt(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                                   delta_bias=t["delta_bias"], h0=t["h0"])
    got = gpu_bwd(inp, cot, ckpt=ck)
    go, gh = oracle_cotangent(cot)
    ref = oracle.selscan_bwd(inp, go, gh)
    check_grads(got, ref, dt, what=f"bwd from checkpoints {CKPT_CASES[i][:5]}")


def test_fwd_ckpt_needs_staged_rows():
    """Rows the tensor copies cannot stage (L not a multiple of 8 in bf16) are refused: no checkpoints."""
    import selective_state_space_152_b300 as ss

    inp = si.random_case(850, 1, 8, 37, 16, in_dtype="bf16")
    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    with pytest.raises(ss.SelscanError) as e:
        ss.selscan_fwd_ckpt(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"], delta_bias=t["delta_bias"])
    assert e.value.status == 4  # SELSCAN_ERR_UNSUPPORTED
