"""selscan_fwd_noalloc: the forward entry point that allocates no device memory.

Some callers may not allocate memory while they run: code that owns a fixed
memory budget, or that runs inside a framework which forbids allocation during
execution.  For them the library offers selscan_fwd_noalloc.  It keeps the
time-block scratch of problems with few rows in one fixed device buffer of the
library, instead of taking it from the CUDA memory pool as selscan_fwd does.

These tests call it through the C ABI (the ctypes binding) on two calls in a
row, with different shapes and inputs and with time blocks forced so that the
fixed buffer is used, the second call writing h_last over h0.  Each result is
checked against the fp64 oracle on the same inputs, within the parity
tolerances of the other GPU tests, for the row-sequential kernel and for the
older sequential kernel that serves rows the tensor copies cannot stage.  They
also check that a problem needing more than the buffer holds is rejected
before anything runs.  This file is named so that pytest collects it last.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import check_h, check_out, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_152_b300 as mod

    mod.load_library()  # fails loudly if the library was not built
    return mod


def _noalloc(ss, inp, nblocks, monkeypatch, inplace=False):
    """selscan_fwd_noalloc on an input dict, with `nblocks` time blocks forced so that the fixed buffer
    is used; float64 numpy (out, h_last).  With `inplace`, h_last is written over h0."""
    import torch

    monkeypatch.setenv("SELSCAN_TBLOCKS", str(nblocks))
    t = {k: to_dev(inp.get(k)) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    Bsz, Dm, L, N = inp["shape"]
    out = torch.full((Bsz, Dm, L), float("nan"), device="cuda")
    hl = t["h0"] if inplace else torch.full((Bsz, Dm, N), float("nan"), device="cuda")
    ss.selscan_fwd_noalloc(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                           delta_bias=t["delta_bias"], h0=t["h0"], out=out, h_last=hl)
    torch.cuda.synchronize()
    f = lambda x: x.cpu().numpy().astype(np.float64)  # noqa: E731
    return f(out), f(hl)


@pytest.mark.parametrize("kern", ["rows", "seq"])
def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(ss, kern, monkeypatch):
    monkeypatch.setenv("SELSCAN_KERNEL", kern)
    # First call: bf16, 16 states, h0 and gate, 4 time blocks.
    a = si.random_case(71, 1, 40, 4096, 16, in_dtype="bf16")
    out, hl = _noalloc(ss, a, 4, monkeypatch)
    ref, href = oracle.selscan_fwd(a)
    check_out(out, ref, "bf16", what="noalloc call 1 out")
    check_h(hl, href, what="noalloc call 1 h_last")
    # Second call right after, on another shape and dtype with more blocks and h_last written over h0:
    # nothing the first call left in the shared buffer may show up in the result.
    b = si.random_case(72, 2, 9, 3000, 12, in_dtype="f32")
    ref, href = oracle.selscan_fwd(b)
    out, hl = _noalloc(ss, b, 5, monkeypatch, inplace=True)
    check_out(out, ref, "f32", what="noalloc call 2 out")
    check_h(hl, href, what="noalloc call 2 h_last (in place)")


def test_noalloc_rejects_a_problem_beyond_its_buffer(ss, monkeypatch):
    import torch

    # 4000 rows x 20 blocks x (2·16 + 1) floats ≈ 10.3 MiB of summaries and start states: more than
    # the 8 MiB buffer.  The call must fail before enqueueing anything.
    Bsz, Dm, L, N = 1, 4000, 10240, 16
    monkeypatch.setenv("SELSCAN_TBLOCKS", "20")
    u = torch.zeros((Bsz, Dm, L), device="cuda", dtype=torch.bfloat16)
    B = torch.zeros((Bsz, N, L), device="cuda", dtype=torch.bfloat16)
    A = -torch.ones((Dm, N), device="cuda")
    out = torch.full((Bsz, Dm, L), 7.0, device="cuda")
    with pytest.raises(ss.SelscanError) as ei:
        ss.selscan_fwd_noalloc(u, u, A, B, B, out=out)
    assert ei.value.status == 8  # SELSCAN_ERR_SCRATCH
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "a rejected call must not write its output"
