"""A bounded wait of the forward kernels made to run out (selscan_probe_wait_timeout): the waits give up,
the device status word records it, a reset clears it, and the context stays usable for a forward call.
The phase that never completes expects bytes from a copy that is never issued, so nothing is in flight
when the waits end and no GPU fault is involved."""
from __future__ import annotations

import time

import pytest

import oracle
import seeded_inputs as si
from gpu_util import check_out, gpu_fwd

pytestmark = pytest.mark.gpu


def test_wait_gives_up_and_reports_it():
    import selective_state_space_152_b300 as ss

    ss.selscan_device_status(reset=True)
    assert ss.selscan_device_status() == 0
    t0 = time.perf_counter()
    completed = ss.selscan_probe_wait_timeout(4096)
    elapsed = time.perf_counter() - t0
    assert completed == 0                      # no wait saw the phase complete
    assert ss.selscan_device_status() == 1     # ... and the kernel said so
    assert ss.selscan_device_status(reset=True) == 1
    assert ss.selscan_device_status() == 0     # the reset cleared the word
    assert elapsed < 30.0
    # The context is still usable: a forward call afterwards matches the oracle and leaves the word at 0.
    inp = si.random_case(61, 2, 24, 96, 16, in_dtype="bf16")
    got, _ = gpu_fwd(inp)
    ref, _ = oracle.selscan_fwd(inp)
    check_out(got, ref, "bf16")
    assert ss.selscan_device_status() == 0


def test_wait_probe_rejects_bad_arguments():
    import selective_state_space_152_b300 as ss

    for polls in (0, -1, (1 << 20) + 1):
        with pytest.raises(ss.SelscanError) as e:
            ss.selscan_probe_wait_timeout(polls)
        assert e.value.status == 2  # SELSCAN_ERR_SHAPE
