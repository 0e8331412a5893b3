"""Failure detection: a bounded device-side wait that runs out is reported, and
the context stays usable.

The ordered relay of the deterministic mode (D_qk up to 128 other than 128)
makes each key tile wait for its turn on a query tile ("SDPA Backward (SM120)",
section "Deterministic vs. non-deterministic dQ": the relay can stall if its
ordering assumption fails). Here the host skews every expected turn by one, so
the first key tile of each query tile waits for a turn that no tile releases
(no fault, no trap: a counter that never reaches the value). With a 20 ms
limit the wait runs out, the kernel reports SDPA_ERR_TIMEOUT through the status
word, and it still completes. A normal call afterwards matches the oracle and
reports no error.
"""
import pytest
import torch

import workloads
from harness import assert_close, gpu_backward, make_case, oracle_backward, to_device

pytestmark = pytest.mark.gpu

W = workloads.Workload
RELAY = W("relay_timeout", 1, 2, 2, 256, 256, 64, 64, causal=True, deterministic=True, seed=71)


def test_relay_wait_runs_out_and_is_reported():
    import attention_backward_sdpa_gb300 as pkg
    case = make_case(RELAY)
    d = to_device(case)
    pkg.debug_relay(wait_limit_ns=20_000_000, turn_skew=1)
    try:
        with pytest.raises(pkg.SdpaError) as err:
            gpu_backward(case, d)  # checks the device status after the call
        assert err.value.code == 6  # SDPA_ERR_TIMEOUT
    finally:
        pkg.debug_relay(0, 0)
    # The status word was cleared by the check; the context is usable.
    pkg.check_device_status()
    dq, dk, dv = gpu_backward(case, d)
    torch.cuda.synchronize()
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), oracle_backward(case)):
        assert_close(name, g.double().cpu().numpy(), r)
