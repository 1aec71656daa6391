"""Failure detection on the GPU without a fault: a bounded wait that runs out.

The channel kernel's, the streamed decode kernel's and the tensor-core SSD kernels' waits
on their mbarriers are bounded; a wait that runs out records an error code in the library's device error word and
the kernel returns (no trap, no hang). Here the staging thread is told to issue no copies
(SSM_B300_FAULT_INJECT=skip_loads) and the wait limit is cut to 2e5 cycles (about 0.1
ms), so every wait for data runs out. The tests check that the call returns, that
ssm_device_error reports a "data never arrived" code, and that a following normal call
on the same context is correct.
"""
import os

import pytest
import torch

import oracle
from parity import TOL_BF16, check
from selective_state_space_141_b300 import inputs, ssm

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _fwd(d):
    y, last = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                     delta_bias=d["delta_bias"], y_dtype=torch.float32, use_workspace=False)
    return y, last


def test_wait_runs_out_and_context_recovers(monkeypatch):
    d = inputs.random_fwd(2, 200, 256, 16, dtype=torch.bfloat16, device=DEV, seed=71)  # channel-kernel shape
    assert ssm.device_error() == 0
    monkeypatch.setenv("SSM_B300_FAULT_INJECT", "skip_loads")
    monkeypatch.setenv("SSM_B300_WAIT_LIMIT_CYCLES", "200000")
    _fwd(d)
    code = ssm.device_error()  # synchronises; the kernel returned on its own
    assert code in (1, 3), f"expected a 'data never arrived' code (1 or 3), got {code}"
    monkeypatch.delenv("SSM_B300_FAULT_INJECT")
    monkeypatch.delenv("SSM_B300_WAIT_LIMIT_CYCLES")
    y, last = _fwd(d)
    assert ssm.device_error() == 0
    yr, sr = oracle.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                       delta_bias=d["delta_bias"])
    check(y, yr, TOL_BF16, False, "y after recovery")
    check(last, sr, TOL_BF16, False, "last_state after recovery")


def test_short_limit_alone_does_not_fire(monkeypatch):
    """A short limit is still far above a healthy wait: no error without the fault."""
    d = inputs.random_fwd(1, 300, 128, 16, dtype=torch.bfloat16, device=DEV, seed=72)
    monkeypatch.setenv("SSM_B300_WAIT_LIMIT_CYCLES", "2000000")
    _fwd(d)
    assert ssm.device_error() == 0


def test_decode_wait_runs_out_and_context_recovers(monkeypatch):
    """The streamed decode kernel's waits: with no copies issued every consumer wait runs
    out, the step returns with a 'data never arrived' code, and a following normal step
    on the same context matches the oracle."""
    w = inputs.DecodeWorkload("t", 4, 256, 16, 1, torch.bfloat16, 73)  # streamed-kernel shape
    d = inputs.decode_inputs(w, DEV)
    g = torch.Generator(device="cpu").manual_seed(74)
    s0 = torch.randn(4, 256, 16, generator=g).to(DEV)
    args = (d["x"][0], d["delta"][0], d["A"], d["B"][0], d["C"][0])
    assert ssm.device_error() == 0
    monkeypatch.setenv("SSM_B300_FAULT_INJECT", "skip_loads")
    monkeypatch.setenv("SSM_B300_WAIT_LIMIT_CYCLES", "200000")
    state = s0.clone()
    ssm.state_update(state, *args, D=d["D"], z=d["z"][0])
    assert ssm.device_error() == 1
    monkeypatch.delenv("SSM_B300_FAULT_INJECT")
    monkeypatch.delenv("SSM_B300_WAIT_LIMIT_CYCLES")
    state = s0.clone()
    y = ssm.state_update(state, *args, D=d["D"], z=d["z"][0])
    assert ssm.device_error() == 0
    yr, sr = oracle.state_update(s0, *args, D=d["D"], z=d["z"][0])
    check(y, yr, TOL_BF16, True, "y after recovery")
    check(state, sr, TOL_BF16, False, "state after recovery")


def test_ssd_waits_run_out_and_context_recovers(monkeypatch):
    """The tensor-core SSD kernels' waits (state walk and read-out, P = 128): with no copies
    issued, the workers' waits for data run out, every role leaves through the shared
    abort flag (the TMEM it holds released), the call returns with an error code, and a
    following normal call on the same context matches the oracle."""
    d = inputs.ssd_inputs(inputs.SsdWorkload("t", 1, 200, 3, 128, 128, 1, 75), DEV)
    kw = dict(D=d["D"], dt_bias=d["dt_bias"], dt_softplus=d["dt_softplus"], y_dtype=torch.float32)
    assert ssm.device_error() == 0
    monkeypatch.setenv("SSM_B300_FAULT_INJECT", "skip_loads")
    monkeypatch.setenv("SSM_B300_WAIT_LIMIT_CYCLES", "200000")
    ssm.ssd_fwd(d["x"], d["delta"], d["A"], d["B"], d["C"], **kw)
    code = ssm.device_error()
    assert code in (1, 4), f"expected a wait-ran-out code, got {code}"
    monkeypatch.delenv("SSM_B300_FAULT_INJECT")
    monkeypatch.delenv("SSM_B300_WAIT_LIMIT_CYCLES")
    y, last = ssm.ssd_fwd(d["x"], d["delta"], d["A"], d["B"], d["C"], **kw)
    assert ssm.device_error() == 0
    yr, lr = oracle.ssd_fwd(d["x"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], dt_bias=d["dt_bias"],
                            dt_softplus=d["dt_softplus"])
    check(y, yr, TOL_BF16, False, "y after recovery")
    check(last, lr, TOL_BF16, False, "last_state after recovery")
