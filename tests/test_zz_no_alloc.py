"""ssm_selective_scan_fwd_noalloc against ssm_selective_scan_fwd_ws, through the C ABI.

The no-allocation entry point is for callers that can only pass the buffers they own
(a fixed memory budget, a plugin interface given just inputs and outputs, a path where
an allocation must not stall or fail). It runs the same kernels as the entry point that
takes a caller-owned workspace, so the two results must be identical bit for bit; that
equality also shows the no-allocation call took the segmented schedule (the unsegmented
kernel associates the recurrence differently and would differ in the last bits). The
shape below takes the segmented schedule, so the built-in scratch array is really used;
two calls in a row with different inputs check that the second call does not depend on
what the first left in the array, and the first is also compared with the oracle on
sampled channels.
"""
import ctypes

import pytest
import torch

from parity import TOL_BF16
from selective_state_space_141_b300 import inputs, ssm
from test_gpu_fwd import check_sampled, sample_channels

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc(lib, d, y, last):
    fn = lib.ssm_selective_scan_fwd_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ssm.SsmTensor)] * 8 + [ctypes.c_int, ctypes.POINTER(ssm.SsmTensor),
                                                          ctypes.POINTER(ssm.SsmTensor), ctypes.c_void_p]
    ds = [ssm.describe(t) for t in (d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                                     y, last)]
    ref = lambda x: None if x is None else ctypes.byref(x)
    return fn(*[ref(x) for x in ds[:8]], 1, ref(ds[8]), ref(ds[9]),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point():
    lib = ssm.load_library()
    b, L, D, N = 1, 20000, 256, 16
    assert ssm.workspace_size(b, L, D, N) > 0, "the shape must take the segmented schedule"
    for seed in (301, 302):  # two calls in a row
        d = inputs.random_fwd(b, L, D, N, dtype=torch.bfloat16, device=DEV, seed=seed)
        y = torch.empty(b, L, D, dtype=torch.float32, device=DEV)
        last = torch.empty(b, D, N, dtype=torch.float32, device=DEV)
        assert _noalloc(lib, d, y, last) == 0
        y_ws, last_ws = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                               delta_bias=d["delta_bias"], y_dtype=torch.float32)
        torch.cuda.synchronize()
        assert ssm.device_error() == 0
        assert torch.equal(y, y_ws), f"y differs from the workspace entry point (seed {seed})"
        assert torch.equal(last, last_ws), f"last_state differs from the workspace entry point (seed {seed})"
        if seed == 301:
            ref = sample_channels(d, per_row=16, rows=1, seed=seed)
            check_sampled(y, last, ref, TOL_BF16, False, "noalloc vs oracle")
