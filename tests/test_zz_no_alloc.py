"""ssm_selective_scan_fwd_noalloc against ssm_selective_scan_fwd_ws, through the C ABI.

The no-allocation entry point is for callers that can only pass the buffers they own
(a fixed memory budget, a plugin interface given just inputs and outputs, a path where
an allocation must not stall or fail). It must give the same result as the entry point
that takes a caller-owned workspace. The shape below takes the segmented schedule, so
the built-in scratch array is really used; two calls in a row with different inputs
also check that the second call does not depend on what the first left in the array.
"""
import ctypes

import pytest
import torch

from parity import TOL_BF16, check
from selective_state_space_141_b300 import inputs, ssm

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
        check(y, y_ws, TOL_BF16, False, f"y (seed {seed})")
        check(last, last_ws, TOL_BF16, False, f"last_state (seed {seed})")
