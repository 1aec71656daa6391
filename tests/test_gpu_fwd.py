"""GPU forward scan vs the fp64 oracle, called through the C ABI.

Small shapes are compared element by element over whole tensors (several tiles plus
ragged tails in L and D). The full-size workloads run the exact launch the bench
times and are compared on seeded samples of channels (each channel is an independent
recurrence, so the oracle computes exactly those channels over the whole sequence).
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from parity import TOL_BF16, TOL_F32, check, to64
from selective_state_space_141_b300 import inputs, ssm

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gpu_fwd(d, y_dtype=None):
    y, last = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                     delta_bias=d["delta_bias"], delta_softplus=d["delta_softplus"],
                                     y_dtype=y_dtype)
    torch.cuda.synchronize()
    assert ssm.device_error() == 0
    return y, last


def oracle_fwd(d):
    return oracle.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                     delta_bias=d["delta_bias"], delta_softplus=d["delta_softplus"])


def to_dev(d):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def sample_channels(d, per_row, rows, seed):
    """Oracle on a seeded sample of channels: {b: (ds, y_ref (L, k), state_ref (k, N))}."""
    rng = np.random.default_rng(seed)
    batch, L, D = d["u"].shape
    out = {}
    for b in sorted(rng.choice(batch, size=min(rows, batch), replace=False).tolist()):
        ds = np.sort(rng.choice(D, size=min(per_row, D), replace=False))
        idx = torch.as_tensor(ds, device=d["u"].device)
        sub = dict(
            u=d["u"][b:b + 1].index_select(2, idx), delta=d["delta"][b:b + 1].index_select(2, idx),
            z=None if d["z"] is None else d["z"][b:b + 1].index_select(2, idx),
            B=d["B"][b:b + 1], C=d["C"][b:b + 1], A=d["A"].index_select(0, idx),
            D=None if d["D"] is None else d["D"].index_select(0, idx),
            delta_bias=None if d["delta_bias"] is None else d["delta_bias"].index_select(0, idx),
            delta_softplus=d["delta_softplus"])
        y, last = oracle_fwd(sub)
        out[b] = (ds, y[0], last[0])
    return out


def check_sampled(y, last, ref, tol, bf16_out, what):
    for b, (ds, yr, sr) in ref.items():
        idx = torch.as_tensor(ds, device=y.device)
        check(y[b].index_select(1, idx), yr, tol, bf16_out, f"{what} y b={b}")
        check(last[b].index_select(0, idx), sr, tol, False, f"{what} last_state b={b}")


# ---- the five workloads (four forward) -----------------------------------------------

def test_tiny_fp32_full():
    d = to_dev(inputs.fwd_inputs(inputs.TINY))
    y, last = gpu_fwd(d)
    yr, sr = oracle_fwd(d)
    check(y, yr, TOL_F32, False, "y")
    check(last, sr, TOL_F32, False, "last_state")


def test_tiny_fp32_time_split(monkeypatch):
    """The tiny fp32 workload runs the time-split schedule (4 sequence segments: aggregate
    pass, shuffle scan of the segment carries, full pass); both it and the single pass
    (SSM_B300_SEGMENTS=0) match the oracle at 1e-5, and they differ in the last bits,
    which shows the segments really ran."""
    d = to_dev(inputs.fwd_inputs(inputs.TINY))
    yr, sr = oracle_fwd(d)
    y_seg, last_seg = gpu_fwd(d)
    monkeypatch.setenv("SSM_B300_SEGMENTS", "0")
    y_one, last_one = gpu_fwd(d)
    for y, last, what in ((y_seg, last_seg, "segmented"), (y_one, last_one, "single pass")):
        check(y, yr, TOL_F32, False, f"y ({what})")
        check(last, sr, TOL_F32, False, f"last_state ({what})")
    assert not torch.equal(y_seg, y_one), "expected the segmented schedule to reassociate the recurrence"


@pytest.mark.parametrize("key", ["m130m", "m1p4b"])
def test_layer_workloads_sampled(key):
    w = inputs.FWD_WORKLOADS[key]
    d = inputs.fwd_inputs(w, DEV)
    ref = sample_channels(d, per_row=64, rows=4, seed=11)  # 256 channels over the whole sequence
    y, last = gpu_fwd(d)
    check_sampled(y, last, ref, TOL_BF16, True, key)
    y32, last32 = gpu_fwd(d, y_dtype=torch.float32)
    check_sampled(y32, last32, ref, TOL_BF16, False, key + " (fp32 out)")
    # The bf16 output is the fp32 output rounded to nearest-even.
    assert torch.equal(y, y32.to(torch.bfloat16))


def test_long_sequence_sampled():
    d = inputs.fwd_inputs(inputs.LONG, DEV)
    ref = sample_channels(d, per_row=256, rows=1, seed=12)  # 256 channels over all 131072 steps
    y, last = gpu_fwd(d)
    check_sampled(y, last, ref, TOL_BF16, True, "long")


def test_long_sequence_lti_vs_convolution():
    """Time-invariant sub-case: the first 4096 outputs equal the convolution with
    K_j = sum_n C_n exp(j dt A_n) dt B_n (brute force, independent of the oracle)."""
    d = inputs.fwd_inputs(inputs.LONG, DEV, lti=True)
    y, _ = gpu_fwd(d, y_dtype=torch.float32)
    T = 4096
    rng = np.random.default_rng(13)
    ds = rng.choice(inputs.LONG.D, size=8, replace=False)
    A, B0, C0 = to64(d["A"]), to64(d["B"][0, 0]), to64(d["C"][0, 0])
    bias, Dk = to64(d["delta_bias"]), to64(d["D"])
    u, z, raw = to64(d["u"][0, :T]), to64(d["z"][0, :T]), to64(d["delta"][0, 0])
    yg = to64(y[0, :T])
    for dd in ds:
        dt = np.logaddexp(0.0, raw[dd] + bias[dd])
        K = (C0 * np.exp(np.arange(T)[:, None] * dt * A[dd]) * dt * B0).sum(-1)
        conv = np.convolve(u[:, dd], K)[:T]
        ref = (conv + Dk[dd] * u[:, dd]) * z[:, dd] * expit(z[:, dd])
        check(yg[:, dd], ref, TOL_BF16, False, f"lti channel {dd}")


# ---- small shapes, whole tensors --------------------------------------------------------

SHAPES = [  # batch, L, D, N
    (1, 1, 1, 16), (2, 2, 3, 16), (1, 31, 33, 16), (3, 32, 64, 16), (2, 33, 65, 8), (1, 100, 96, 4),
    (2, 257, 130, 16), (1, 1000, 40, 16), (4, 64, 512, 16),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_random_shapes(shape, dtype):
    b, L, D, N = shape
    d = to_dev(inputs.random_fwd(b, L, D, N, dtype=dtype, seed=sum(shape)))
    yr, sr = oracle_fwd(d)
    if dtype == torch.float32:
        y, last = gpu_fwd(d)
        check(y, yr, TOL_F32, False, "y")
        check(last, sr, TOL_F32, False, "last")
    else:
        y, last = gpu_fwd(d)
        check(y, yr, TOL_BF16, True, "y bf16")
        y32, _ = gpu_fwd(d, y_dtype=torch.float32)
        check(y32, yr, TOL_BF16, False, "y fp32-out")
        check(last, sr, TOL_BF16, False, "last")


@pytest.mark.parametrize("flags", [(0, 0, 0, 1), (1, 0, 0, 1), (0, 1, 0, 1), (0, 0, 1, 1), (1, 1, 1, 0),
                                   (0, 0, 0, 0)], ids=lambda f: "D%dz%dbias%dsp%d" % f)
def test_optional_inputs(flags):
    has_D, has_z, has_bias, sp = flags
    d = to_dev(inputs.random_fwd(2, 70, 48, 16, dtype=torch.float32, seed=5, has_bias=bool(has_bias),
                                 has_D=bool(has_D), has_z=bool(has_z), delta_softplus=bool(sp)))
    if not sp:  # positive step sizes without softplus (the default bias is negative)
        d["delta"] = d["delta"].abs() * 0.05
        if d["delta_bias"] is not None:
            d["delta_bias"] = d["delta_bias"].abs() * 0.01
    yr, sr = oracle_fwd(d)
    y, last = gpu_fwd(d)
    check(y, yr, TOL_F32, False, "y")
    check(last, sr, TOL_F32, False, "last")


def test_zero_length_zeroes_last_state():
    d = to_dev(inputs.random_fwd(2, 0, 16, 16, dtype=torch.bfloat16))
    last = torch.full((2, 16, 16), 7.0, device=DEV)
    y, last = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                     delta_bias=d["delta_bias"], last_state=last)
    torch.cuda.synchronize()
    assert y.numel() == 0 and torch.all(last == 0)


def test_empty_batch_noop():
    d = to_dev(inputs.random_fwd(0, 5, 16, 16, dtype=torch.bfloat16))
    y, last = gpu_fwd(d)
    assert y.numel() == 0 and last.numel() == 0


def test_delta_zero_holds_state():
    d = to_dev(inputs.random_fwd(1, 50, 32, 16, dtype=torch.float32, has_bias=False, delta_softplus=False))
    d["delta"].zero_()
    y, last = gpu_fwd(d)
    assert torch.all(last == 0)
    ref = to64(d["D"]) * to64(d["u"]) * to64(d["z"]) * expit(to64(d["z"]))
    check(y, ref, TOL_F32, False, "y = D u silu(z)")


def test_large_delta_resets_state():
    d = to_dev(inputs.random_fwd(1, 40, 32, 16, dtype=torch.float32, has_bias=False, has_D=False, has_z=False,
                                 delta_softplus=False))
    d["delta"].fill_(50.0)
    y, last = gpu_fwd(d)
    h = 50.0 * to64(d["B"])[0][:, None, :] * to64(d["u"])[0][:, :, None]  # (L, D, N)
    ref = np.einsum("ln,ldn->ld", to64(d["C"])[0], h)
    check(y[0], ref, TOL_F32, False, "y")
    check(last[0], h[-1], TOL_F32, False, "last")


def test_rerun_is_deterministic():
    d = to_dev(inputs.random_fwd(2, 300, 96, 16, dtype=torch.bfloat16, seed=3))
    y1, s1 = gpu_fwd(d)
    y2, s2 = gpu_fwd(d)
    assert torch.equal(y1, y2) and torch.equal(s1, s2)


# ---- each forward kernel variant on its own ---------------------------------------------

CHAN_SHAPES = [  # shapes the TMA channel kernel accepts (bf16, D % 8 == 0, N in {8, 16})
    (1, 1, 8, 16), (2, 63, 136, 16), (2, 64, 128, 16), (3, 65, 256, 8), (1, 200, 1000, 16), (1, 1000, 264, 16),
    (2, 130, 384, 16),
]


@pytest.mark.parametrize("variant", ["generic", "chan"])
@pytest.mark.parametrize("shape", CHAN_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_variants_vs_oracle(shape, variant, monkeypatch):
    monkeypatch.setenv("SSM_B300_FORWARD_KERNEL", variant)
    b, L, D, N = shape
    d = to_dev(inputs.random_fwd(b, L, D, N, dtype=torch.bfloat16, seed=100 + sum(shape)))
    yr, sr = oracle_fwd(d)
    y, last = gpu_fwd(d)
    check(y, yr, TOL_BF16, True, f"{variant} y")
    check(last, sr, TOL_BF16, False, f"{variant} last")
    y32, _ = gpu_fwd(d, y_dtype=torch.float32)
    check(y32, yr, TOL_BF16, False, f"{variant} y fp32-out")


@pytest.mark.parametrize("flags", [(0, 0, 0, 1), (1, 1, 0, 0)], ids=["bare", "D_z_nosoftplus"])
def test_chan_optional_inputs(flags, monkeypatch):
    monkeypatch.setenv("SSM_B300_FORWARD_KERNEL", "chan")
    has_D, has_z, has_bias, sp = flags
    d = to_dev(inputs.random_fwd(2, 150, 256, 16, dtype=torch.bfloat16, seed=7, has_bias=bool(has_bias),
                                 has_D=bool(has_D), has_z=bool(has_z), delta_softplus=bool(sp)))
    if not sp:
        d["delta"] = (d["delta"].float().abs() * 0.05).to(torch.bfloat16)
    yr, sr = oracle_fwd(d)
    y, last = gpu_fwd(d, y_dtype=torch.float32)
    check(y, yr, TOL_BF16, False, "y")
    check(last, sr, TOL_BF16, False, "last")


# ---- the segmented schedule (long sequences over few channels) --------------------------

SEG_SHAPES = [(1, 20000, 256, 16), (1, 10007, 136, 16), (2, 9000, 128, 8)]


@pytest.mark.parametrize("shape", SEG_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_segmented_vs_oracle(shape):
    b, L, D, N = shape
    assert ssm.workspace_size(b, L, D, N) > 0, "shape expected to use the segmented schedule"
    d = to_dev(inputs.random_fwd(b, L, D, N, dtype=torch.bfloat16, seed=200 + sum(shape)))
    yr, sr = oracle_fwd(d)
    y, last = gpu_fwd(d, y_dtype=torch.float32)
    check(y, yr, TOL_BF16, False, "segmented y")
    check(last, sr, TOL_BF16, False, "segmented last_state")
    y0, last0 = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                       delta_bias=d["delta_bias"], y_dtype=torch.float32, use_workspace=False)
    torch.cuda.synchronize()
    check(y0, yr, TOL_BF16, False, "unsegmented y")
    check(y, y0, TOL_BF16, False, "segmented vs unsegmented")


def test_workspace_too_small_falls_back():
    b, L, D, N = 1, 20000, 256, 16
    d = to_dev(inputs.random_fwd(b, L, D, N, dtype=torch.bfloat16, seed=77))
    small = torch.empty(64, dtype=torch.uint8, device=DEV)
    y, last = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                     delta_bias=d["delta_bias"], y_dtype=torch.float32, workspace=small)
    torch.cuda.synchronize()
    yr, sr = oracle_fwd(d)
    check(y, yr, TOL_BF16, False, "fallback y")


# ---- the time-split schedule through the plain entry point (no workspace) -------------------

def test_long_sequence_plain_call_sampled():
    """The long sequence through ssm_selective_scan_fwd itself: no workspace, so the
    segmented schedule keeps its carries in y; sampled channels against the oracle."""
    d = inputs.fwd_inputs(inputs.LONG, DEV)
    assert ssm.workspace_size(1, inputs.LONG.L, inputs.LONG.D, 16) > 0, "the shape must segment"
    ref = sample_channels(d, per_row=32, rows=1, seed=14)
    y, last = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                     delta_bias=d["delta_bias"], use_workspace=False)
    torch.cuda.synchronize()
    assert ssm.device_error() == 0
    check_sampled(y, last, ref, TOL_BF16, True, "long (plain call)")
    y_ws, last_ws = gpu_fwd(d)
    assert torch.equal(y, y_ws) and torch.equal(last, last_ws), "plain call differs from the workspace schedule"


def test_long_sequence_plain_call_lti_vs_convolution():
    d = inputs.fwd_inputs(inputs.LONG, DEV, lti=True)
    y, _ = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                  delta_bias=d["delta_bias"], y_dtype=torch.float32, use_workspace=False)
    torch.cuda.synchronize()
    T = 4096
    rng = np.random.default_rng(15)
    A, B0, C0 = to64(d["A"]), to64(d["B"][0, 0]), to64(d["C"][0, 0])
    bias, Dk = to64(d["delta_bias"]), to64(d["D"])
    u, z, raw = to64(d["u"][0, :T]), to64(d["z"][0, :T]), to64(d["delta"][0, 0])
    yg = to64(y[0, :T])
    for dd in rng.choice(inputs.LONG.D, size=8, replace=False):
        dt = np.logaddexp(0.0, raw[dd] + bias[dd])
        K = (C0 * np.exp(np.arange(T)[:, None] * dt * A[dd]) * dt * B0).sum(-1)
        ref = (np.convolve(u[:, dd], K)[:T] + Dk[dd] * u[:, dd]) * z[:, dd] * expit(z[:, dd])
        check(yg[:, dd], ref, TOL_BF16, False, f"lti channel {dd} (plain call)")


@pytest.mark.parametrize("y_dtype", [torch.bfloat16, torch.float32], ids=["bf16y", "f32y"])
@pytest.mark.parametrize("shape", [(1, 20000, 256, 16), (2, 9000, 128, 8), (1, 12001, 64, 16), (1, 40000, 64, 16)],
                         ids=lambda s: "x".join(map(str, s)))
def test_plain_call_segments_vs_oracle(shape, y_dtype):
    """Shapes with few channels and long sequences segment without a workspace; whole
    tensors against the oracle (ragged last segment and chunk), h0 included."""
    b, L, D, N = shape
    d = to_dev(inputs.random_fwd(b, L, D, N, dtype=torch.bfloat16, seed=L + D))
    assert ssm.workspace_size(b, L, D, N) > 0, "the shape must segment"
    h0 = torch.randn(b, D, N, generator=torch.Generator().manual_seed(5)).to(DEV)
    y, last = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                     delta_bias=d["delta_bias"], y_dtype=y_dtype, use_workspace=False, h0=h0)
    torch.cuda.synchronize()
    assert ssm.device_error() == 0
    yr, sr = oracle.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                       delta_bias=d["delta_bias"], h0=h0)
    check(y, yr, TOL_BF16, y_dtype == torch.bfloat16, "y")
    check(last, sr, TOL_BF16, False, "last_state")


@pytest.mark.parametrize("shape", [(1, 4096, 32, 16), (1, 2000, 64, 8), (2, 1500, 40, 4)],
                         ids=lambda s: "x".join(map(str, s)))
def test_fp32_segments_vs_oracle(shape, monkeypatch):
    """fp32 I/O (generic kernel) split into 2 .. 64 sequence segments: the carry scan's
    warps and their block carry, against the oracle at 1e-5, h0 included."""
    b, L, D, N = shape
    d = to_dev(inputs.random_fwd(b, L, D, N, dtype=torch.float32, seed=L + 3 * D))
    h0 = torch.randn(b, D, N, generator=torch.Generator().manual_seed(6)).to(DEV)
    yr, sr = oracle.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                       delta_bias=d["delta_bias"], h0=h0)
    y, last = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                     delta_bias=d["delta_bias"], h0=h0, use_workspace=False)
    torch.cuda.synchronize()
    assert ssm.device_error() == 0
    check(y, yr, TOL_F32, False, "y")
    check(last, sr, TOL_F32, False, "last_state")
